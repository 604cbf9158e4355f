// C ABI of the attention forward library: argument validation, tensor-map
// construction, launch, and the device status word.  See include/fa.h for
// the contract.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_bwd_dispatch.h"
#include "fa_dispatch.h"
#include "fa_schedule.h"

// {code, wait site, block} of the first device-side failure since the last read
__device__ unsigned int g_fa_status[4];

// Scratch of fa_fwd_varlen_noalloc: the varlen planning workspace (task count,
// task counter, task records) as a file-scope device array, one per device.
// 1 MiB holds (2^20 - 256) / 32 = 32 760 task records.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
__device__ __align__(256) unsigned char g_fa_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
// 5 (d_qk, d_v) pairs x {non-causal, causal} x the kernel modes (fixed-length, FMA-pipe exp2, varlen,
// dynamic assignment, split-KV)
constexpr int kVariants = fa::kNumModes;
constexpr int kNumKernels = 5 * 2 * kVariants;
constexpr int kVariantFixed = fa::kModeFixed, kVariantEmu = fa::kModeEmu, kVariantVarlen = fa::kModeVarlen,
              kVariantDyn = fa::kModeDyn, kVariantSplit = fa::kModeSplit, kVariantDirect = fa::kModeDirect;
// The direct epilogue (O rows stored from registers) is the default for every
// fixed-length problem: since a task's first P V waits only for the O-free
// arrival after one stage's epilogue, it measures at least as fast as the
// staged TMA store on long tasks too (GB300, 20 launches, two rounds: asym
// +4.0 %, mha8k +0.2 / +1.9 %, causal 8k +1.1 %, 16k +0.9 %, mqa +0.1 / +1.2 %,
// gqa -0.2 / +1.1 %; short causal rows +2.6 to +4.7 %).  store_mode 1 still
// selects the staged TMA store.

// variable-length batches: workspace = [task count (int) at byte 0, task counter (uint) at byte 16,
// padding to 256 B][VarlenTask records]
constexpr size_t kVarlenHeaderBytes = 256;
constexpr size_t kVarlenCounterOffset = 16;
constexpr int kVarlenMaxBatch = 16384;  // sequences one planning CTA sorts in shared memory
constexpr int kPlanThreads = 1024;
constexpr unsigned int kSiteVarlenSeqlens = 501;  // a cu_seqlens entry is out of order or out of range
constexpr unsigned int kSiteVarlenCapacity = 502; // more tasks than the workspace holds

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int64_t l2_bytes = 0;
  int smem_optin = 0;
  unsigned int* status = nullptr;
  void* noalloc_scratch = nullptr;  // g_fa_noalloc_scratch on this device
  bool kernel_ready[kNumKernels] = {};
  bool debug_ready[5 * 2 * 2 * 3] = {};  // (d_qk, d_v) pair x causal x (fixed, direct) x (trace, check, stagger)
  bool bwd_ready[3 * 2 * 2] = {};   // ((64,64), (128,128), (192,128)) x (dK/dV, dQ) x (non-causal, causal)
  bool bwd_trace_ready[2 * 2] = {};  // the event-log build, (128,128): (dK/dV, dQ) x (non-causal, causal)
  bool bwd_varlen_ready[3 * 2 * 2] = {};  // the variable-length build, as bwd_ready
  bool bwd_plan_ready = false;            // the backward's varlen planning kernel
  bool plan_ready = false;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int kernel_index(int dq, int dv, int causal, int variant) {
  int pair = -1;
  if (dq == 64 && dv == 64) pair = 0;
  if (dq == 128 && dv == 64) pair = 1;
  if (dq == 128 && dv == 128) pair = 2;
  if (dq == 192 && dv == 64) pair = 3;
  if (dq == 192 && dv == 128) pair = 4;
  return pair < 0 ? -1 : (pair * 2 + (causal ? 1 : 0)) * kVariants + variant;
}

bool get_entry(int dq, int dv, int causal, int variant, fa::KernelEntry* e) {
  if (dq == 64) return fa::entry_d64(dv, causal, variant, e);
  if (dq == 128) return fa::entry_d128(dv, causal, variant, e);
  if (dq == 192) return fa::entry_d192(dv, causal, variant, e);
  return false;
}

// build variants: var = fa::kVarTrace, fa::kVarCheck or fa::kVarStagger, variant fixed or direct
bool get_debug_entry(int dq, int dv, int causal, int variant, int var, fa::KernelEntry* e) {
  if (var == fa::kVarTrace) return fa::entry_trace(dq, dv, causal, variant, e);
  if (var == fa::kVarStagger) return fa::entry_stagger(dq, dv, causal, variant, e);
  if (var == fa::kVarCheck)
    return dq == 192 ? fa::entry_check_b(dq, dv, causal, variant, e) : fa::entry_check_a(dq, dv, causal, variant, e);
  return false;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device pointer on `dev` (or managed memory)?
bool is_device_ptr(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

int init_device(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FA_ERR_CUDA;
    if (prop.major != 10) return FA_ERR_UNSUPPORTED;  // tcgen05 / TMEM: Blackwell datacenter parts
    st.sms = prop.multiProcessorCount;
    st.l2_bytes = prop.l2CacheSize;
    st.smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
    void* sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
    st.status = static_cast<unsigned int*>(sym);
    if (cudaMemset(st.status, 0, sizeof(unsigned int) * 4) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaGetSymbolAddress(&sym, g_fa_noalloc_scratch) != cudaSuccess) return FA_ERR_CUDA;
    st.noalloc_scratch = sym;
    // the header (task count, task counter) starts cleared; every call's
    // planning kernel rewrites both before the attention kernel reads them
    if (cudaMemset(st.noalloc_scratch, 0, kVarlenHeaderBytes) != cudaSuccess) return FA_ERR_CUDA;
    // the two clears above run on the legacy default stream, which is not
    // ordered against a caller's non-blocking stream: finish them before this
    // call enqueues anything, so that neither lands after a kernel on the
    // caller's stream has written the status word or the scratch header
    if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FA_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.ready = true;
  }
  *out = &st;
  return FA_OK;
}

// Per device and kernel: allow the large dynamic shared memory and check the
// register count the warp-role split assumes (the roles move registers with
// setmaxnreg; their total must fit what the CTA is launched with).
int prepare_kernel(DeviceState* st, bool* ready, const fa::KernelEntry& e) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (*ready) return FA_OK;
  if (e.smem > st->smem_optin) return FA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, e.smem) != cudaSuccess)
    return FA_ERR_CUDA;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, e.fn) != cudaSuccess) return FA_ERR_CUDA;
  // setmaxnreg.inc would wait forever if the launch left fewer registers than the split needs
  if (attr.numRegs * fa::kThreads < fa::kRegBudgetPerCta || attr.maxThreadsPerBlock < fa::kThreads)
    return FA_ERR_UNSUPPORTED;
  *ready = true;
  return FA_OK;
}

int encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
           const cuuint32_t* box) {
  cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                        dims, strides_bytes, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Q or O viewed as (d, pack, groups, S, B): one box is 128 rows = (128/pack
// positions) x (pack heads) x 64 columns.
int encode_q_like(CUtensorMap* m, const void* base, int B, int S, int H, int d, int pack) {
  const cuuint64_t e = 2;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(pack), static_cast<cuuint64_t>(H / pack),
                        static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  // with one batch (varlen) the batch stride is never used: keep it small so
  // that the encoder's stride limit does not depend on the sequence length
  cuuint64_t strides[4] = {d * e, static_cast<cuuint64_t>(pack) * d * e, static_cast<cuuint64_t>(H) * d * e,
                           static_cast<cuuint64_t>(B > 1 ? S : 1) * H * d * e};
  cuuint32_t box[5] = {64, static_cast<cuuint32_t>(pack), 1, static_cast<cuuint32_t>(fa::kBM / pack), 1};
  return encode(m, base, 5, dims, strides, box);
}

// K or V viewed as (d, Hkv, S, B): one box is box_rows keys x 64 columns of a head.
int encode_kv(CUtensorMap* m, const void* base, int B, int S, int H, int d, int box_rows = fa::kBN) {
  const cuuint64_t e = 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {d * e, static_cast<cuuint64_t>(H) * d * e,
                           static_cast<cuuint64_t>(B > 1 ? S : 1) * H * d * e};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  return encode(m, base, 4, dims, strides, box);
}

// Test hook: y_fma[i] = the FMA-pipe 2^x above, y_mufu[i] = ex2.approx, for
// comparing the two on the device.
__global__ void exp2_selftest_kernel(const float* x, float* y_fma, float* y_mufu, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float a = x[i], b = (i + 1 < n) ? x[i + 1] : 0.f;
  float ya, yb;
  fa::ex2_fma_x2(fa::f2_pack(a, b), ya, yb);
  y_fma[i] = ya;
  y_mufu[i] = fa::ex2_approx(a);
  if (i + 1 < n) {
    y_fma[i + 1] = yb;
    y_mufu[i + 1] = fa::ex2_approx(b);
  }
}

__global__ void fill_f32(float* p, int64_t n, float v) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    p[i] = v;
}

// ---------------------------------------------------------------------------
// variable-length batches: the planning kernel
// ---------------------------------------------------------------------------
// One CTA.  Checks cu_seqlens, sorts the sequences by the K/V blocks of their
// heaviest tile (longest first, ties by index; "FlashAttention-4 wiki", "Core
// methods": LPT scheduling with a preprocessing kernel for varlen), then
// writes every sequence's tasks in that order.  Shared memory: the sort values
// (a power of two >= batch) and the first task of each sorted position.
size_t plan_smem_bytes(int batch) {
  int npow2 = 1;
  while (npow2 < batch) npow2 <<= 1;
  return static_cast<size_t>(npow2) * sizeof(uint64_t) + static_cast<size_t>(batch + 1) * sizeof(int);
}

__device__ void plan_error(unsigned int* status, int* count, unsigned int site, int index) {
  *count = 0;
  if (atomicCAS(&status[0], 0u, static_cast<unsigned int>(FA_ERR_INVALID_ARG)) == 0u) {
    status[1] = site;
    status[2] = static_cast<unsigned int>(index);
  }
}

__global__ void __launch_bounds__(kPlanThreads) varlen_plan_kernel(
    const int* cu_q, const int* cu_k, int batch, int64_t total_q, int64_t total_k, fa::Problem base, int d_qk,
    int d_v, int64_t l2_budget, fa::VarlenTask* tasks, int* count, unsigned int* sched_next, int64_t capacity,
    unsigned int* status) {
  extern __shared__ __align__(16) uint8_t plan_smem[];
  __shared__ int bad_index;
  __shared__ long long warp_sums[kPlanThreads / 32];
  int npow2 = 1;
  while (npow2 < batch) npow2 <<= 1;
  uint64_t* vals = reinterpret_cast<uint64_t*>(plan_smem);
  int* start = reinterpret_cast<int*>(vals + npow2);
  const int tid = threadIdx.x;

  if (tid == 0) {
    bad_index = INT_MAX;
    *sched_next = 0;  // the attention kernel's dynamic task counter
  }
  __syncthreads();
  for (int i = tid; i < npow2; i += kPlanThreads) {
    uint64_t v = 0;  // padding sorts after every sequence
    if (i < batch) {
      const int q0 = cu_q[i], q1 = cu_q[i + 1], k0 = cu_k[i], k1 = cu_k[i + 1];
      if (q0 < 0 || q1 < q0 || q1 > total_q || k0 < 0 || k1 < k0 || k1 > total_k) atomicMin(&bad_index, i);
      v = fa::varlen_sort_value(fa::varlen_key(q1 - q0, k1 - k0), i);
    }
    vals[i] = v;
  }
  __syncthreads();
  if (bad_index != INT_MAX) {
    if (tid == 0) plan_error(status, count, kSiteVarlenSeqlens, bad_index);
    return;
  }

  // bitonic sort, descending
  for (int k = 2; k <= npow2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < npow2; i += kPlanThreads) {
        const int l = i ^ j;
        if (l > i) {
          const uint64_t a = vals[i], b = vals[l];
          if (((i & k) == 0) ? (a < b) : (a > b)) {
            vals[i] = b;
            vals[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }

  // tasks per sorted position, exclusive scan: thread tid owns positions [lo, hi)
  const int per = (batch + kPlanThreads - 1) / kPlanThreads;
  const int lo = tid * per < batch ? tid * per : batch;
  const int hi = lo + per < batch ? lo + per : batch;
  auto tasks_at = [&](int pos) -> long long {
    const int b = fa::varlen_sort_index(vals[pos]);
    const int sq = cu_q[b + 1] - cu_q[b], sk = cu_k[b + 1] - cu_k[b];
    if (sq == 0) return 0;
    return fa::varlen_sequence_problem(base, sq, sk, d_qk, d_v, l2_budget).num_tasks;
  };
  long long mine = 0;
  for (int i = lo; i < hi; ++i) mine += tasks_at(i);
  long long incl = mine;  // inclusive scan inside the warp
  const int lane = tid & 31, warp = tid >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long w = warp_sums[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const long long total = warp_sums[kPlanThreads / 32 - 1];
  if (total > capacity) {
    if (tid == 0) plan_error(status, count, kSiteVarlenCapacity, 0);
    return;
  }
  long long run = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - mine;
  for (int i = lo; i < hi; ++i) {
    start[i] = static_cast<int>(run);
    run += tasks_at(i);
  }
  if (tid == 0) start[batch] = static_cast<int>(total);
  __syncthreads();

  // emit: task t belongs to the last sorted position whose first task is <= t
  for (int t = tid; t < static_cast<int>(total); t += kPlanThreads) {
    int a = 0, z = batch - 1;
    while (a < z) {
      const int mid = (a + z + 1) >> 1;
      if (start[mid] <= t) a = mid;
      else z = mid - 1;
    }
    const int b = fa::varlen_sort_index(vals[a]);
    const int q0 = cu_q[b], k0 = cu_k[b];
    const fa::Problem seq = fa::varlen_sequence_problem(base, cu_q[b + 1] - q0, cu_k[b + 1] - k0, d_qk, d_v, l2_budget);
    tasks[t] = fa::varlen_record(seq, b, q0, k0, t - start[a]);
  }
  if (tid == 0) *count = static_cast<int>(total);
}

// ---------------------------------------------------------------------------
// split-KV: the merge kernel
// ---------------------------------------------------------------------------
constexpr int kMaxSplits = 1024;

// One warp per output row (b, pos, head), each lane DV / 32 columns.  The
// ranges' states combine exactly after rescaling to a common base ("Infra:
// Flash Attention", "How softmax is computed in pieces"; "Prefill and decode":
// segments computed apart and merged): with O_s = U_s / l_s and
// LSE_s = m_s + log l_s per range s,
//   LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
// A range without a visible key has LSE_s = -inf and weight 0; a row with none
// at all gets O = 0, LSE = -inf.
template <int DV>
__global__ void __launch_bounds__(256) splitkv_merge_kernel(const float* __restrict__ opart,
                                                            const float* __restrict__ lpart,
                                                            uint16_t* __restrict__ o, float* __restrict__ lse,
                                                            int B, int Sq, int Hq, int splits) {
  constexpr int kPer = DV / 32;
  static_assert(kPer == 2 || kPer == 4, "d_v 64 or 128");
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(B) * Sq * Hq;
  const int64_t lstride = rows;          // per range in lpart ([B, Hq, Sq] per range)
  const int64_t ostride = rows * DV;     // per range in opart ([B, Sq, Hq, DV] per range)
  const int64_t step = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += step) {
    const int64_t bs = row / Hq;  // b * Sq + pos
    const int head = static_cast<int>(row - bs * Hq);
    const int64_t b = bs / Sq;
    const int pos = static_cast<int>(bs - b * Sq);
    const int64_t li = (b * Hq + head) * Sq + pos;
    float m = -INFINITY;
    for (int s = 0; s < splits; ++s) m = fmaxf(m, lpart[s * lstride + li]);
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < splits; ++s) {
        const float l = lpart[s * lstride + li];
        if (l == -INFINITY) continue;
        const float w = expf(l - m);
        wsum += w;
        const float* src = opart + s * ostride + row * DV + lane * kPer;
        if constexpr (kPer == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          acc[0] += w * x.x, acc[1] += w * x.y, acc[2] += w * x.z, acc[3] += w * x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src);
          acc[0] += w * x.x, acc[1] += w * x.y;
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint32_t packed[kPer / 2];
#pragma unroll
    for (int i = 0; i < kPer / 2; ++i) packed[i] = fa::pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    uint16_t* dst = o + row * DV + lane * kPer;
    if constexpr (kPer == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = packed[0];
    }
    if (lane == 0 && lse != nullptr) lse[li] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

// Options, heads, head dims and scale (shared by the fixed-length and varlen calls).
int validate_common(int heads_q, int heads_kv, int d_qk, int d_v, float scale, const fa_options& opt) {
  if (heads_q < 1 || heads_kv < 1) return FA_ERR_INVALID_ARG;
  if (heads_q % heads_kv != 0) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale)) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (kernel_index(d_qk, d_v, 0, 0) < 0) return FA_ERR_UNSUPPORTED;
  if (opt.pack < 0 || opt.grid < 0 ||
      (opt.debug_flags & ~(fa::kDebugSkipPArrive | fa::kDebugCountRescale | fa::kDebugChecks |
                           fa::kDebugPlantBadTask)) != 0)
    return FA_ERR_INVALID_ARG;
  // the planted fault is for the checking build only
  if ((opt.debug_flags & fa::kDebugPlantBadTask) && !(opt.debug_flags & fa::kDebugChecks)) return FA_ERR_INVALID_ARG;
  if (opt.trace != nullptr &&
      (opt.trace_ctas < 1 || opt.trace_cap < 1 || (reinterpret_cast<uintptr_t>(opt.trace) & 7u) != 0))
    return FA_ERR_INVALID_ARG;
  if (opt.exp_emu != 0 && opt.exp_emu != 1) return FA_ERR_INVALID_ARG;
  // the O-rescale counter is compiled into the FMA-exp2 kernels and the checking build only
  if ((opt.debug_flags & fa::kDebugCountRescale) != 0 && opt.exp_emu != 1 && !(opt.debug_flags & fa::kDebugChecks))
    return FA_ERR_UNSUPPORTED;
  if (opt.store_mode < 0 || opt.store_mode > 2) return FA_ERR_INVALID_ARG;
  if (opt.no_balance != 0 && opt.no_balance != 1) return FA_ERR_INVALID_ARG;
  if (opt.stagger != 0 && opt.stagger != 1) return FA_ERR_INVALID_ARG;
  // the kept reference may lag the row maximum by up to tau (log2 units), so
  // unnormalised weights reach 2^tau: keep them far inside the fp32 range
  if (!(opt.tau >= 0.f && opt.tau <= 64.f)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(opt.timeout_s) || opt.timeout_s > 3600.0) return FA_ERR_INVALID_ARG;
  if (opt.pack > 0) {
    const int ratio = heads_q / heads_kv;
    if (fa::kBM % opt.pack != 0 || ratio % opt.pack != 0) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

int validate(const void* q, const void* k, const void* v, void* o, const float* lse, int batch, int heads_q,
             int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, float scale, const fa_options& opt) {
  if (batch < 0 || seqlen_q < 0 || seqlen_k < 0) return FA_ERR_INVALID_ARG;
  const int rc = validate_common(heads_q, heads_kv, d_qk, d_v, scale, opt);
  if (rc != FA_OK) return rc;
  if (batch == 0 || seqlen_q == 0) return FA_OK;  // nothing to compute; pointers unused
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(opt.workspace))
    return FA_ERR_INVALID_ARG;
  // every TMA extent and index must fit in 32 bits
  const int64_t big = int64_t(1) << 31;
  if (static_cast<int64_t>(seqlen_q) + seqlen_k >= big) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace

extern "C" {

void fa_options_default(fa_options* opts) {
  if (!opts) return;
  opts->tau = 8.0f;
  opts->pack = 0;
  opts->grid = 0;
  opts->timeout_s = 1.0;
  opts->debug_flags = 0;
  opts->exp_emu = 0;
  opts->workspace = nullptr;
  opts->store_mode = 0;
  opts->no_balance = 0;
  opts->trace = nullptr;
  opts->trace_ctas = 0;
  opts->trace_cap = 0;
  opts->stagger = 0;
}

int fa_version(void) { return 100; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK:
      return "FA_OK";
    case FA_ERR_INVALID_ARG:
      return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED:
      return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA:
      return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_TIMEOUT:
      return "FA_ERR_DEVICE_TIMEOUT";
    case FA_ERR_DEVICE_CHECK:
      return "FA_ERR_DEVICE_CHECK";
    default:
      return "FA_ERR_UNKNOWN";
  }
}

// The fixed-length forward.  num_splits < 0: the plain call (fa_fwd_ex);
// num_splits >= 0: split-KV (0 = choose), partial results in split_ws and a
// merge kernel after the attention kernel; a problem that needs no split runs
// the plain kernel.
static int fixed_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
                     int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
                     int num_splits, void* split_ws, size_t split_ws_bytes, const fa_options* opts,
                     fa_stream_t stream_) {
  fa_options opt;
  fa_options_default(&opt);
  if (opts) opt = *opts;
  if (opt.tau < 0.f) opt.tau = 8.0f;
  if (opt.timeout_s <= 0.0) opt.timeout_s = 1.0;
  causal = causal ? 1 : 0;

  int rc = validate(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, scale, opt);
  if (rc != FA_OK) return rc;
  if (opt.workspace != nullptr && opt.exp_emu) return FA_ERR_UNSUPPORTED;  // one or the other
  const bool split_api = num_splits >= 0;
  if (split_api && (opt.workspace != nullptr || opt.exp_emu)) return FA_ERR_UNSUPPORTED;
  if (split_api && num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  if (split_api && !aligned16(split_ws)) return FA_ERR_INVALID_ARG;
  if (batch == 0 || seqlen_q == 0) return FA_OK;
  if (scale == 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d_qk));
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* st = nullptr;
  rc = init_device(dev, &st);
  if (rc != FA_OK) return rc;
  if (!is_device_ptr(q, dev) || !is_device_ptr(k, dev) || !is_device_ptr(v, dev) || !is_device_ptr(o, dev) ||
      (lse != nullptr && !is_device_ptr(lse, dev)) ||
      (opt.workspace != nullptr && !is_device_ptr(opt.workspace, dev)))
    return FA_ERR_INVALID_ARG;

  if (seqlen_k == 0) {  // no key anywhere: O = 0, lse = -inf
    const size_t obytes = static_cast<size_t>(batch) * seqlen_q * heads_q * d_v * 2;
    if (cudaMemsetAsync(o, 0, obytes, stream) != cudaSuccess) return FA_ERR_CUDA;
    if (lse) {
      const int64_t n = static_cast<int64_t>(batch) * heads_q * seqlen_q;
      fill_f32<<<st->sms * 4, 256, 0, stream>>>(lse, n, -INFINITY);
      if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    }
    return FA_OK;
  }

  fa::Problem prob = fa::make_problem(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal,
                                      fa::causal_section_budget(st->l2_bytes), opt.pack);
  if (split_api) {
    fa::set_splits(prob, num_splits > 0 ? num_splits : fa::choose_splits(prob, st->sms));
    if (prob.splits > 1) {
      if (split_ws == nullptr || split_ws_bytes < fa_splitkv_workspace_size(batch, heads_q, seqlen_q, d_v,
                                                                           prob.splits) ||
          !is_device_ptr(split_ws, dev))
        return FA_ERR_INVALID_ARG;
    }
  }
  const bool split = split_api && prob.splits > 1;
  const bool direct = opt.store_mode != 1;
  const int variant = split ? kVariantSplit
                            : (opt.workspace != nullptr ? kVariantDyn
                                                        : (opt.exp_emu ? kVariantEmu
                                                                       : (direct ? kVariantDirect : kVariantFixed)));
  // the build variants (event log, checks, stagger) exist for the fixed-length
  // static modes only, one at a time
  const int nvar = (opt.trace != nullptr ? 1 : 0) + ((opt.debug_flags & fa::kDebugChecks) ? 1 : 0) +
                   (opt.stagger ? 1 : 0);
  const int dbg = opt.trace != nullptr ? fa::kVarTrace
                                       : ((opt.debug_flags & fa::kDebugChecks) ? fa::kVarCheck
                                                                                : (opt.stagger ? fa::kVarStagger : 0));
  if (dbg != 0 && (nvar > 1 || (variant != kVariantFixed && variant != kVariantDirect))) return FA_ERR_UNSUPPORTED;
  const int idx = kernel_index(d_qk, d_v, causal, variant);
  fa::KernelEntry entry;
  bool* ready = nullptr;
  if (dbg == 0) {
    if (idx < 0 || !get_entry(d_qk, d_v, causal, variant, &entry)) return FA_ERR_UNSUPPORTED;
    ready = &st->kernel_ready[idx];
  } else {
    if (idx < 0 || !get_debug_entry(d_qk, d_v, causal, variant, dbg, &entry)) return FA_ERR_UNSUPPORTED;
    ready = &st->debug_ready[((idx / kVariants) * 2 + (variant == kVariantDirect ? 1 : 0)) * 3 +
                             (dbg == fa::kVarTrace ? 0 : (dbg == fa::kVarCheck ? 1 : 2))];
    if (opt.trace != nullptr && !is_device_ptr(opt.trace, dev)) return FA_ERR_INVALID_ARG;
  }
  rc = prepare_kernel(st, ready, entry);
  if (rc != FA_OK) return rc;
  const int64_t ctas = opt.grid > 0 ? opt.grid : st->sms;
  // balanced static order: without the mask the tiles of a partial last wave
  // run as key halves on the two stages of a CTA; with it, heavy and light
  // m_blocks are paired on one CTA
  if ((variant == kVariantFixed || variant == kVariantDirect || variant == kVariantEmu) && !opt.no_balance)
    fa::set_balance(prob, ctas);

  fa::Params p;
  std::memset(&p, 0, sizeof(p));
  p.prob = prob;
  if (p.prob.num_tasks >= (int64_t(1) << 31)) return FA_ERR_INVALID_ARG;  // the device decodes tasks in 32 bits
  if (encode_q_like(&p.tm_q, q, batch, seqlen_q, heads_q, d_qk, p.prob.pack) != FA_OK) return FA_ERR_CUDA;
  if (encode_kv(&p.tm_k, k, batch, seqlen_k, heads_kv, d_qk) != FA_OK) return FA_ERR_CUDA;
  if (encode_kv(&p.tm_v, v, batch, seqlen_k, heads_kv, d_v) != FA_OK) return FA_ERR_CUDA;
  if (encode_q_like(&p.tm_o, o, batch, seqlen_q, heads_q, d_v, p.prob.pack) != FA_OK) return FA_ERR_CUDA;
  p.lse = lse;
  p.lse_hstride = seqlen_q;
  p.lse_bstride = static_cast<int64_t>(heads_q) * seqlen_q;
  p.o = static_cast<uint16_t*>(o);
  p.o_row_stride = static_cast<int64_t>(heads_q) * d_v;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 ? 1 : 0;
  p.status = st->status;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.tau = opt.tau;
  p.timeout_ns = static_cast<unsigned long long>(opt.timeout_s * 1e9);
  p.debug_flags = opt.debug_flags;
  p.trace = opt.trace;
  p.trace_ctas = opt.trace_ctas;
  p.trace_cap = opt.trace_cap;

  int64_t grid = ctas;
  if (grid > p.prob.num_tasks) grid = p.prob.num_tasks;
  if (grid < 1) return FA_OK;
  if (opt.workspace != nullptr) {  // dynamic assignment: the counter starts at 0 for this launch
    p.sched_next = static_cast<unsigned int*>(opt.workspace);
    if (cudaMemsetAsync(opt.workspace, 0, FA_SCHED_WORKSPACE_BYTES, stream) != cudaSuccess) return FA_ERR_CUDA;
  }
  const int64_t rows = static_cast<int64_t>(batch) * seqlen_q * heads_q;
  if (split) {
    p.opart = static_cast<float*>(split_ws);
    p.lpart = p.opart + static_cast<int64_t>(prob.splits) * rows * d_v;
  }
  if (entry.launch(p, static_cast<int>(grid), stream) != cudaSuccess) return FA_ERR_CUDA;
  if (split) {
    const int warps_per_block = 8;
    int64_t blocks = (rows + warps_per_block - 1) / warps_per_block;
    if (blocks > static_cast<int64_t>(st->sms) * 16) blocks = static_cast<int64_t>(st->sms) * 16;
    if (d_v == 128)
      splitkv_merge_kernel<128><<<static_cast<int>(blocks), 32 * warps_per_block, 0, stream>>>(
          p.opart, p.lpart, static_cast<uint16_t*>(o), lse, batch, seqlen_q, heads_q, prob.splits);
    else
      splitkv_merge_kernel<64><<<static_cast<int>(blocks), 32 * warps_per_block, 0, stream>>>(
          p.opart, p.lpart, static_cast<uint16_t*>(o), lse, batch, seqlen_q, heads_q, prob.splits);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
              int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
              const fa_options* opts, fa_stream_t stream) {
  return fixed_fwd(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale, -1,
                   nullptr, 0, opts, stream);
}

size_t fa_splitkv_workspace_size(int batch, int heads_q, int seqlen_q, int d_v, int num_splits) {
  if (batch < 0 || heads_q < 0 || seqlen_q < 0 || d_v < 0 || num_splits < 1) return 0;
  if (num_splits == 1) return 0;
  return static_cast<size_t>(num_splits) * batch * seqlen_q * heads_q * (d_v + 1) * sizeof(float);
}

int fa_splitkv_num_splits(int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v,
                          int causal, int pack, int num_sms) {
  if (batch < 1 || seqlen_q < 1 || seqlen_k < 1 || heads_q < 1 || heads_kv < 1 || heads_q % heads_kv ||
      num_sms < 1)
    return 1;
  if (pack < 0 || (pack > 0 && (fa::kBM % pack != 0 || (heads_q / heads_kv) % pack != 0))) return 1;
  fa::Problem p = fa::make_problem(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal ? 1 : 0,
                                   int64_t(64) << 20, pack);
  fa::set_splits(p, fa::choose_splits(p, num_sms));
  return p.splits;
}

int fa_fwd_splitkv_ex(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
                      int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
                      int num_splits, void* workspace, size_t workspace_bytes, const fa_options* opts,
                      fa_stream_t stream) {
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  return fixed_fwd(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale,
                   num_splits, workspace, workspace_bytes, opts, stream);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
                   int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
                   int num_splits, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return fa_fwd_splitkv_ex(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale,
                           num_splits, workspace, workspace_bytes, nullptr, stream);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q, int heads_kv,
           int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale, fa_stream_t stream) {
  return fa_fwd_ex(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale, nullptr,
                   stream);
}

size_t fa_varlen_workspace_size(int batch, int heads_q, int64_t total_q) {
  if (batch < 0 || heads_q < 1 || total_q < 0) return 0;
  return kVarlenHeaderBytes + sizeof(fa::VarlenTask) * static_cast<size_t>(fa::varlen_max_tasks(batch, heads_q, total_q));
}

// The varlen forward; noalloc = true takes the workspace from the library's
// static scratch instead of the caller (workspace arguments ignored).
static int varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                      const int* cu_seqlens_k, int batch, int64_t total_q, int64_t total_k, int heads_q,
                      int heads_kv, int d_qk, int d_v, int causal, float scale, void* workspace,
                      size_t workspace_bytes, bool noalloc, const fa_options* opts, fa_stream_t stream_) {
  fa_options opt;
  fa_options_default(&opt);
  if (opts) opt = *opts;
  if (opt.tau < 0.f) opt.tau = 8.0f;
  if (opt.timeout_s <= 0.0) opt.timeout_s = 1.0;
  causal = causal ? 1 : 0;

  if (batch < 0 || batch > kVarlenMaxBatch || total_q < 0 || total_k < 0) return FA_ERR_INVALID_ARG;
  int rc = validate_common(heads_q, heads_kv, d_qk, d_v, scale, opt);
  if (rc != FA_OK) return rc;
  if (opt.exp_emu != 0) return FA_ERR_UNSUPPORTED;  // the FMA-pipe exp2 is built for fixed-length batches only
  // so are the debug builds
  if (opt.trace != nullptr || (opt.debug_flags & fa::kDebugChecks) || opt.stagger) return FA_ERR_UNSUPPORTED;
  if (opt.workspace != nullptr) return FA_ERR_INVALID_ARG;  // varlen calls take their workspace as an argument
  if (batch == 0 || total_q == 0) return FA_OK;
  // TMA coordinates (row + 128) and the task count stay inside 32 bits
  const int64_t big = int64_t(1) << 31;
  if (total_q + total_k + 4 * fa::kBM >= big) return FA_ERR_INVALID_ARG;
  const int64_t max_tasks = fa::varlen_max_tasks(batch, heads_q, total_q);
  if (max_tasks >= big) return FA_ERR_INVALID_ARG;
  if (noalloc) {  // the static scratch must hold this call's task list
    if (fa_varlen_workspace_size(batch, heads_q, total_q) > kNoAllocScratchBytes) return FA_ERR_INVALID_ARG;
    workspace = nullptr;
    workspace_bytes = 0;
  }
  if (q == nullptr || o == nullptr || cu_seqlens_q == nullptr || cu_seqlens_k == nullptr ||
      (!noalloc && workspace == nullptr))
    return FA_ERR_INVALID_ARG;
  if (total_k > 0 && (k == nullptr || v == nullptr)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace) ||
      (total_k > 0 && (!aligned16(k) || !aligned16(v))))
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
    return FA_ERR_INVALID_ARG;
  if (!noalloc && workspace_bytes < fa_varlen_workspace_size(batch, heads_q, total_q)) return FA_ERR_INVALID_ARG;
  if (scale == 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d_qk));
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* st = nullptr;
  rc = init_device(dev, &st);
  if (rc != FA_OK) return rc;
  if (noalloc) {
    workspace = st->noalloc_scratch;
    workspace_bytes = kNoAllocScratchBytes;
  }
  if (!is_device_ptr(q, dev) || !is_device_ptr(o, dev) || !is_device_ptr(cu_seqlens_q, dev) ||
      !is_device_ptr(cu_seqlens_k, dev) || !is_device_ptr(workspace, dev) ||
      (total_k > 0 && (!is_device_ptr(k, dev) || !is_device_ptr(v, dev))) ||
      (lse != nullptr && !is_device_ptr(lse, dev)))
    return FA_ERR_INVALID_ARG;

  if (total_k == 0) {  // no key in any sequence: O = 0, lse = -inf
    if (cudaMemsetAsync(o, 0, static_cast<size_t>(total_q) * heads_q * d_v * 2, stream) != cudaSuccess)
      return FA_ERR_CUDA;
    if (lse) {
      fill_f32<<<st->sms * 4, 256, 0, stream>>>(lse, static_cast<int64_t>(heads_q) * total_q, -INFINITY);
      if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    }
    return FA_OK;
  }

  const int idx = kernel_index(d_qk, d_v, causal, kVariantVarlen);
  fa::KernelEntry entry;
  if (idx < 0 || !get_entry(d_qk, d_v, causal, kVariantVarlen, &entry)) return FA_ERR_UNSUPPORTED;
  rc = prepare_kernel(st, &st->kernel_ready[idx], entry);
  if (rc != FA_OK) return rc;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!st->plan_ready) {
      if (cudaFuncSetAttribute(varlen_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(plan_smem_bytes(kVarlenMaxBatch))) != cudaSuccess)
        return FA_ERR_CUDA;
      st->plan_ready = true;
    }
  }

  fa::Params p;
  std::memset(&p, 0, sizeof(p));
  // the fields every sequence shares; lengths travel with each task
  p.prob = fa::make_problem(1, heads_q, heads_kv, 1, 1, d_qk, d_v, causal, st->l2_bytes / 2, opt.pack);
  const int tq = static_cast<int>(total_q), tk = static_cast<int>(total_k);
  if (encode_q_like(&p.tm_q, q, 1, tq, heads_q, d_qk, p.prob.pack) != FA_OK) return FA_ERR_CUDA;
  if (encode_kv(&p.tm_k, k, 1, tk, heads_kv, d_qk) != FA_OK) return FA_ERR_CUDA;
  if (encode_kv(&p.tm_v, v, 1, tk, heads_kv, d_v) != FA_OK) return FA_ERR_CUDA;
  if (encode_q_like(&p.tm_o, o, 1, tq, heads_q, d_v, p.prob.pack) != FA_OK) return FA_ERR_CUDA;
  p.lse = lse;
  p.lse_hstride = total_q;
  p.lse_bstride = 0;
  p.o = static_cast<uint16_t*>(o);
  p.o_row_stride = static_cast<int64_t>(heads_q) * d_v;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 ? 1 : 0;
  int* count = static_cast<int*>(workspace);
  fa::VarlenTask* tasks =
      reinterpret_cast<fa::VarlenTask*>(static_cast<uint8_t*>(workspace) + kVarlenHeaderBytes);
  p.vtasks = tasks;
  p.vtask_count = count;
  p.sched_next = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + kVarlenCounterOffset);
  p.status = st->status;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.tau = opt.tau;
  p.timeout_ns = static_cast<unsigned long long>(opt.timeout_s * 1e9);
  p.debug_flags = opt.debug_flags;

  const int64_t capacity = static_cast<int64_t>((workspace_bytes - kVarlenHeaderBytes) / sizeof(fa::VarlenTask));
  varlen_plan_kernel<<<1, kPlanThreads, plan_smem_bytes(batch), stream>>>(
      cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, p.prob, d_qk, d_v, st->l2_bytes / 2, tasks, count,
      p.sched_next, capacity < max_tasks ? capacity : max_tasks, st->status);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;

  int64_t grid = opt.grid > 0 ? opt.grid : st->sms;
  if (grid > max_tasks) grid = max_tasks;
  if (entry.launch(p, static_cast<int>(grid), stream) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

int fa_fwd_varlen_ex(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                     const int* cu_seqlens_k, int batch, int64_t total_q, int64_t total_k, int heads_q,
                     int heads_kv, int d_qk, int d_v, int causal, float scale, void* workspace,
                     size_t workspace_bytes, const fa_options* opts, fa_stream_t stream) {
  return varlen_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, heads_q, heads_kv, d_qk,
                    d_v, causal, scale, workspace, workspace_bytes, false, opts, stream);
}

int fa_fwd_varlen_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int64_t total_q,
                          int64_t total_k, int heads_q, int heads_kv, int d_qk, int d_v, int causal, float scale,
                          fa_stream_t stream) {
  return varlen_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, heads_q, heads_kv, d_qk,
                    d_v, causal, scale, nullptr, 0, true, nullptr, stream);
}

size_t fa_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int batch, int64_t total_q, int64_t total_k, int heads_q, int heads_kv,
                  int d_qk, int d_v, int causal, float scale, void* workspace, size_t workspace_bytes,
                  fa_stream_t stream) {
  return fa_fwd_varlen_ex(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, heads_q, heads_kv,
                          d_qk, d_v, causal, scale, workspace, workspace_bytes, nullptr, stream);
}

int fa_varlen_plan_host(const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int heads_q, int heads_kv,
                        int d_qk, int d_v, int causal, int64_t l2_bytes, int pack, fa_varlen_task* out,
                        int64_t capacity, int64_t* count) {
  if (count == nullptr || batch < 0 || batch > kVarlenMaxBatch || capacity < 0) return FA_ERR_INVALID_ARG;
  if (batch > 0 && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)) return FA_ERR_INVALID_ARG;
  fa_options opt;
  fa_options_default(&opt);
  opt.pack = pack;
  const int rc = validate_common(heads_q, heads_kv, d_qk, d_v, 1.f, opt);
  if (rc != FA_OK) return rc;
  if (l2_bytes <= 0) l2_bytes = int64_t(64) << 20;
  for (int i = 0; i < batch; ++i)
    if (cu_seqlens_q[i] < 0 || cu_seqlens_q[i + 1] < cu_seqlens_q[i] || cu_seqlens_k[i] < 0 ||
        cu_seqlens_k[i + 1] < cu_seqlens_k[i])
      return FA_ERR_INVALID_ARG;
  const fa::Problem base = fa::make_problem(1, heads_q, heads_kv, 1, 1, d_qk, d_v, causal ? 1 : 0, l2_bytes, pack);
  std::vector<uint64_t> vals(static_cast<size_t>(batch));
  for (int i = 0; i < batch; ++i)
    vals[i] = fa::varlen_sort_value(
        fa::varlen_key(cu_seqlens_q[i + 1] - cu_seqlens_q[i], cu_seqlens_k[i + 1] - cu_seqlens_k[i]), i);
  std::sort(vals.begin(), vals.end(), [](uint64_t a, uint64_t b) { return a > b; });
  int64_t n = 0;
  for (int pos = 0; pos < batch; ++pos) {
    const int b = fa::varlen_sort_index(vals[pos]);
    const int q0 = cu_seqlens_q[b], k0 = cu_seqlens_k[b];
    const int sq = cu_seqlens_q[b + 1] - q0, sk = cu_seqlens_k[b + 1] - k0;
    if (sq == 0) continue;
    const fa::Problem seq = fa::varlen_sequence_problem(base, sq, sk, d_qk, d_v, l2_bytes);
    for (int64_t i = 0; i < seq.num_tasks; ++i, ++n) {
      if (out == nullptr || n >= capacity) continue;
      const fa::VarlenTask r = fa::varlen_record(seq, b, q0, k0, static_cast<int>(i));
      out[n].b = r.b, out[n].g = r.g, out[n].mblock = r.mb, out[n].reserved = 0;
      out[n].q_row0 = r.q_row0, out[n].seqlen_q = r.sq, out[n].k_row0 = r.k_row0, out[n].seqlen_k = r.sk;
    }
  }
  *count = n;
  return FA_OK;
}

size_t fa_bwd_workspace_size(int batch, int heads_q, int seqlen_q) {
  if (batch < 0 || heads_q < 1 || seqlen_q < 0) return 0;
  const int64_t sq_pad = (static_cast<int64_t>(seqlen_q) + fa::kBM - 1) / fa::kBM * fa::kBM;
  return static_cast<size_t>(2) * batch * heads_q * sq_pad * sizeof(float);
}

int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
              void* dq, void* dk, void* dv, int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k,
              int d_qk, int d_v, int causal, float scale, void* workspace, size_t workspace_bytes,
              const fa_options* opts, fa_stream_t stream_) {
  fa_options opt;
  fa_options_default(&opt);
  if (opts) opt = *opts;
  if (opt.timeout_s <= 0.0) opt.timeout_s = 1.0;
  causal = causal ? 1 : 0;
  if (batch < 0 || seqlen_q < 0 || seqlen_k < 0 || heads_q < 1 || heads_kv < 1 || heads_q % heads_kv)
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (opt.grid < 0 || !std::isfinite(opt.timeout_s) || opt.timeout_s > 3600.0) return FA_ERR_INVALID_ARG;
  if ((opt.debug_flags & ~fa::kDebugSkipPArrive) != 0) return FA_ERR_INVALID_ARG;
  if (opt.exp_emu != 0 || opt.workspace != nullptr || opt.pack > 1 || opt.stagger) return FA_ERR_UNSUPPORTED;
  const bool trace = opt.trace != nullptr;
  if (trace && (opt.trace_ctas < 1 || opt.trace_cap < 1 || (reinterpret_cast<uintptr_t>(opt.trace) & 7u) != 0))
    return FA_ERR_INVALID_ARG;
  const int pair = (d_qk == 64 && d_v == 64) ? 0 : ((d_qk == 128 && d_v == 128) ? 1 : ((d_qk == 192 && d_v == 128) ? 2 : -1));
  if (pair < 0) return FA_ERR_UNSUPPORTED;
  if (trace && pair != 1) return FA_ERR_UNSUPPORTED;  // the event-log build is (128, 128) only
  if (batch == 0) return FA_OK;
  const int64_t big = int64_t(1) << 31;
  if (static_cast<int64_t>(seqlen_q) + seqlen_k + 4 * fa::kBM >= big) return FA_ERR_INVALID_ARG;
  const bool any_q = seqlen_q > 0, any_k = seqlen_k > 0;
  if ((any_q && (q == nullptr || o == nullptr || lse == nullptr || dout == nullptr || dq == nullptr)) ||
      (any_k && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr)))
    return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return FA_ERR_INVALID_ARG;
  if (any_q && any_k && (workspace == nullptr || workspace_bytes < fa_bwd_workspace_size(batch, heads_q, seqlen_q)))
    return FA_ERR_INVALID_ARG;
  if (scale == 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d_qk));
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* st = nullptr;
  int rc = init_device(dev, &st);
  if (rc != FA_OK) return rc;
  auto dev_ok = [&](const void* ptr) { return ptr == nullptr || is_device_ptr(ptr, dev); };
  if (!dev_ok(q) || !dev_ok(k) || !dev_ok(v) || !dev_ok(o) || !dev_ok(lse) || !dev_ok(dout) || !dev_ok(dq) ||
      !dev_ok(dk) || !dev_ok(dv) || !dev_ok(workspace) || !dev_ok(opt.trace))
    return FA_ERR_INVALID_ARG;

  // degenerate shapes: no query (dK = dV = 0) or no key (dQ = 0)
  if (!any_q || !any_k) {
    if (any_k) {
      const size_t rows = static_cast<size_t>(batch) * seqlen_k * heads_kv;
      if (cudaMemsetAsync(dk, 0, rows * d_qk * 2, stream) != cudaSuccess ||
          cudaMemsetAsync(dv, 0, rows * d_v * 2, stream) != cudaSuccess)
        return FA_ERR_CUDA;
    }
    if (any_q) {
      const size_t bytes = static_cast<size_t>(batch) * seqlen_q * heads_q * d_qk * 2;
      if (cudaMemsetAsync(dq, 0, bytes, stream) != cudaSuccess) return FA_ERR_CUDA;
    }
    return FA_OK;
  }

  fa::BwdEntry ent[2];
  for (int kind = 0; kind < 2; ++kind) {
    const bool found = trace ? fa::bwd_trace_entry(d_qk, d_v, kind, causal, &ent[kind])
                             : fa::bwd_entry(d_qk, d_v, kind, causal, &ent[kind]);
    if (!found) return FA_ERR_UNSUPPORTED;
    bool& ready = trace ? st->bwd_trace_ready[kind * 2 + causal] : st->bwd_ready[(pair * 2 + kind) * 2 + causal];
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!ready) {
      if (ent[kind].smem > st->smem_optin) return FA_ERR_UNSUPPORTED;
      if (cudaFuncSetAttribute(ent[kind].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ent[kind].smem) !=
          cudaSuccess)
        return FA_ERR_CUDA;
      ready = true;
    }
  }

  const int sq_pad = (seqlen_q + fa::kBM - 1) / fa::kBM * fa::kBM;
  float* l2 = static_cast<float*>(workspace);
  float* dvec = l2 + static_cast<int64_t>(batch) * heads_q * sq_pad;
  if (fa::launch_bwd_prep(d_v, o, dout, lse, l2, dvec, batch, heads_q, seqlen_q, sq_pad, st->sms * 16, stream) !=
      cudaSuccess)
    return FA_ERR_CUDA;

  const int ratio = heads_q / heads_kv;
  const int64_t l2_budget = st->l2_bytes / 2;
  for (int kind = 0; kind < 2; ++kind) {
    fa::BwdParams p;
    std::memset(&p, 0, sizeof(p));
    const bool kv = kind == fa::kBwdDkDv;
    // resident / streamed tiles: K, V with Q, dO streamed (dK/dV); Q, dO with K, V streamed (dQ)
    const void* r0 = kv ? k : q;
    const void* r1 = kv ? v : dout;
    const void* t0 = kv ? q : k;
    const void* t1 = kv ? dout : v;
    const int hr = kv ? heads_kv : heads_q, sr = kv ? seqlen_k : seqlen_q;
    const int ht = kv ? heads_q : heads_kv, stt = kv ? seqlen_q : seqlen_k;
    // streamed tiles travel as 64-row halves (one per stage); R0 / T0 (K, Q)
    // have d_qk columns, R1 / T1 (V, dO) d_v
    if (encode_kv(&p.tm_r0, r0, batch, sr, hr, d_qk) != FA_OK || encode_kv(&p.tm_r1, r1, batch, sr, hr, d_v) != FA_OK ||
        encode_kv(&p.tm_t0, t0, batch, stt, ht, d_qk, 64) != FA_OK ||
        encode_kv(&p.tm_t1, t1, batch, stt, ht, d_v, 64) != FA_OK)
      return FA_ERR_CUDA;
    p.l2 = l2;
    p.dvec = dvec;
    p.out0 = static_cast<uint16_t*>(kv ? dv : dq);
    p.out1 = static_cast<uint16_t*>(kv ? dk : nullptr);
    p.status = st->status;
    p.B = batch, p.Hq = heads_q, p.Hkv = heads_kv, p.Sq = seqlen_q, p.Sk = seqlen_k, p.sq_pad = sq_pad;
    p.vec_hstride = sq_pad;
    p.ratio = ratio, p.causal = causal;
    p.mq = (seqlen_q + fa::kBM - 1) / fa::kBM;
    p.nk = (seqlen_k + fa::kBN - 1) / fa::kBN;
    p.units = batch * hr;
    p.blocks = kv ? p.nk : p.mq;
    // causal sections: units whose streamed tiles fit in half the L2 together
    const int64_t streamed = static_cast<int64_t>(stt) * (d_qk + d_v) * 2 * (kv ? ratio : 1);
    int64_t su = streamed > 0 ? l2_budget / streamed : 1;
    if (su < 1) su = 1;
    if (su > p.units) su = p.units;
    p.section_units = static_cast<int>(su);
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.timeout_ns = static_cast<unsigned long long>(opt.timeout_s * 1e9);
    p.debug_flags = opt.debug_flags;
    if (trace) {  // the dK/dV kernel's log first, then the dQ kernel's
      p.trace = opt.trace + static_cast<int64_t>(kind) * opt.trace_ctas * fa::kTraceTracks * (opt.trace_cap + 1);
      p.trace_ctas = opt.trace_ctas;
      p.trace_cap = opt.trace_cap;
    }
    const int64_t tasks = static_cast<int64_t>(p.units) * p.blocks;
    if (tasks >= big) return FA_ERR_INVALID_ARG;
    int64_t grid = opt.grid > 0 ? opt.grid : st->sms;
    if (grid > tasks) grid = tasks;
    // paired causal order: heavy and light blocks of a unit on one CTA
    p.pair_grid = p.pair_body = p.pair_r = 0;
    if (causal && !opt.no_balance && p.blocks >= 2 && p.blocks % 2 == 0 && grid >= 2) {
      const int64_t pairs = tasks / 2;
      p.pair_grid = static_cast<int>(grid);
      p.pair_body = static_cast<int>(2 * (pairs / grid) * grid);
      p.pair_r = static_cast<int>(pairs % grid);
    }
    if (ent[kind].launch(p, static_cast<int>(grid), stream) != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
           void* dk, void* dv, int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v,
           int causal, float scale, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return fa_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal,
                   scale, workspace, workspace_bytes, nullptr, stream);
}

// ---------------------------------------------------------------------------
// backward of a variable-length batch
// ---------------------------------------------------------------------------
namespace {

// Workspace of fa_bwd_varlen: a 256-byte header (the two task counts), the
// dK/dV and dQ task records at their upper bounds, then the l2 and dvec
// vectors [Hq, pad_stride] (each sequence's rows padded to 128).
struct BwdVarlenLayout {
  int64_t kv_cap = 0, q_cap = 0, pad_stride = 0;
  size_t off_kv = 0, off_q = 0, off_l2 = 0, off_dvec = 0, bytes = 0;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

bool bwd_varlen_layout(int batch, int heads_q, int heads_kv, int64_t total_q, int64_t total_k, BwdVarlenLayout* L) {
  if (batch < 0 || heads_q < 1 || heads_kv < 1 || total_q < 0 || total_k < 0) return false;
  const int64_t big = int64_t(1) << 31;
  if (total_q >= big || total_k >= big) return false;
  const int64_t qb = (total_q + fa::kBM - 1) / fa::kBM + batch, kb = (total_k + fa::kBN - 1) / fa::kBN + batch;
  L->kv_cap = heads_kv * kb;
  L->q_cap = heads_q * qb;
  L->pad_stride = fa::kBM * qb;
  if (L->kv_cap >= big || L->q_cap >= big || L->pad_stride * heads_q >= big) return false;
  const size_t rec = sizeof(fa::VarlenTask);
  L->off_kv = 256;
  L->off_q = L->off_kv + static_cast<size_t>(L->kv_cap) * rec;
  L->off_l2 = align256(L->off_q + static_cast<size_t>(L->q_cap) * rec);
  const size_t vec = static_cast<size_t>(heads_q) * L->pad_stride * sizeof(float);
  L->off_dvec = align256(L->off_l2 + vec);
  L->bytes = L->off_dvec + vec;
  return true;
}

}  // namespace

size_t fa_bwd_varlen_workspace_size(int batch, int heads_q, int heads_kv, int64_t total_q, int64_t total_k) {
  BwdVarlenLayout L;
  return bwd_varlen_layout(batch, heads_q, heads_kv, total_q, total_k, &L) ? L.bytes : 0;
}

int fa_bwd_varlen_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                     int64_t total_q, int64_t total_k, int heads_q, int heads_kv, int d_qk, int d_v, int causal,
                     float scale, void* workspace, size_t workspace_bytes, const fa_options* opts,
                     fa_stream_t stream_) {
  fa_options opt;
  fa_options_default(&opt);
  if (opts) opt = *opts;
  if (opt.timeout_s <= 0.0) opt.timeout_s = 1.0;
  causal = causal ? 1 : 0;
  if (batch < 0 || batch > fa::kVarlenPlanMaxBatch || heads_q < 1 || heads_kv < 1 || heads_q % heads_kv)
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (opt.grid < 0 || !std::isfinite(opt.timeout_s) || opt.timeout_s > 3600.0) return FA_ERR_INVALID_ARG;
  if ((opt.debug_flags & ~fa::kDebugSkipPArrive) != 0) return FA_ERR_INVALID_ARG;
  if (opt.exp_emu != 0 || opt.workspace != nullptr || opt.pack > 1 || opt.stagger || opt.trace != nullptr)
    return FA_ERR_UNSUPPORTED;
  const int pair = (d_qk == 64 && d_v == 64) ? 0 : ((d_qk == 128 && d_v == 128) ? 1 : ((d_qk == 192 && d_v == 128) ? 2 : -1));
  if (pair < 0) return FA_ERR_UNSUPPORTED;
  BwdVarlenLayout L;
  if (!bwd_varlen_layout(batch, heads_q, heads_kv, total_q, total_k, &L)) return FA_ERR_INVALID_ARG;
  if (batch == 0) return FA_OK;
  const bool any_q = total_q > 0, any_k = total_k > 0;
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return FA_ERR_INVALID_ARG;
  if ((any_q && (q == nullptr || o == nullptr || lse == nullptr || dout == nullptr || dq == nullptr)) ||
      (any_k && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr)))
    return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) != 0 || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u) != 0)
    return FA_ERR_INVALID_ARG;
  if (any_q && any_k && (workspace == nullptr || workspace_bytes < L.bytes)) return FA_ERR_INVALID_ARG;
  if (scale == 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d_qk));
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* st = nullptr;
  int rc = init_device(dev, &st);
  if (rc != FA_OK) return rc;
  auto dev_ok = [&](const void* ptr) { return ptr == nullptr || is_device_ptr(ptr, dev); };
  if (!dev_ok(q) || !dev_ok(k) || !dev_ok(v) || !dev_ok(o) || !dev_ok(lse) || !dev_ok(dout) || !dev_ok(dq) ||
      !dev_ok(dk) || !dev_ok(dv) || !dev_ok(workspace) || !dev_ok(cu_seqlens_q) || !dev_ok(cu_seqlens_k))
    return FA_ERR_INVALID_ARG;

  // no query anywhere: dK = dV = 0; no key anywhere: dQ = 0 (whole tensors)
  if (!any_q || !any_k) {
    if (any_k) {
      const size_t rows = static_cast<size_t>(total_k) * heads_kv;
      if (cudaMemsetAsync(dk, 0, rows * d_qk * 2, stream) != cudaSuccess ||
          cudaMemsetAsync(dv, 0, rows * d_v * 2, stream) != cudaSuccess)
        return FA_ERR_CUDA;
    }
    if (any_q && cudaMemsetAsync(dq, 0, static_cast<size_t>(total_q) * heads_q * d_qk * 2, stream) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_OK;
  }

  fa::BwdEntry ent[2];
  for (int kind = 0; kind < 2; ++kind) {
    if (!fa::bwd_varlen_entry(d_qk, d_v, kind, causal, &ent[kind])) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    bool& ready = st->bwd_varlen_ready[(pair * 2 + kind) * 2 + causal];
    if (!ready) {
      if (ent[kind].smem > st->smem_optin) return FA_ERR_UNSUPPORTED;
      if (cudaFuncSetAttribute(ent[kind].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ent[kind].smem) !=
          cudaSuccess)
        return FA_ERR_CUDA;
      ready = true;
    }
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* counts = reinterpret_cast<int*>(ws);
  fa::VarlenTask* kv_tasks = reinterpret_cast<fa::VarlenTask*>(ws + L.off_kv);
  fa::VarlenTask* q_tasks = reinterpret_cast<fa::VarlenTask*>(ws + L.off_q);
  float* l2 = reinterpret_cast<float*>(ws + L.off_l2);
  float* dvec = reinterpret_cast<float*>(ws + L.off_dvec);
  {
    std::lock_guard<std::mutex> lock(g_mutex);  // the planner's first call sets its shared-memory attribute
    if (fa::launch_bwd_varlen_plan(cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, heads_q, heads_kv, causal,
                                   kv_tasks, q_tasks, counts, st->status, &st->bwd_plan_ready, stream) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  const int pad_stride = static_cast<int>(L.pad_stride);
  if (fa::launch_bwd_prep_varlen(d_v, o, dout, lse, l2, dvec, q_tasks, counts + 1, heads_q, total_q, pad_stride,
                                 st->sms * 16, stream) != cudaSuccess)
    return FA_ERR_CUDA;

  const int tq = static_cast<int>(total_q), tk = static_cast<int>(total_k);
  for (int kind = 0; kind < 2; ++kind) {
    fa::BwdParams p;
    std::memset(&p, 0, sizeof(p));
    const bool kv = kind == fa::kBwdDkDv;
    const void* r0 = kv ? k : q;
    const void* r1 = kv ? v : dout;
    const void* t0 = kv ? q : k;
    const void* t1 = kv ? dout : v;
    const int hr = kv ? heads_kv : heads_q, sr = kv ? tk : tq;
    const int ht = kv ? heads_q : heads_kv, stt = kv ? tq : tk;
    if (encode_kv(&p.tm_r0, r0, 1, sr, hr, d_qk) != FA_OK || encode_kv(&p.tm_r1, r1, 1, sr, hr, d_v) != FA_OK ||
        encode_kv(&p.tm_t0, t0, 1, stt, ht, d_qk, 64) != FA_OK || encode_kv(&p.tm_t1, t1, 1, stt, ht, d_v, 64) != FA_OK)
      return FA_ERR_CUDA;
    p.l2 = l2;
    p.dvec = dvec;
    p.out0 = static_cast<uint16_t*>(kv ? dv : dq);
    p.out1 = static_cast<uint16_t*>(kv ? dk : nullptr);
    p.status = st->status;
    p.B = 1, p.Hq = heads_q, p.Hkv = heads_kv;
    p.ratio = heads_q / heads_kv, p.causal = causal;
    p.section_units = 1;
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.timeout_ns = static_cast<unsigned long long>(opt.timeout_s * 1e9);
    p.debug_flags = opt.debug_flags;
    p.vec_hstride = pad_stride;
    p.vtasks = kv ? kv_tasks : q_tasks;
    p.vcount = counts + kind;
    const int grid = opt.grid > 0 ? opt.grid : st->sms;
    if (ent[kind].launch(p, grid, stream) != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                  int64_t total_q, int64_t total_k, int heads_q, int heads_kv, int d_qk, int d_v, int causal,
                  float scale, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return fa_bwd_varlen_ex(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                          heads_q, heads_kv, d_qk, d_v, causal, scale, workspace, workspace_bytes, nullptr, stream);
}

int fa_device_status(fa_stream_t stream, int* out) { return fa_device_status_detail(stream, out, nullptr); }

int fa_device_status_detail(fa_stream_t stream, int* out, unsigned int detail[3]) {
  if (out == nullptr) return FA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* st = nullptr;
  int rc = init_device(dev, &st);
  if (rc != FA_OK) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int w[4] = {0, 0, 0, 0};
  if (cudaMemcpy(w, st->status, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemset(st->status, 0, sizeof(w)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  *out = w[0] == 0 ? FA_OK
                   : (w[0] == fa::kStatusTimeout ? FA_ERR_DEVICE_TIMEOUT
                                                 : (w[0] == fa::kStatusCheck ? FA_ERR_DEVICE_CHECK
                                                                             : static_cast<int>(w[0])));
  if (detail) {
    detail[0] = w[0];
    detail[1] = w[1];
    detail[2] = w[2];
  }
  return FA_OK;
}

int fa_debug_rescale_count(fa_stream_t stream, unsigned int* out) {
  if (out == nullptr) return FA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* st = nullptr;
  int rc = init_device(dev, &st);
  if (rc != FA_OK) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpy(out, st->status + 3, sizeof(unsigned int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemset(st->status + 3, 0, sizeof(unsigned int)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

int fa_selftest_exp2(const float* x, float* y_fma, float* y_mufu, int n, fa_stream_t stream) {
  if (n < 0 || (n > 0 && (x == nullptr || y_fma == nullptr || y_mufu == nullptr))) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* st = nullptr;
  const int rc = init_device(dev, &st);
  if (rc != FA_OK) return rc;
  if (!is_device_ptr(x, dev) || !is_device_ptr(y_fma, dev) || !is_device_ptr(y_mufu, dev)) return FA_ERR_INVALID_ARG;
  const int pairs = (n + 1) / 2;
  exp2_selftest_kernel<<<(pairs + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(x, y_fma, y_mufu, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_make_plan(int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal,
                 int64_t l2_bytes, int pack, fa_plan* out) {
  if (out == nullptr) return FA_ERR_INVALID_ARG;
  if (batch < 0 || seqlen_q < 0 || seqlen_k < 0 || heads_q < 1 || heads_kv < 1 || heads_q % heads_kv)
    return FA_ERR_INVALID_ARG;
  if (kernel_index(d_qk, d_v, 0, 0) < 0) return FA_ERR_UNSUPPORTED;
  if (pack < 0 || (pack > 0 && (fa::kBM % pack != 0 || (heads_q / heads_kv) % pack != 0))) return FA_ERR_INVALID_ARG;
  if (l2_bytes <= 0) l2_bytes = fa::kCausalSectionBytes;  // what fa_fwd uses on an L2 of 16 MiB or more
  const fa::Problem p =
      fa::make_problem(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal ? 1 : 0, l2_bytes, pack);
  out->batch = p.B, out->heads_q = p.Hq, out->heads_kv = p.Hkv, out->seqlen_q = p.Sq, out->seqlen_k = p.Sk;
  out->causal = p.causal, out->pack = p.pack, out->groups = p.groups, out->pos_per_tile = p.pos_per_tile;
  out->tiles = p.tiles, out->mblocks = p.mblocks, out->kv_blocks = p.kv_blocks, out->ratio = p.ratio;
  out->section_units = p.section_units, out->heavy_levels = p.heavy_levels, out->num_tasks = p.num_tasks;
  out->tail_first = p.tail_first;
  out->grid = 0;
  return FA_OK;
}

static fa::Problem problem_of(const fa_plan* pl) {
  fa::Problem p{};
  p.B = pl->batch, p.Hq = pl->heads_q, p.Hkv = pl->heads_kv, p.Sq = pl->seqlen_q, p.Sk = pl->seqlen_k;
  p.causal = pl->causal, p.pack = pl->pack, p.groups = pl->groups, p.pos_per_tile = pl->pos_per_tile;
  p.tiles = pl->tiles, p.mblocks = pl->mblocks, p.kv_blocks = pl->kv_blocks, p.ratio = pl->ratio;
  p.section_units = pl->section_units, p.heavy_levels = pl->heavy_levels;
  p.num_tasks = static_cast<int64_t>(pl->batch) * pl->groups * pl->mblocks;  // the plain order
  p.tail_first = p.num_tasks;
  p.splits = 1, p.split_blocks = pl->kv_blocks;
  fa::set_divisors(p);
  if (pl->grid > 0) fa::set_balance(p, pl->grid);
  return p;
}

int fa_plan_set_grid(fa_plan* plan, int grid) {
  if (plan == nullptr || grid < 1 || plan->grid != 0) return FA_ERR_INVALID_ARG;
  plan->grid = grid;
  const fa::Problem p = problem_of(plan);
  plan->num_tasks = p.num_tasks;
  plan->tail_first = p.tail_first;
  return FA_OK;
}

int fa_plan_task(const fa_plan* plan, int64_t task, fa_task* out) {
  if (plan == nullptr || out == nullptr || task < 0 || task >= plan->num_tasks) return FA_ERR_INVALID_ARG;
  const fa::Task t = fa::decode_task(problem_of(plan), task);
  out->b = t.b, out->g = t.g, out->mblock = t.mb, out->kv_head = t.kvh;
  for (int s = 0; s < 2; ++s) out->pos0[s] = t.pos0[s], out->n_blocks[s] = t.n[s];
  out->key_split = t.ksplit;
  return FA_OK;
}

int fa_plan_block_masked(const fa_plan* plan, int pos0, int j) {
  if (plan == nullptr) return 0;
  return fa::block_needs_mask(problem_of(plan), pos0, j) ? 1 : 0;
}

int fa_plan_first_masked_block(const fa_plan* plan, int pos0) {
  if (plan == nullptr) return 0;
  return fa::first_masked_block(plan->seqlen_k, plan->seqlen_k - plan->seqlen_q, plan->causal, pos0);
}

}  // extern "C"
