// C ABI of the attention forward library: argument validation, tensor-map
// construction, launch, and the device status word.  See include/fa.h for
// the contract.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_dispatch.h"
#include "fa_schedule.h"

// {code, wait site, block} of the first device-side failure since the last read
__device__ unsigned int g_fa_status[4];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kNumKernels = 20;  // 5 (d_qk, d_v) pairs x {non-causal, causal} x {MUFU, FMA-emulated exp}

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int64_t l2_bytes = 0;
  int smem_optin = 0;
  unsigned int* status = nullptr;
  bool kernel_ready[kNumKernels] = {};
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int kernel_index(int dq, int dv, int causal, int emu) {
  int pair = -1;
  if (dq == 64 && dv == 64) pair = 0;
  if (dq == 128 && dv == 64) pair = 1;
  if (dq == 128 && dv == 128) pair = 2;
  if (dq == 192 && dv == 64) pair = 3;
  if (dq == 192 && dv == 128) pair = 4;
  return pair < 0 ? -1 : pair * 4 + (causal ? 2 : 0) + (emu ? 1 : 0);
}

bool get_entry(int dq, int dv, int causal, int emu, fa::KernelEntry* e) {
  if (dq == 64) return fa::entry_d64(dv, causal, emu, e);
  if (dq == 128) return fa::entry_d128(dv, causal, emu, e);
  if (dq == 192) return fa::entry_d192(dv, causal, emu, e);
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
int prepare_kernel(DeviceState* st, int idx, const fa::KernelEntry& e) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (st->kernel_ready[idx]) return FA_OK;
  if (e.smem > st->smem_optin) return FA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(e.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, e.smem) != cudaSuccess)
    return FA_ERR_CUDA;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, e.fn) != cudaSuccess) return FA_ERR_CUDA;
  // setmaxnreg.inc would wait forever if the launch left fewer registers than the split needs
  if (attr.numRegs * fa::kThreads < fa::kRegBudgetPerCta || attr.maxThreadsPerBlock < fa::kThreads)
    return FA_ERR_UNSUPPORTED;
  st->kernel_ready[idx] = true;
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
  cuuint64_t strides[4] = {d * e, static_cast<cuuint64_t>(pack) * d * e, static_cast<cuuint64_t>(H) * d * e,
                           static_cast<cuuint64_t>(S) * H * d * e};
  cuuint32_t box[5] = {64, static_cast<cuuint32_t>(pack), 1, static_cast<cuuint32_t>(fa::kBM / pack), 1};
  return encode(m, base, 5, dims, strides, box);
}

// K or V viewed as (d, Hkv, S, B): one box is 128 keys x 64 columns of a head.
int encode_kv(CUtensorMap* m, const void* base, int B, int S, int H, int d) {
  const cuuint64_t e = 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {d * e, static_cast<cuuint64_t>(H) * d * e, static_cast<cuuint64_t>(S) * H * d * e};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(fa::kBN), 1};
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

int validate(const void* q, const void* k, const void* v, void* o, const float* lse, int batch, int heads_q,
             int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, float scale, const fa_options& opt) {
  if (batch < 0 || seqlen_q < 0 || seqlen_k < 0 || heads_q < 1 || heads_kv < 1) return FA_ERR_INVALID_ARG;
  if (heads_q % heads_kv != 0) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale)) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (kernel_index(d_qk, d_v, 0, 0) < 0) return FA_ERR_UNSUPPORTED;
  if (opt.pack < 0 || opt.grid < 0 || (opt.debug_flags & ~fa::kDebugSkipPArrive) != 0) return FA_ERR_INVALID_ARG;
  if (opt.exp_emu != 0 && opt.exp_emu != 1) return FA_ERR_INVALID_ARG;
  // the kept reference may lag the row maximum by up to tau (log2 units), so
  // unnormalised weights reach 2^tau: keep them far inside the fp32 range
  if (!(opt.tau >= 0.f && opt.tau <= 64.f)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(opt.timeout_s) || opt.timeout_s > 3600.0) return FA_ERR_INVALID_ARG;
  if (opt.pack > 0) {
    const int ratio = heads_q / heads_kv;
    if (fa::kBM % opt.pack != 0 || ratio % opt.pack != 0) return FA_ERR_INVALID_ARG;
  }
  if (batch == 0 || seqlen_q == 0) return FA_OK;  // nothing to compute; pointers unused
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
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
    default:
      return "FA_ERR_UNKNOWN";
  }
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
              int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
              const fa_options* opts, fa_stream_t stream_) {
  fa_options opt;
  fa_options_default(&opt);
  if (opts) opt = *opts;
  if (opt.tau < 0.f) opt.tau = 8.0f;
  if (opt.timeout_s <= 0.0) opt.timeout_s = 1.0;
  causal = causal ? 1 : 0;

  int rc = validate(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, scale, opt);
  if (rc != FA_OK) return rc;
  if (batch == 0 || seqlen_q == 0) return FA_OK;
  if (scale == 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d_qk));
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* st = nullptr;
  rc = init_device(dev, &st);
  if (rc != FA_OK) return rc;
  if (!is_device_ptr(q, dev) || !is_device_ptr(k, dev) || !is_device_ptr(v, dev) || !is_device_ptr(o, dev) ||
      (lse != nullptr && !is_device_ptr(lse, dev)))
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

  const int idx = kernel_index(d_qk, d_v, causal, opt.exp_emu);
  fa::KernelEntry entry;
  if (idx < 0 || !get_entry(d_qk, d_v, causal, opt.exp_emu, &entry)) return FA_ERR_UNSUPPORTED;
  rc = prepare_kernel(st, idx, entry);
  if (rc != FA_OK) return rc;

  fa::Params p;
  std::memset(&p, 0, sizeof(p));
  p.prob = fa::make_problem(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, st->l2_bytes / 2,
                            opt.pack);
  if (p.prob.num_tasks >= (int64_t(1) << 31)) return FA_ERR_INVALID_ARG;  // the device decodes tasks in 32 bits
  if (encode_q_like(&p.tm_q, q, batch, seqlen_q, heads_q, d_qk, p.prob.pack) != FA_OK) return FA_ERR_CUDA;
  if (encode_kv(&p.tm_k, k, batch, seqlen_k, heads_kv, d_qk) != FA_OK) return FA_ERR_CUDA;
  if (encode_kv(&p.tm_v, v, batch, seqlen_k, heads_kv, d_v) != FA_OK) return FA_ERR_CUDA;
  if (encode_q_like(&p.tm_o, o, batch, seqlen_q, heads_q, d_v, p.prob.pack) != FA_OK) return FA_ERR_CUDA;
  p.lse = lse;
  p.status = st->status;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.tau = opt.tau;
  p.timeout_ns = static_cast<unsigned long long>(opt.timeout_s * 1e9);
  p.debug_flags = opt.debug_flags;

  int64_t grid = opt.grid > 0 ? opt.grid : st->sms;
  if (grid > p.prob.num_tasks) grid = p.prob.num_tasks;
  if (grid < 1) return FA_OK;
  if (entry.launch(p, static_cast<int>(grid), stream) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q, int heads_kv,
           int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale, fa_stream_t stream) {
  return fa_fwd_ex(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale, nullptr,
                   stream);
}

int fa_device_status(fa_stream_t stream, int* out, unsigned int detail[3]) {
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
  *out = w[0] == 0 ? FA_OK : (w[0] == fa::kStatusTimeout ? FA_ERR_DEVICE_TIMEOUT : static_cast<int>(w[0]));
  if (detail) {
    detail[0] = w[0];
    detail[1] = w[1];
    detail[2] = w[2];
  }
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
  if (l2_bytes <= 0) l2_bytes = int64_t(64) << 20;
  const fa::Problem p =
      fa::make_problem(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal ? 1 : 0, l2_bytes, pack);
  out->batch = p.B, out->heads_q = p.Hq, out->heads_kv = p.Hkv, out->seqlen_q = p.Sq, out->seqlen_k = p.Sk;
  out->causal = p.causal, out->pack = p.pack, out->groups = p.groups, out->pos_per_tile = p.pos_per_tile;
  out->tiles = p.tiles, out->mblocks = p.mblocks, out->kv_blocks = p.kv_blocks, out->ratio = p.ratio;
  out->section_units = p.section_units, out->num_tasks = p.num_tasks;
  return FA_OK;
}

static fa::Problem problem_of(const fa_plan* pl) {
  fa::Problem p;
  p.B = pl->batch, p.Hq = pl->heads_q, p.Hkv = pl->heads_kv, p.Sq = pl->seqlen_q, p.Sk = pl->seqlen_k;
  p.causal = pl->causal, p.pack = pl->pack, p.groups = pl->groups, p.pos_per_tile = pl->pos_per_tile;
  p.tiles = pl->tiles, p.mblocks = pl->mblocks, p.kv_blocks = pl->kv_blocks, p.ratio = pl->ratio;
  p.section_units = pl->section_units, p.num_tasks = pl->num_tasks;
  return p;
}

int fa_plan_task(const fa_plan* plan, int64_t task, fa_task* out) {
  if (plan == nullptr || out == nullptr || task < 0 || task >= plan->num_tasks) return FA_ERR_INVALID_ARG;
  const fa::Task t = fa::decode_task(problem_of(plan), task);
  out->b = t.b, out->g = t.g, out->mblock = t.mb, out->kv_head = t.kvh;
  for (int s = 0; s < 2; ++s) out->pos0[s] = t.pos0[s], out->n_blocks[s] = t.n[s];
  return FA_OK;
}

int fa_plan_block_masked(const fa_plan* plan, int pos0, int j) {
  if (plan == nullptr) return 0;
  return fa::block_needs_mask(problem_of(plan), pos0, j) ? 1 : 0;
}

}  // extern "C"
