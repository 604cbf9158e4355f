// The variable-length build of the attention backward kernels: task
// records from the planning kernel instead of the fixed-length grid, packed
// (total rows, heads, d) tensors, per-sequence lengths and masks.  Head dims
// (64, 64), (128, 128) and (192, 128).
#include <climits>

#include "fa.h"
#include "fa_bwd_dispatch.h"

namespace fa {

template <int DQ, int DV>
static BwdEntry pick_bwd_varlen(int kind, int causal) {
  if (kind == kBwdDkDv)
    return causal ? make_bwd_entry<DQ, DV, kBwdDkDv, true, kBwdVarlen>()
                  : make_bwd_entry<DQ, DV, kBwdDkDv, false, kBwdVarlen>();
  return causal ? make_bwd_entry<DQ, DV, kBwdDq, true, kBwdVarlen>()
                : make_bwd_entry<DQ, DV, kBwdDq, false, kBwdVarlen>();
}

bool bwd_varlen_entry(int dq, int dv, int kind, int causal, BwdEntry* out) {
  if (kind != kBwdDkDv && kind != kBwdDq) return false;
  if (dq == 64 && dv == 64) {
    *out = pick_bwd_varlen<64, 64>(kind, causal);
    return true;
  }
  if (dq == 128 && dv == 128) {
    *out = pick_bwd_varlen<128, 128>(kind, causal);
    return true;
  }
  if (dq == 192 && dv == 128) {
    *out = pick_bwd_varlen<192, 128>(kind, causal);
    return true;
  }
  return false;
}

cudaError_t launch_bwd_prep_varlen(int dv, const void* o, const void* dout, const float* lse, float* l2, float* dvec,
                                   const VarlenTask* dq_tasks, const int* dq_count, int Hq, int64_t total_q,
                                   int vec_hstride, int grid, cudaStream_t stream) {
  const uint16_t* o16 = static_cast<const uint16_t*>(o);
  const uint16_t* g16 = static_cast<const uint16_t*>(dout);
  if (dv == 128)
    fa_bwd_prep_varlen_kernel<128><<<grid, 256, 0, stream>>>(o16, g16, lse, l2, dvec, dq_tasks, dq_count, Hq,
                                                              total_q, vec_hstride);
  else
    fa_bwd_prep_varlen_kernel<64><<<grid, 256, 0, stream>>>(o16, g16, lse, l2, dvec, dq_tasks, dq_count, Hq,
                                                             total_q, vec_hstride);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// planning: one CTA checks cu_seqlens, sorts the sequences by their longest
// side in 128-row blocks (longest first, ties by index: the longest-first
// order of the forward's planner), and writes, in that order, the dK/dV
// tasks (sequence, K/V head, key block) and the dQ tasks (sequence, query
// head, query block) of every sequence, block by block, heaviest first, each record with the sequence's
// padded row offset in the l2 / dvec vectors (sequences in batch order,
// 128-row blocks), first rows and lengths.
// ---------------------------------------------------------------------------
constexpr int kBwdPlanThreads = 1024;
constexpr unsigned int kSiteBwdVarlenSeqlens = 501;  // the forward planner's site for bad cu_seqlens

size_t bwd_varlen_plan_smem_bytes(int batch) {
  int npow2 = 1;
  while (npow2 < batch) npow2 <<= 1;
  return static_cast<size_t>(npow2) * sizeof(uint64_t) + 3 * static_cast<size_t>(batch + 1) * sizeof(int);
}

// exclusive scan of f(i), i in [0, n), into out[0 .. n] (out[n] = the total),
// over one CTA: each thread sums a contiguous run, then the runs are scanned
__device__ __forceinline__ void plan_scan_begin(int n, int& lo, int& hi) {
  const int per = (n + kBwdPlanThreads - 1) / kBwdPlanThreads;
  lo = min(static_cast<int>(threadIdx.x) * per, n);
  hi = min(lo + per, n);
}

template <class F>
__device__ long long plan_exclusive_scan(int n, F f, int* out, long long* warp_sums) {
  int lo, hi;
  plan_scan_begin(n, lo, hi);
  long long mine = 0;
  for (int i = lo; i < hi; ++i) mine += f(i);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = mine;
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
    warp_sums[lane] = w;
  }
  __syncthreads();
  const long long total = warp_sums[kBwdPlanThreads / 32 - 1];
  long long run = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - mine;
  for (int i = lo; i < hi; ++i) {
    out[i] = static_cast<int>(run);
    run += f(i);
  }
  if (threadIdx.x == 0) out[n] = static_cast<int>(total);
  __syncthreads();  // out complete; warp_sums free for the next scan
  return total;
}

__global__ void __launch_bounds__(kBwdPlanThreads) bwd_varlen_plan_kernel(
    const int* cu_q, const int* cu_k, int batch, int64_t total_q, int64_t total_k, int Hq, int Hkv, int causal,
    VarlenTask* kv_tasks, VarlenTask* q_tasks, int* counts, unsigned int* status) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int bad_index;
  __shared__ long long warp_sums[kBwdPlanThreads / 32];
  int npow2 = 1;
  while (npow2 < batch) npow2 <<= 1;
  uint64_t* vals = reinterpret_cast<uint64_t*>(smem);
  int* pad_off = reinterpret_cast<int*>(vals + npow2);  // [batch + 1], batch order
  int* kv_start = pad_off + (batch + 1);                 // [batch + 1], sorted order
  int* q_start = kv_start + (batch + 1);
  const int tid = threadIdx.x;
  if (tid == 0) bad_index = INT_MAX;
  __syncthreads();
  for (int i = tid; i < npow2; i += kBwdPlanThreads) {
    uint64_t v = 0;  // padding sorts after every sequence
    if (i < batch) {
      const int q0 = cu_q[i], q1 = cu_q[i + 1], k0 = cu_k[i], k1 = cu_k[i + 1];
      if (q0 < 0 || q1 < q0 || q1 > total_q || k0 < 0 || k1 < k0 || k1 > total_k) atomicMin(&bad_index, i);
      const int key = max((q1 - q0 + kBM - 1) / kBM, (k1 - k0 + kBN - 1) / kBN);
      v = varlen_sort_value(key, i);
    }
    vals[i] = v;
  }
  __syncthreads();
  if (bad_index != INT_MAX) {
    if (tid == 0) {
      counts[0] = counts[1] = 0;
      if (atomicCAS(&status[0], 0u, static_cast<unsigned int>(FA_ERR_INVALID_ARG)) == 0u) {
        status[1] = kSiteBwdVarlenSeqlens;
        status[2] = static_cast<unsigned int>(bad_index);
      }
    }
    return;
  }
  for (int k = 2; k <= npow2; k <<= 1) {  // bitonic sort, descending
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < npow2; i += kBwdPlanThreads) {
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
  auto sq_of = [&](int b) { return cu_q[b + 1] - cu_q[b]; };
  auto sk_of = [&](int b) { return cu_k[b + 1] - cu_k[b]; };
  plan_exclusive_scan(batch, [&](int b) -> long long { return static_cast<long long>(kBM) * ((sq_of(b) + kBM - 1) / kBM); },
                      pad_off, warp_sums);
  const long long n_kv = plan_exclusive_scan(
      batch,
      [&](int pos) -> long long {
        const int b = varlen_sort_index(vals[pos]);
        return static_cast<long long>(Hkv) * ((sk_of(b) + kBN - 1) / kBN);
      },
      kv_start, warp_sums);
  const long long n_q = plan_exclusive_scan(
      batch,
      [&](int pos) -> long long {
        const int b = varlen_sort_index(vals[pos]);
        return static_cast<long long>(Hq) * ((sq_of(b) + kBM - 1) / kBM);
      },
      q_start, warp_sums);
  // task t belongs to the last sorted position whose first task is <= t
  auto find = [&](const int* start, int t) {
    int a = 0, z = batch - 1;
    while (a < z) {
      const int mid = (a + z + 1) >> 1;
      if (start[mid] <= t) a = mid;
      else z = mid - 1;
    }
    return a;
  };
  for (int kind = 0; kind < 2; ++kind) {
    const int* start = kind == 0 ? kv_start : q_start;
    VarlenTask* out = kind == 0 ? kv_tasks : q_tasks;
    const int n = static_cast<int>(kind == 0 ? n_kv : n_q);
    for (int t = tid; t < n; t += kBwdPlanThreads) {
      const int pos = find(start, t);
      const int b = varlen_sort_index(vals[pos]);
      const int sq = sq_of(b), sk = sk_of(b);
      const int nblk = kind == 0 ? (sk + kBN - 1) / kBN : (sq + kBM - 1) / kBM;
      // block-major inside a sequence, heaviest block first (under the
      // mask: the first key blocks for dK/dV, the last query blocks for dQ),
      // so that round-robin over the list deals each CTA a similar load
      const int H = kind == 0 ? Hkv : Hq;
      const int i = t - start[pos];
      const int j = i / H;
      VarlenTask r;
      r.b = b, r.g = i - j * H, r.mb = (kind == 1 && causal) ? nblk - 1 - j : j, r.reserved = pad_off[b];
      r.q_row0 = cu_q[b], r.sq = sq, r.k_row0 = cu_k[b], r.sk = sk;
      out[t] = r;
    }
  }
  if (tid == 0) {
    counts[0] = static_cast<int>(n_kv);
    counts[1] = static_cast<int>(n_q);
  }
}

cudaError_t launch_bwd_varlen_plan(const int* cu_q, const int* cu_k, int batch, int64_t total_q, int64_t total_k,
                                   int Hq, int Hkv, int causal, VarlenTask* kv_tasks, VarlenTask* q_tasks, int* counts,
                                   unsigned int* status, bool* attr_ready, cudaStream_t stream) {
  const size_t smem = bwd_varlen_plan_smem_bytes(batch);
  if (!*attr_ready) {  // once per device (the caller holds the library's lock)
    const cudaError_t e = cudaFuncSetAttribute(bwd_varlen_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(bwd_varlen_plan_smem_bytes(kVarlenPlanMaxBatch)));
    if (e != cudaSuccess) return e;
    *attr_ready = true;
  }
  bwd_varlen_plan_kernel<<<1, kBwdPlanThreads, smem, stream>>>(cu_q, cu_k, batch, total_q, total_k, Hq, Hkv,
                                                               causal, kv_tasks, q_tasks, counts, status);
  return cudaGetLastError();
}

}  // namespace fa
