// Backward launch table (instantiated in fa_bwd.cu, its own translation unit).
#pragma once
#include <cuda_runtime.h>

#include "fa_bwd.cuh"

namespace fa {

struct BwdEntry {
  const void* fn;  // the __global__ function (for attributes)
  int smem;        // dynamic shared memory bytes
  cudaError_t (*launch)(const BwdParams& p, int grid, cudaStream_t stream);
};

template <int DQ, int DV, int KIND, bool CAUSAL, int VAR>
cudaError_t launch_bwd(const BwdParams& p, int grid, cudaStream_t stream) {
  fa_bwd_kernel<DQ, DV, KIND, CAUSAL, VAR><<<grid, kBwdThreads, BwdLayout<DQ, DV>::kDynSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int DQ, int DV, int KIND, bool CAUSAL, int VAR = 0>
BwdEntry make_bwd_entry() {
  return BwdEntry{reinterpret_cast<const void*>(&fa_bwd_kernel<DQ, DV, KIND, CAUSAL, VAR>),
                  BwdLayout<DQ, DV>::kDynSmem, &launch_bwd<DQ, DV, KIND, CAUSAL, VAR>};
}

// false when (d_qk, d_v, kind, causal) is not built
bool bwd_entry(int dq, int dv, int kind, int causal, BwdEntry* out);

// the event-log build (fa_options.trace): (d_qk, d_v) = (128, 128) only
bool bwd_trace_entry(int dq, int dv, int kind, int causal, BwdEntry* out);

// the variable-length build: the same head dims as bwd_entry
bool bwd_varlen_entry(int dq, int dv, int kind, int causal, BwdEntry* out);

// sequences one backward planning CTA sorts in shared memory
constexpr int kVarlenPlanMaxBatch = 8192;

// the backward's planning kernel for a variable-length batch: counts[0] dK/dV
// tasks, counts[1] dQ tasks, their records; bad cu_seqlens: both counts 0 and
// FA_ERR_INVALID_ARG with site 501 and the sequence in the status word.  While
// *attr_ready is false (once per device; callers serialise it) the kernel's
// shared-memory attribute is set first.
cudaError_t launch_bwd_varlen_plan(const int* cu_q, const int* cu_k, int batch, int64_t total_q, int64_t total_k,
                                   int Hq, int Hkv, int causal, VarlenTask* kv_tasks, VarlenTask* q_tasks, int* counts,
                                   unsigned int* status, bool* attr_ready, cudaStream_t stream);

// D and LSE * log2(e) for a variable-length batch, per row of each dQ task
// record (count on the device), at h * vec_hstride + the sequence's padded offset + row
cudaError_t launch_bwd_prep_varlen(int dv, const void* o, const void* dout, const float* lse, float* l2, float* dvec,
                                   const VarlenTask* dq_tasks, const int* dq_count, int Hq, int64_t total_q,
                                   int vec_hstride, int grid, cudaStream_t stream);

// D = rowsum(dO * O) (over d_v) and LSE * log2(e) per row, padded to whole 128-row blocks
cudaError_t launch_bwd_prep(int dv, const void* o, const void* dout, const float* lse, float* l2, float* dvec, int B,
                            int Hq, int Sq, int sq_pad, int max_blocks, cudaStream_t stream);

}  // namespace fa
