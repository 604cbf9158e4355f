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

// D = rowsum(dO * O) (over d_v) and LSE * log2(e) per row, padded to whole 128-row blocks
cudaError_t launch_bwd_prep(int dv, const void* o, const void* dout, const float* lse, float* l2, float* dvec, int B,
                            int Hq, int Sq, int sq_pad, int max_blocks, cudaStream_t stream);

}  // namespace fa
