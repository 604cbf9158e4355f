// Kernel table: one entry per (d_qk, d_v, causal) instantiation.  Each head
// dimension lives in its own translation unit so the build compiles them in
// parallel.
#pragma once
#include <cuda_runtime.h>

#include "fa_kernel.cuh"

namespace fa {

typedef cudaError_t (*LaunchFn)(const Params& p, int grid, cudaStream_t stream);

struct KernelEntry {
  const void* fn;  // the __global__ function (for attributes)
  int smem;        // dynamic shared memory bytes
  LaunchFn launch;
};

template <int DQ, int DV, bool CAUSAL>
cudaError_t launch_kernel(const Params& p, int grid, cudaStream_t stream) {
  fa_fwd_kernel<DQ, DV, CAUSAL><<<grid, kThreads, Layout<DQ, DV>::kDynSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int DQ, int DV, bool CAUSAL>
KernelEntry make_entry() {
  return KernelEntry{reinterpret_cast<const void*>(&fa_fwd_kernel<DQ, DV, CAUSAL>), Layout<DQ, DV>::kDynSmem,
                     &launch_kernel<DQ, DV, CAUSAL>};
}

// defined in fa_inst_d{64,128,192}.cu; false when (dq, dv) is not built
bool entry_d64(int dv, int causal, KernelEntry* out);
bool entry_d128(int dv, int causal, KernelEntry* out);
bool entry_d192(int dv, int causal, KernelEntry* out);

}  // namespace fa
