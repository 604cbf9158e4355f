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

template <int DQ, int DV, bool CAUSAL, bool EMU>
cudaError_t launch_kernel(const Params& p, int grid, cudaStream_t stream) {
  fa_fwd_kernel<DQ, DV, CAUSAL, EMU><<<grid, kThreads, Layout<DQ, DV>::kDynSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int DQ, int DV, bool CAUSAL, bool EMU>
KernelEntry make_entry() {
  return KernelEntry{reinterpret_cast<const void*>(&fa_fwd_kernel<DQ, DV, CAUSAL, EMU>), Layout<DQ, DV>::kDynSmem,
                     &launch_kernel<DQ, DV, CAUSAL, EMU>};
}

template <int DQ, int DV>
KernelEntry pick_entry(int causal, int emu) {
  if (causal) return emu ? make_entry<DQ, DV, true, true>() : make_entry<DQ, DV, true, false>();
  return emu ? make_entry<DQ, DV, false, true>() : make_entry<DQ, DV, false, false>();
}

// defined in fa_inst_d{64,128,192}.cu; false when (dq, dv) is not built
bool entry_d64(int dv, int causal, int emu, KernelEntry* out);
bool entry_d128(int dv, int causal, int emu, KernelEntry* out);
bool entry_d192(int dv, int causal, int emu, KernelEntry* out);

}  // namespace fa
