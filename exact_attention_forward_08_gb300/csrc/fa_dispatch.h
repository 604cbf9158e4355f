// Kernel table: one entry per (d_qk, d_v, causal, mode) instantiation; the
// modes are fixed-length, fixed-length with the FMA-pipe exp2, varlen (its
// tasks always assigned dynamically), fixed-length with dynamic task
// assignment, split-KV, and fixed-length with the direct epilogue.  Each head
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

template <int DQ, int DV, bool CAUSAL, int MODE>
cudaError_t launch_kernel(const Params& p, int grid, cudaStream_t stream) {
  fa_fwd_kernel<DQ, DV, CAUSAL, MODE><<<grid, kThreads, Layout<DQ, DV>::kDynSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int DQ, int DV, bool CAUSAL, int MODE>
KernelEntry make_entry() {
  return KernelEntry{reinterpret_cast<const void*>(&fa_fwd_kernel<DQ, DV, CAUSAL, MODE>), Layout<DQ, DV>::kDynSmem,
                     &launch_kernel<DQ, DV, CAUSAL, MODE>};
}

// variant = kernel mode (kModeFixed .. kModeSplit)
template <int DQ, int DV, bool CAUSAL>
KernelEntry pick_variant(int variant) {
  switch (variant) {
    case kModeEmu: return make_entry<DQ, DV, CAUSAL, kModeEmu>();
    case kModeVarlen: return make_entry<DQ, DV, CAUSAL, kModeVarlen>();
    case kModeDyn: return make_entry<DQ, DV, CAUSAL, kModeDyn>();
    case kModeSplit: return make_entry<DQ, DV, CAUSAL, kModeSplit>();
    case kModeDirect: return make_entry<DQ, DV, CAUSAL, kModeDirect>();
    default: return make_entry<DQ, DV, CAUSAL, kModeFixed>();
  }
}

template <int DQ, int DV>
KernelEntry pick_entry(int causal, int variant) {
  return causal ? pick_variant<DQ, DV, true>(variant) : pick_variant<DQ, DV, false>(variant);
}

// defined in fa_inst_d{64,128,192}.cu; false when (dq, dv) is not built
bool entry_d64(int dv, int causal, int variant, KernelEntry* out);
bool entry_d128(int dv, int causal, int variant, KernelEntry* out);
bool entry_d192(int dv, int causal, int variant, KernelEntry* out);

}  // namespace fa
