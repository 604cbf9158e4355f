// Kernel table: one entry per (d_qk, d_v, causal, mode) instantiation; the
// modes are fixed-length, fixed-length with the FMA-pipe exp2, varlen (its
// tasks always assigned dynamically), fixed-length with dynamic task
// assignment, split-KV, and fixed-length with the direct epilogue.  Each head
// dimension lives in its own translation unit so the build compiles them in
// parallel.  The debug instantiations (event log, checks) of the
// fixed-length and direct-epilogue modes live in translation units of their
// own.
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

template <int DQ, int DV, bool CAUSAL, int MODE, int VAR = 0>
cudaError_t launch_kernel(const Params& p, int grid, cudaStream_t stream) {
  fa_fwd_kernel<DQ, DV, CAUSAL, MODE, VAR><<<grid, kThreads, Layout<DQ, DV>::kDynSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int DQ, int DV, bool CAUSAL, int MODE, int VAR = 0>
KernelEntry make_entry() {
  return KernelEntry{reinterpret_cast<const void*>(&fa_fwd_kernel<DQ, DV, CAUSAL, MODE, VAR>),
                     Layout<DQ, DV>::kDynSmem, &launch_kernel<DQ, DV, CAUSAL, MODE, VAR>};
}

// build variant: mode kModeFixed or kModeDirect, VAR a combination of kVarTrace, kVarCheck, kVarStagger
template <int DQ, int DV, int VAR>
KernelEntry pick_debug(int causal, int variant) {
  if (variant == kModeDirect)
    return causal ? make_entry<DQ, DV, true, kModeDirect, VAR>() : make_entry<DQ, DV, false, kModeDirect, VAR>();
  return causal ? make_entry<DQ, DV, true, kModeFixed, VAR>() : make_entry<DQ, DV, false, kModeFixed, VAR>();
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

// build variants (fa_dbg_trace.cu, fa_dbg_check_a.cu, fa_dbg_check_b.cu):
// the event log and the stagger ablation for (128, 128) and (192, 128), the
// checks for every pair; false when not built
bool entry_trace(int dq, int dv, int causal, int variant, KernelEntry* out);
bool entry_stagger(int dq, int dv, int causal, int variant, KernelEntry* out);
bool entry_check_a(int dq, int dv, int causal, int variant, KernelEntry* out);  // d_qk 64, 128
bool entry_check_b(int dq, int dv, int causal, int variant, KernelEntry* out);  // d_qk 192

}  // namespace fa
