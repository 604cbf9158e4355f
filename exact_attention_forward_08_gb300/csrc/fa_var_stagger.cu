// Staggered-exponential instantiations of the attention forward kernel (VAR =
// kVarStagger, an ablation): the benchmark head dims (128, 128) and
// (192, 128), fixed-length and direct epilogue modes.
#include "fa_dispatch.h"

namespace fa {

bool entry_stagger(int dq, int dv, int causal, int variant, KernelEntry* out) {
  if (variant != kModeFixed && variant != kModeDirect) return false;
  if (dq == 128 && dv == 128) {
    *out = pick_debug<128, 128, kVarStagger>(causal, variant);
    return true;
  }
  if (dq == 192 && dv == 128) {
    *out = pick_debug<192, 128, kVarStagger>(causal, variant);
    return true;
  }
  return false;
}

}  // namespace fa
