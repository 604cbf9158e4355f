// Checking instantiations of the attention forward kernel (VAR = kVarCheck)
// for d_qk = 192, fixed-length and direct epilogue modes.
#include "fa_dispatch.h"

namespace fa {

bool entry_check_b(int dq, int dv, int causal, int variant, KernelEntry* out) {
  if (variant != kModeFixed && variant != kModeDirect) return false;
  if (dq == 192 && dv == 64) {
    *out = pick_debug<192, 64, kVarCheck>(causal, variant);
    return true;
  }
  if (dq == 192 && dv == 128) {
    *out = pick_debug<192, 128, kVarCheck>(causal, variant);
    return true;
  }
  return false;
}

}  // namespace fa
