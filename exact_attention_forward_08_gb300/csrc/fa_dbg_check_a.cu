// Checking instantiations of the attention forward kernel (VAR = kVarCheck)
// for d_qk = 64 and 128, fixed-length and direct epilogue modes.
#include "fa_dispatch.h"

namespace fa {

bool entry_check_a(int dq, int dv, int causal, int variant, KernelEntry* out) {
  if (variant != kModeFixed && variant != kModeDirect) return false;
  if (dq == 64 && dv == 64) {
    *out = pick_debug<64, 64, kVarCheck>(causal, variant);
    return true;
  }
  if (dq == 128 && dv == 64) {
    *out = pick_debug<128, 64, kVarCheck>(causal, variant);
    return true;
  }
  if (dq == 128 && dv == 128) {
    *out = pick_debug<128, 128, kVarCheck>(causal, variant);
    return true;
  }
  return false;
}

}  // namespace fa
