// Instantiations of the attention forward kernel for d_qk = 64.
#include "fa_dispatch.h"

namespace fa {

bool entry_d64(int dv, int causal, int variant, KernelEntry* out) {
  if (dv == 64) {
    *out = pick_entry<64, 64>(causal, variant);
    return true;
  }
  return false;
}

}  // namespace fa
