// Instantiations of the attention forward kernel for d_qk = 192.
#include "fa_dispatch.h"

namespace fa {

bool entry_d192(int dv, int causal, int variant, KernelEntry* out) {
  if (dv == 64) {
    *out = pick_entry<192, 64>(causal, variant);
    return true;
  }
  if (dv == 128) {
    *out = pick_entry<192, 128>(causal, variant);
    return true;
  }
  return false;
}

}  // namespace fa
