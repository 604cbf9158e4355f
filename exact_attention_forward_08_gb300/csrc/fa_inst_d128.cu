// Instantiations of the attention forward kernel for d_qk = 128.
#include "fa_dispatch.h"

namespace fa {

bool entry_d128(int dv, int causal, int variant, KernelEntry* out) {
  if (dv == 64) {
    *out = pick_entry<128, 64>(causal, variant);
    return true;
  }
  if (dv == 128) {
    *out = pick_entry<128, 128>(causal, variant);
    return true;
  }
  return false;
}

}  // namespace fa
