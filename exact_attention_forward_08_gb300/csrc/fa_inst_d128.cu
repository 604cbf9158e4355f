// Instantiations of the attention forward kernel for d_qk = 128.
#include "fa_dispatch.h"

namespace fa {

bool entry_d128(int dv, int causal, KernelEntry* out) {
  if (dv == 64) {
    *out = causal ? make_entry<128, 64, true>() : make_entry<128, 64, false>();
    return true;
  }
  if (dv == 128) {
    *out = causal ? make_entry<128, 128, true>() : make_entry<128, 128, false>();
    return true;
  }
  return false;
}

}  // namespace fa
