// Instantiations of the attention forward kernel for d_qk = 192.
#include "fa_dispatch.h"

namespace fa {

bool entry_d192(int dv, int causal, KernelEntry* out) {
  if (dv == 64) {
    *out = causal ? make_entry<192, 64, true>() : make_entry<192, 64, false>();
    return true;
  }
  if (dv == 128) {
    *out = causal ? make_entry<192, 128, true>() : make_entry<192, 128, false>();
    return true;
  }
  return false;
}

}  // namespace fa
