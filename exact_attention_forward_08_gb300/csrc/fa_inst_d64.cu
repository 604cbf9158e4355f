// Instantiations of the attention forward kernel for d_qk = 64.
#include "fa_dispatch.h"

namespace fa {

bool entry_d64(int dv, int causal, KernelEntry* out) {
  if (dv == 64) {
    *out = causal ? make_entry<64, 64, true>() : make_entry<64, 64, false>();
    return true;
  }
  return false;
}

}  // namespace fa
