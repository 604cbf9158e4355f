// The event-log build of the attention backward kernels (fa_options.trace):
// (d_qk, d_v) = (128, 128), both kernels, with and without the causal mask.
#include "fa_bwd_dispatch.h"

namespace fa {

bool bwd_trace_entry(int dq, int dv, int kind, int causal, BwdEntry* out) {
  if (dq != 128 || dv != 128) return false;
  if (kind == kBwdDkDv)
    *out = causal ? make_bwd_entry<128, 128, kBwdDkDv, true, kVarTrace>()
                  : make_bwd_entry<128, 128, kBwdDkDv, false, kVarTrace>();
  else if (kind == kBwdDq)
    *out = causal ? make_bwd_entry<128, 128, kBwdDq, true, kVarTrace>()
                  : make_bwd_entry<128, 128, kBwdDq, false, kVarTrace>();
  else
    return false;
  return true;
}

}  // namespace fa
