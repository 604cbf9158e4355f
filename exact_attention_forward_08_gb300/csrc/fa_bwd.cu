// Instantiations of the attention backward kernels: (d_qk, d_v) = (64, 64),
// (128, 128) and (192, 128).
#include "fa_bwd_dispatch.h"

namespace fa {

template <int DQ, int DV>
static BwdEntry pick_bwd(int kind, int causal) {
  if (kind == kBwdDkDv)
    return causal ? make_bwd_entry<DQ, DV, kBwdDkDv, true>() : make_bwd_entry<DQ, DV, kBwdDkDv, false>();
  return causal ? make_bwd_entry<DQ, DV, kBwdDq, true>() : make_bwd_entry<DQ, DV, kBwdDq, false>();
}

bool bwd_entry(int dq, int dv, int kind, int causal, BwdEntry* out) {
  if (kind != kBwdDkDv && kind != kBwdDq) return false;
  if (dq == 64 && dv == 64) {
    *out = pick_bwd<64, 64>(kind, causal);
    return true;
  }
  if (dq == 128 && dv == 128) {
    *out = pick_bwd<128, 128>(kind, causal);
    return true;
  }
  if (dq == 192 && dv == 128) {
    *out = pick_bwd<192, 128>(kind, causal);
    return true;
  }
  return false;
}

cudaError_t launch_bwd_prep(int dv, const void* o, const void* dout, const float* lse, float* l2, float* dvec, int B,
                            int Hq, int Sq, int sq_pad, int max_blocks, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(B) * Hq * sq_pad;
  int64_t blocks = (rows + 7) / 8;  // 8 warps per block, one row per warp
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) return cudaSuccess;
  const uint16_t* o16 = static_cast<const uint16_t*>(o);
  const uint16_t* g16 = static_cast<const uint16_t*>(dout);
  if (dv == 128)
    fa_bwd_prep_kernel<128><<<static_cast<int>(blocks), 256, 0, stream>>>(o16, g16, lse, l2, dvec, B, Hq, Sq, sq_pad);
  else
    fa_bwd_prep_kernel<64><<<static_cast<int>(blocks), 256, 0, stream>>>(o16, g16, lse, l2, dvec, B, Hq, Sq, sq_pad);
  return cudaGetLastError();
}

}  // namespace fa
