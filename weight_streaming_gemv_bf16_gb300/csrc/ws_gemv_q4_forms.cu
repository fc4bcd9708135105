// Streaming GEMV over 4-bit group-128 weights: the decode-chain forms at
// batch 1 (QKV with RMSNorm, Wo and Wd with the residual, gate/up with
// RMSNorm and SwiGLU, the LM head with RMSNorm and argmax).
#include "ws_gemv_kernel.cuh"

namespace ws {

#define WS_Q4F(nm, rt, f) \
  if (nmat == nm && RT == rt && F == f) return (GemvKernel)k_stream_gemv<1, nm, rt, f, true>;

GemvKernel pick_form_q4_b1(int BT, int nmat, int RT, int F) {
  if (BT != 1) return nullptr;
  WS_Q4F(1, 1, F_RMS_F32) WS_Q4F(1, 2, F_RMS_F32) WS_Q4F(1, 4, F_RMS_F32)
  WS_Q4F(1, 1, F_BF16_RESID) WS_Q4F(1, 2, F_BF16_RESID) WS_Q4F(1, 4, F_BF16_RESID)
  WS_Q4F(1, 1, F_RMS_ARGMAX) WS_Q4F(1, 2, F_RMS_ARGMAX) WS_Q4F(1, 4, F_RMS_ARGMAX)
  WS_Q4F(2, 1, F_RMS_SWIGLU) WS_Q4F(2, 2, F_RMS_SWIGLU)
  return nullptr;
}

}  // namespace ws
