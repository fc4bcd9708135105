// Streaming GEMV over 4-bit group-128 weights: the decode-chain forms at
// batch tiles 2 and 4 that beat the general kernel there (QKV with RMSNorm,
// Wo and Wd with the residual).  Gate/up stays on the general kernel (its
// form measured slower: 19.0 against 14.4 us a launch at batch 4, 13.1
// against 11.3 at batch 2); the LM head at these batches takes the
// tensor-core kernel.
#include "ws_gemv_kernel.cuh"

namespace ws {

#define WS_Q4F(bt, nm, rt, f) \
  if (BT == bt && nmat == nm && RT == rt && F == f) return (GemvKernel)k_stream_gemv<bt, nm, rt, f, true>;
#define WS_Q4FORMS(bt)                                                               \
  WS_Q4F(bt, 1, 1, F_RMS_F32) WS_Q4F(bt, 1, 2, F_RMS_F32) WS_Q4F(bt, 1, 4, F_RMS_F32) \
  WS_Q4F(bt, 1, 1, F_BF16_RESID) WS_Q4F(bt, 1, 2, F_BF16_RESID) WS_Q4F(bt, 1, 4, F_BF16_RESID)

GemvKernel pick_form_q4_b24(int BT, int nmat, int RT, int F) {
  WS_Q4FORMS(2) WS_Q4FORMS(4)
  return nullptr;
}

}  // namespace ws
