// Streaming GEMV instantiations of the decode-chain forms for batch 16 (rows
// per task 1, 2): each holds only the staging path and epilogue of its op.
#include "ws_gemv_kernel.cuh"

namespace ws {

#define WS_FORM(bt, nm, rt, f) \
  if (BT == bt && nmat == nm && RT == rt && F == f) return (GemvKernel)k_stream_gemv<bt, nm, rt, f>;
#define WS_FORMS(bt, rt)                                                           \
  WS_FORM(bt, 1, rt, F_RMS_F32) WS_FORM(bt, 2, rt, F_RMS_SWIGLU)                  \
  WS_FORM(bt, 1, rt, F_RMS_ARGMAX) WS_FORM(bt, 1, rt, F_BF16_RESID)                \
  WS_FORM(bt, 1, rt, F_BF16_F32) WS_FORM(bt, 1, rt, F_LN_GELU)

GemvKernel pick_form_b16(int BT, int nmat, int RT, int F) {
  WS_FORMS(16, 1) WS_FORMS(16, 2)
  return nullptr;
}

}  // namespace ws
