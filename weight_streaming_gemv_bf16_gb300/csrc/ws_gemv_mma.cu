// Tensor-core streaming GEMV instantiations: the decode-chain forms at batch
// tiles 8 and 16.
#include "ws_gemv_mma.cuh"

namespace ws {

#define WS_MMA(bt, nm, f) \
  if (BT == bt && nmat == nm && F == f) return (GemvKernel)k_stream_gemv_mma<bt, nm, f>;
#define WS_MMAS(bt)                                                                \
  WS_MMA(bt, 1, F_RMS_F32) WS_MMA(bt, 2, F_RMS_SWIGLU) WS_MMA(bt, 1, F_RMS_ARGMAX) \
  WS_MMA(bt, 1, F_BF16_RESID) WS_MMA(bt, 1, F_BF16_F32)

GemvKernel pick_kernel_mma(int BT, int nmat, int F) {
  WS_MMAS(8) WS_MMAS(16)
  return nullptr;
}

}  // namespace ws
