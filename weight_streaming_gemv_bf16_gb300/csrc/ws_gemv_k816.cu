// Streaming GEMV instantiations for batch 5-8 (rows per task 1, 2, 4).
#include "ws_gemv_kernel.cuh"

namespace ws {

#define WS_INST(bt, nm, rt) \
  if (BT == bt && nmat == nm && RT == rt) return (GemvKernel)k_stream_gemv<bt, nm, rt, F_ANY>;

GemvKernel pick_kernel_b816(int BT, int nmat, int RT) {
  WS_INST(8, 1, 1) WS_INST(8, 1, 2) WS_INST(8, 1, 4)
  WS_INST(8, 2, 1) WS_INST(8, 2, 2) WS_INST(8, 2, 4)
  return nullptr;
}

}  // namespace ws
