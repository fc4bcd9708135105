// Streaming GEMV instantiations for batch 1 and 2 (rows per task 1, 2, 4).
#include "ws_gemv_kernel.cuh"

namespace ws {

#define WS_INST(bt, nm, rt) \
  if (BT == bt && nmat == nm && RT == rt) return (GemvKernel)k_stream_gemv<bt, nm, rt, F_ANY>;

GemvKernel pick_kernel_b12(int BT, int nmat, int RT) {
  WS_INST(1, 1, 1) WS_INST(1, 1, 2) WS_INST(1, 1, 4)
  WS_INST(1, 2, 1) WS_INST(1, 2, 2) WS_INST(1, 2, 4)
  WS_INST(2, 1, 1) WS_INST(2, 1, 2) WS_INST(2, 1, 4)
  WS_INST(2, 2, 1) WS_INST(2, 2, 2) WS_INST(2, 2, 4)
  return nullptr;
}

}  // namespace ws
