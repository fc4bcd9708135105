// Streaming GEMV instantiations for batch 9-16: rows per task 1 and 2 (a
// task's outputs, RT x 16, fill at most the 32 lanes of the reduction).
#include "ws_gemv_kernel.cuh"

namespace ws {

#define WS_INST(bt, nm, rt) \
  if (BT == bt && nmat == nm && RT == rt) return (GemvKernel)k_stream_gemv<bt, nm, rt, F_ANY>;

GemvKernel pick_kernel_b16(int BT, int nmat, int RT) {
  WS_INST(16, 1, 1) WS_INST(16, 1, 2)
  WS_INST(16, 2, 1) WS_INST(16, 2, 2)
  return nullptr;
}

}  // namespace ws
