// Tensor-core streaming GEMV over 4-bit group-128 weights for the decode-chain
// forms at batch 1..4 ("One Token, Kernel by Kernel: A Decode Step on a
// Laptop GPU", "4-bit weights": at 4 bits even a GEMV becomes partly an
// instruction problem).  Expanding the codes costs about one integer
// operation per weight; the multiply-adds go to the MMA, so the kernel is
// bound by HBM rather than by the integer pipe the CUDA-core version fills.
#include "ws_gemv_mma.cuh"

namespace ws {

#define WS_Q4M(nm, f) \
  if (nmat == nm && F == f) return (GemvKernel)k_stream_gemv_mma<8, nm, f, true>;

GemvKernel pick_kernel_q4mma(int nmat, int F) {
  WS_Q4M(1, F_RMS_F32) WS_Q4M(1, F_BF16_RESID) WS_Q4M(1, F_BF16_F32)
  WS_Q4M(2, F_RMS_SWIGLU) WS_Q4M(1, F_RMS_ARGMAX)
  return nullptr;
}

}  // namespace ws
