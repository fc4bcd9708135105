// ws_gemv_q4.cu -- the streaming GEMV over 4-bit group-128 weights ("One
// Token, Kernel by Kernel: A Decode Step on a Laptop GPU", "4-bit weights":
// every linear layer quantised to 4-bit integers in groups of 128, 3.76 times
// fewer bytes than bf16), general instantiations for batch 1, 2 and 4, and
// the quantiser that writes the packed format from bf16 weights.
#include <cuda_bf16.h>

#include "ws_gemv_kernel.cuh"

namespace ws {

GemvKernel pick_form_q4_b1(int BT, int nmat, int RT, int F);
GemvKernel pick_form_q4_b24(int BT, int nmat, int RT, int F);

#define WS_Q4(bt, nm, rt) \
  if (BT == bt && nmat == nm && RT == rt) return (GemvKernel)k_stream_gemv<bt, nm, rt, F_ANY, true>;

GemvKernel pick_kernel_q4(int BT, int nmat, int RT, int F) {
  if (F != F_ANY) return BT == 1 ? pick_form_q4_b1(BT, nmat, RT, F) : pick_form_q4_b24(BT, nmat, RT, F);
  WS_Q4(1, 1, 1) WS_Q4(1, 1, 2) WS_Q4(1, 1, 4) WS_Q4(1, 2, 1) WS_Q4(1, 2, 2)
  WS_Q4(2, 1, 1) WS_Q4(2, 1, 2) WS_Q4(2, 1, 4) WS_Q4(2, 2, 1) WS_Q4(2, 2, 2)
  WS_Q4(4, 1, 1) WS_Q4(4, 1, 2) WS_Q4(4, 1, 4) WS_Q4(4, 2, 1) WS_Q4(4, 2, 2)
  return nullptr;
}

// Min-max quantisation of one group per warp, every decision in fp32 with
// explicit round-to-nearest operations (no contraction):
//   s = bf16((max - min) / 15), z = bf16(min + 8 s),
//   q = clamp(rint((w - z) / s) + 8, 0, 15)   (q = 8 when s is 0).
// Lane l holds weights 4l .. 4l+3 of the group; lanes 2i and 2i+1 build
// word i (k = 8i .. 8i+7: even k in the low half's nibbles, odd k in the
// high half's).  The output rows are zero-filled beforehand (the padding).
__global__ void __launch_bounds__(256) k_quantize_q4(const uint16_t* __restrict__ W,
                                                     uint8_t* __restrict__ out, int M, int K) {
  const int lane = threadIdx.x & 31;
  const long long gid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int ng = K / kQ4Group;
  if (gid >= (long long)M * ng) return;
  const int m = (int)(gid / ng), g = (int)(gid - (long long)m * ng);
  const uint2 raw = *reinterpret_cast<const uint2*>(W + (size_t)m * K + g * kQ4Group + 4 * lane);
  const float w[4] = {bf16lo(raw.x), bf16hi(raw.x), bf16lo(raw.y), bf16hi(raw.y)};
  float lo = fminf(fminf(w[0], w[1]), fminf(w[2], w[3]));
  float hi = fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
  const float s = __bfloat162float(sb);
  const __nv_bfloat16 zb = __float2bfloat16_rn(__fadd_rn(lo, __fmul_rn(8.0f, s)));
  const float z = __bfloat162float(zb);
  uint32_t q[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float v = 8.0f;
    if (s != 0.0f) v = __fadd_rn(rintf(__fdiv_rn(__fsub_rn(w[e], z), s)), 8.0f);
    v = fminf(fmaxf(v, 0.0f), 15.0f);
    q[e] = (uint32_t)v;
  }
  // even lane: k = 8i + {0,1,2,3} -> nibbles 0, 4, 1, 5 (bits 0, 16, 4, 20);
  // odd lane: k = 8i + {4,5,6,7} -> nibbles 2, 6, 3, 7 (bits 8, 24, 12, 28)
  const int sh = (lane & 1) ? 8 : 0;
  uint32_t word = (q[0] << sh) | (q[1] << (16 + sh)) | (q[2] << (4 + sh)) | (q[3] << (20 + sh));
  word |= __shfl_xor_sync(0xffffffffu, word, 1);
  const int u = g / 4, gi = g % 4;
  const int gu = min(4, ng - 4 * u);
  uint8_t* row = out + (size_t)m * q4_prefix(K) + (size_t)u * kQ4SuperBytes;
  if (!(lane & 1)) reinterpret_cast<uint32_t*>(row + gi * 64)[lane >> 1] = word;
  if (lane == 0) {
    const uint32_t pair = (uint32_t)__bfloat16_as_ushort(sb) |
                          ((uint32_t)__bfloat16_as_ushort(zb) << 16);
    *reinterpret_cast<uint32_t*>(row + gu * 64 + gi * 4) = pair;
  }
}

cudaError_t launch_quantize_q4(const void* W, void* out, int M, int K, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, (size_t)M * q4_prefix(K), st);
  if (e != cudaSuccess) return e;
  const long long groups = (long long)M * (K / kQ4Group);
  const long long blocks = (groups + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  k_quantize_q4<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(W),
                                                 static_cast<uint8_t*>(out), M, K);
  return cudaGetLastError();
}

}  // namespace ws
