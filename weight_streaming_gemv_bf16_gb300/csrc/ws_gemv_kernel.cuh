// ws_gemv_kernel.cuh -- the streaming GEMV kernel (device code), included by
// the translation units that instantiate it for each batch size.
//
// y[b][m] = sum_k W[m][k] * x[b][k], bf16 W and x, fp32 accumulation ("One
// Token, Kernel by Kernel: A Decode Step on a Laptop GPU", Step 1, "What one
// block launches").  Design for GB300:
//  * every warp is an independent pipeline: it owns whole rows (a task of RT
//    rows, one K split), streams them from HBM through its own ring of
//    shared-memory stages with 1-D bulk async copies (cp.async.bulk, mbarrier
//    completion, L2 evict-first since each weight byte is read once), and
//    refills a stage as soon as its lanes have read it; no warp ever waits for
//    another in the main loop;
//  * the first stages are issued before griddepcontrol.wait: weights do not
//    depend on the previous op, so inside a chain the next op's weights stream
//    in while the previous op finishes (programmatic dependent launch);
//  * lanes take 16-byte chunks of each row and accumulate with the
//    mixed-precision fma (bf16 operands, fp32 addend, one rounding: the same
//    result as unpacking to fp32 and fmaf, in one instruction per product),
//    RT rows at a time (independent chains); at the end of a task a warp
//    reduce-scatter (halving shuffles) leaves the total of output (row r,
//    batch b) in lane group r*BT+b, whose first lane runs its epilogue;
//  * split-K for skinny shapes: partial sums go to a workspace and the last
//    split of a row group (atomic ticket) adds them in split order, so the
//    result does not depend on the order CTAs finish in; the ticket is reset
//    for the next call or graph replay ("Making small PyTorch ops faster on a
//    laptop GPU", "A full decode step is a different story": the last block
//    to finish merges and resets the ticket);
//  * the activations are normalised once per CTA (RMSNorm or LayerNorm
//    prologue in fp32, all threads, vector loads) and rounded once to bf16
//    into shared memory.
// This kernel multiplies on CUDA cores: at batch <= 4 the product is bound by
// HBM.  From batch 5 the chain forms with at least 8 Mi weights run the
// warp-level tensor-core kernel of ws_gemv_mma.cuh instead.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ws_common.cuh"
#include "ws_device.cuh"

namespace ws {

typedef void (*GemvKernel)(const GemvParams);

__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Two fp32 values rounded to bf16 (round to nearest even) and packed, lo in
// the low half: one conversion instruction for the pair.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void raise_device_error(int* err, int code) {
  if (err) atomicExch(err, code);
}

// Epilogue for one output element (segment seg, row m, batch row b).  v0 is
// the dot product with the first matrix, v1 with the second (SwiGLU up).
// res_s, when given, holds the residual input of rows res_row0 .. res_row0 +
// res_n - 1 (batch row b at b * res_n), read ahead into shared memory.
template <int EPI>  // the epilogue kind, or -1: p.epilogue
__device__ __forceinline__ void apply_epilogue(const GemvParams& p, int seg, int m, int b,
                                               float v0, float v1, float& best_v, int& best_i,
                                               const float* res_s = nullptr, int res_row0 = 0,
                                               int res_n = 0) {
  const Seg& S = p.seg[seg];
  const size_t o = (size_t)b * S.M + m;
  switch (EPI >= 0 ? EPI : p.epilogue) {
    case EPI_F32:
      static_cast<float*>(S.out)[o] = v0;
      break;
    case EPI_BF16:
      static_cast<__nv_bfloat16*>(S.out)[o] = __float2bfloat16_rn(v0);
      break;
    case EPI_RESID: {
      const float* src = p.res_in ? p.res_in : static_cast<const float*>(S.out);
      const float r = res_s ? res_s[b * res_n + (m - res_row0)] : __ldcg(src + o);
      static_cast<float*>(S.out)[o] = r + v0;
      break;
    }
    case EPI_BIAS_GELU: {
      const float t = bf16_round(v0 + __uint_as_float((uint32_t)p.bias[m] << 16));
      const float e = erff(t * 0.70710678118654752f);
      const float z = 0.5f * t * (1.0f + e);
      static_cast<__nv_bfloat16*>(S.out)[o] = __float2bfloat16_rn(z);
      if (p.pre_out) reinterpret_cast<__nv_bfloat16*>(p.pre_out)[o] = __float2bfloat16_rn(t);
      // d/dt of t Phi(t): Phi(t) + t phi(t), phi the standard normal density
      if (p.gelu_grad)
        p.gelu_grad[o] = 0.5f * (1.0f + e) + t * 0.39894228040143268f * expf(-0.5f * t * t);
      break;
    }
    case EPI_SWIGLU: {
      const float sv = v0 / (1.0f + expf(-v0)) * v1;
      static_cast<__nv_bfloat16*>(S.out)[o] = __float2bfloat16_rn(sv);
      break;
    }
    case EPI_ARGMAX: {
      if (p.logits) p.logits[o] = v0;
      const int row = S.row_base + m;
      if (arg_better(v0, row, best_v, best_i)) {
        best_v = v0;
        best_i = row;
      }
      break;
    }
    default:
      break;
  }
}

// Eight consecutive activations x[b][8c .. 8c+7] as fp32.  Activations are
// read at the L2 (ld.global.cg): inside the persistent chain kernel another
// SM wrote them after this SM may have cached an older copy in L1.
__device__ __forceinline__ void load_x8(const GemvParams& p, int b, int c, float (&v)[8]) {
  if (p.x_dtype == DT_F32) {
    const float4* src =
        reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + (size_t)b * p.K) + 2 * c;
    const float4 a = __ldcg(src), d = __ldcg(src + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = d.x; v[5] = d.y; v[6] = d.z; v[7] = d.w;
  } else {
    const uint4 u = __ldcg(
        reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + (size_t)b * p.K) + c);
    v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
    v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
  }
}

// Sum of s[b] over the kThreads compute threads for every batch row; the
// totals land in tot[b].  (The staging code below synchronises the compute
// threads only, with named barrier 1.)
template <int BT>
__device__ __forceinline__ void block_sum(float (&s)[BT], float* red, float* tot, int B, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    const float w = warp_sum(s[b]);
    if (lane == 0) red[warp * BT + b] = w;
  }
  consumer_sync(kThreads);
  if (tid < B) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += red[w * BT + tid];
    tot[tid] = t;
  }
  consumer_sync(kThreads);
}

// Per-row statistics of the prologue over the full K, by all threads with
// vector loads: RMSNorm r = rsqrt(mean x^2 + eps); LayerNorm mean and
// rstd = rsqrt(mean (x - mean)^2 + eps) (two passes).
template <int BT>
__device__ void prologue_stats(const GemvParams& p, float* stats, float* red, int tid) {
  if (p.prologue == PRO_NONE) return;
  const int nch = p.K >> 3;
  float* tot = red + kWarps * BT;
  float s[BT];
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    s[b] = 0.f;
    if (b < p.B)
      for (int c = tid; c < nch; c += kThreads) {
        float v[8];
        load_x8(p, b, c, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) s[b] = p.prologue == PRO_RMSNORM ? fmaf(v[e], v[e], s[b]) : s[b] + v[e];
      }
  }
  block_sum<BT>(s, red, tot, p.B, tid);
  if (p.prologue == PRO_RMSNORM) {
    if (tid < p.B) stats[2 * tid] = rsqrtf(tot[tid] / (float)p.K + p.eps);
    consumer_sync(kThreads);
    return;
  }
  if (tid < p.B) stats[2 * tid] = tot[tid] / (float)p.K;
  consumer_sync(kThreads);
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    s[b] = 0.f;
    if (b < p.B) {
      const float mean = stats[2 * b];
      for (int c = tid; c < nch; c += kThreads) {
        float v[8];
        load_x8(p, b, c, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) s[b] = fmaf(v[e] - mean, v[e] - mean, s[b]);
      }
    }
  }
  block_sum<BT>(s, red, tot, p.B, tid);
  if (tid < p.B) stats[2 * tid + 1] = rsqrtf(tot[tid] / (float)p.K + p.eps);
  consumer_sync(kThreads);
}

// Normalise eight activations of batch row b at column 8*cg and pack them as
// bf16 (one rounding).
__device__ __forceinline__ uint4 normalise8(const GemvParams& p, const float* stats, int b, int cg,
                                           float (&v)[8]) {
  const int k = cg * 8;
  if (p.prologue == PRO_RMSNORM) {
    const float r = stats[2 * b];
    const uint4 g = *reinterpret_cast<const uint4*>(p.gamma + k);
    const float gf[8] = {bf16lo(g.x), bf16hi(g.x), bf16lo(g.y), bf16hi(g.y),
                         bf16lo(g.z), bf16hi(g.z), bf16lo(g.w), bf16hi(g.w)};
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = v[e] * r * gf[e];
  } else if (p.prologue == PRO_LAYERNORM) {
    const float mean = stats[2 * b], rstd = stats[2 * b + 1];
    const uint4 g = *reinterpret_cast<const uint4*>(p.gamma + k);
    const uint4 bt = *reinterpret_cast<const uint4*>(p.beta + k);
    const float gf[8] = {bf16lo(g.x), bf16hi(g.x), bf16lo(g.y), bf16hi(g.y),
                         bf16lo(g.z), bf16hi(g.z), bf16lo(g.w), bf16hi(g.w)};
    const float bf[8] = {bf16lo(bt.x), bf16hi(bt.x), bf16lo(bt.y), bf16hi(bt.y),
                         bf16lo(bt.z), bf16hi(bt.z), bf16lo(bt.w), bf16hi(bt.w)};
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (v[e] - mean) * rstd * gf[e] + bf[e];
  }
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One-round staging for the RMSNorm prologue on fp32 activations when each
// thread has at most kOneRound 8-column chunks (B x K / 8 <= kOneRound x
// kThreads), the case of every RMSNorm in a decode chain.  The thread reads
// its chunks once and keeps them in registers across the CTA reduction, and
// normalises them with gamma read before the dependency wait (gamma does not
// depend on the previous op): one round of activation latency instead of the
// two of prologue_stats + stage_x, in compact code.  Same arithmetic: fp32
// sums of squares, x * r * gamma rounded once to bf16.

// Row b[i] and chunk c[i] of the chunks o0 + i * step (i < N) of a [rows][nch]
// array of 8-column chunks, stepped without a division per chunk (integer
// division is long code, and these run once per launch with cold caches).
template <int N, int BT = 2>
__device__ __forceinline__ void chunk_coords(int o0, int step, int nch, int (&b)[N], int (&c)[N]) {
  if constexpr (BT == 1) {  // one row: the callers only use chunks o < nch
#pragma unroll
    for (int i = 0; i < N; ++i) {
      b[i] = o0 + i * step < nch ? 0 : 1;
      c[i] = o0 + i * step;
    }
    return;
  }
  int bb = 0, cc = o0;
  while (cc >= nch) { cc -= nch; ++bb; }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    b[i] = bb;
    c[i] = cc;
    cc += step;
    while (cc >= nch) { cc -= nch; ++bb; }
  }
}

template <int NR, int BT>  // chunks per thread, batch tile
__device__ __forceinline__ void gamma_preload(const GemvParams& p, int tid, uint4 (&g)[NR]) {
  int b[NR], c[NR];
  chunk_coords<NR, BT>(tid, kThreads, p.K >> 3, b, c);
#pragma unroll
  for (int i = 0; i < NR; ++i)
    g[i] = b[i] < p.B ? *reinterpret_cast<const uint4*>(p.gamma + c[i] * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
}

// NG = NR: gamma was read per chunk before the dependency wait (g[i]);
// NG = 1 (batch tiles 8 and 16): gamma is read after the reduction instead,
// so that a thread's up to twelve activation chunks are all in flight at once
// rather than competing with twelve more chunks of gamma for registers
// (measured, the LayerNorm twin below: 7.2 us of staging at batch 16).
template <int BT, int NR, int NG>  // NR chunks per thread
__device__ void stage_rms_one_round(const GemvParams& p, float* stats, float* red, uint16_t* xs,
                                    int tid, const uint4 (&g)[NG]) {
  static_assert(NG == NR || NG == 1, "gamma per chunk, or read late");
  constexpr bool late = NG != NR;
  const int nch = p.K >> 3, n = p.B * nch;
  float* tot = red + kWarps * BT;
  float v[NR][8];
  float s[BT];
  int rb[NR], rc[NR];
  chunk_coords<NR, BT>(tid, kThreads, nch, rb, rc);
#pragma unroll
  for (int b = 0; b < BT; ++b) s[b] = 0.f;
  // every load first (fp32, rows K apart: o = b * nch + c), then the sums
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int o = tid + i * kThreads;
    if (o < n) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x)) + 2 * o;
      const float4 lo4 = __ldcg(src), hi4 = __ldcg(src + 1);
      v[i][0] = lo4.x; v[i][1] = lo4.y; v[i][2] = lo4.z; v[i][3] = lo4.w;
      v[i][4] = hi4.x; v[i][5] = hi4.y; v[i][6] = hi4.z; v[i][7] = hi4.w;
    }
  }
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int o = tid + i * kThreads;
    if (o < n) {
      float t = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) t = fmaf(v[i][e], v[i][e], t);
#pragma unroll
      for (int bb = 0; bb < BT; ++bb)
        if (bb == rb[i]) s[bb] += t;
    }
  }
  block_sum<BT>(s, red, tot, p.B, tid);
  if (tid < p.B) stats[2 * tid] = rsqrtf(tot[tid] / (float)p.K + p.eps);
  consumer_sync(kThreads);
  uint4* xs4 = reinterpret_cast<uint4*>(xs);
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int o = tid + i * kThreads;
    if (o < n) {
      const float r = stats[2 * rb[i]];
      const uint4 gi = late ? __ldg(reinterpret_cast<const uint4*>(p.gamma) + rc[i]) : g[late ? 0 : i];
      const float gf[8] = {bf16lo(gi.x), bf16hi(gi.x), bf16lo(gi.y), bf16hi(gi.y),
                           bf16lo(gi.z), bf16hi(gi.z), bf16lo(gi.w), bf16hi(gi.w)};
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = pack_bf16x2(v[i][2 * e] * r * gf[2 * e], v[i][2 * e + 1] * r * gf[2 * e + 1]);
      xs4[o] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  // batch rows the kernel computes past B read zeros
  for (int o = n + tid; o < BT * nch; o += kThreads) xs4[o] = make_uint4(0u, 0u, 0u, 0u);
}

// LayerNorm per column chunk as in gamma_preload, for beta.
template <int NR, int BT>
__device__ __forceinline__ void beta_preload(const GemvParams& p, int tid, uint4 (&g)[NR]) {
  int b[NR], c[NR];
  chunk_coords<NR, BT>(tid, kThreads, p.K >> 3, b, c);
#pragma unroll
  for (int i = 0; i < NR; ++i)
    g[i] = b[i] < p.B ? *reinterpret_cast<const uint4*>(p.beta + c[i] * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
}

// One-round LayerNorm staging on bf16 activations (NR 8-column chunks per
// thread over the whole K, read once and kept in registers): the mean, then
// the variance about it from the same registers (two CTA reductions, one
// round of memory latency), then (x - mean) * rstd * gamma + beta rounded once
// to bf16 for this split's columns [c0, c0 + nch).  The arithmetic of
// prologue_stats + stage_x, with the sums grouped by thread.
// With NG = 1 (batch tiles 8 and 16) gamma and beta are read after the
// reductions, and the activations stay in registers as their bf16 words (four
// registers a chunk, widened at each use): a thread's chunks are all loaded
// before any is used.  With gamma and beta held per chunk and the widened
// values kept, the staging took 7.2 us at batch 16 against 2.3 at batch 4
// (768 columns: six chunks a thread at batch 16, two at batch 4).
template <int BT, int NR, int NG>
__device__ void stage_ln_one_round(const GemvParams& p, float* stats, float* red, uint16_t* xs,
                                   int c0, int nch, int tid, const uint4 (&g)[NG],
                                   const uint4 (&bt)[NG]) {
  static_assert(NG == NR || NG == 1, "gamma and beta per chunk, or read late");
  constexpr bool late = NG != NR;
  const int kch = p.K >> 3, n = p.B * kch;
  float* tot = red + kWarps * BT;
  uint4 u[NR];
  float s[BT];
  int rb[NR], rc[NR];
  chunk_coords<NR, BT>(tid, kThreads, kch, rb, rc);
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x));
#pragma unroll
  for (int b = 0; b < BT; ++b) s[b] = 0.f;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int o = tid + i * kThreads;
    u[i] = o < n ? __ldcg(src + o) : make_uint4(0u, 0u, 0u, 0u);  // rows K apart: o = b * kch + c
  }
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int o = tid + i * kThreads;
    if (o < n) {
      const float v[8] = {bf16lo(u[i].x), bf16hi(u[i].x), bf16lo(u[i].y), bf16hi(u[i].y),
                          bf16lo(u[i].z), bf16hi(u[i].z), bf16lo(u[i].w), bf16hi(u[i].w)};
      float t = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) t += v[e];
#pragma unroll
      for (int bb = 0; bb < BT; ++bb)
        if (bb == rb[i]) s[bb] += t;
    }
  }
  block_sum<BT>(s, red, tot, p.B, tid);
  if (tid < p.B) stats[2 * tid] = tot[tid] / (float)p.K;
  consumer_sync(kThreads);
#pragma unroll
  for (int b = 0; b < BT; ++b) s[b] = 0.f;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int o = tid + i * kThreads;
    if (o < n) {
      const float mean = stats[2 * rb[i]];
      const float v[8] = {bf16lo(u[i].x), bf16hi(u[i].x), bf16lo(u[i].y), bf16hi(u[i].y),
                          bf16lo(u[i].z), bf16hi(u[i].z), bf16lo(u[i].w), bf16hi(u[i].w)};
      float t = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) t = fmaf(v[e] - mean, v[e] - mean, t);
#pragma unroll
      for (int bb = 0; bb < BT; ++bb)
        if (bb == rb[i]) s[bb] += t;
    }
  }
  block_sum<BT>(s, red, tot, p.B, tid);
  if (tid < p.B) stats[2 * tid + 1] = rsqrtf(tot[tid] / (float)p.K + p.eps);
  consumer_sync(kThreads);
  uint4* xs4 = reinterpret_cast<uint4*>(xs);
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int o = tid + i * kThreads;
    const int c = rc[i] - c0;
    if (o < n && c >= 0 && c < nch) {
      const float mean = stats[2 * rb[i]], rstd = stats[2 * rb[i] + 1];
      const uint4 gi = late ? __ldg(reinterpret_cast<const uint4*>(p.gamma) + rc[i]) : g[late ? 0 : i];
      const uint4 bi = late ? __ldg(reinterpret_cast<const uint4*>(p.beta) + rc[i]) : bt[late ? 0 : i];
      const float gf[8] = {bf16lo(gi.x), bf16hi(gi.x), bf16lo(gi.y), bf16hi(gi.y),
                           bf16lo(gi.z), bf16hi(gi.z), bf16lo(gi.w), bf16hi(gi.w)};
      const float bf[8] = {bf16lo(bi.x), bf16hi(bi.x), bf16lo(bi.y), bf16hi(bi.y),
                           bf16lo(bi.z), bf16hi(bi.z), bf16lo(bi.w), bf16hi(bi.w)};
      const float v[8] = {bf16lo(u[i].x), bf16hi(u[i].x), bf16lo(u[i].y), bf16hi(u[i].y),
                          bf16lo(u[i].z), bf16hi(u[i].z), bf16lo(u[i].w), bf16hi(u[i].w)};
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = pack_bf16x2((v[2 * e] - mean) * rstd * gf[2 * e] + bf[2 * e],
                           (v[2 * e + 1] - mean) * rstd * gf[2 * e + 1] + bf[2 * e + 1]);
      xs4[rb[i] * nch + c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  // batch rows the kernel computes past B read zeros
  for (int o = p.B * nch + tid; o < BT * nch; o += kThreads) xs4[o] = make_uint4(0u, 0u, 0u, 0u);
}

// Staging by rows when a row has at most 32 * MC 8-column chunks (K <= 256 *
// MC), at batch tiles 8 and 16 and, for the forms that gain from it, 4 (the
// kernel decides): warp w normalises batch rows w + 8 j (j < BT / 8; below
// eight rows warps w < BT, row w) by itself, lane l taking the row's chunks
// l, l + 32, ..., so the statistics need warp shuffles only -- no CTA
// barrier -- and the code stays short.  A
// launch starts with cold instruction caches, and the CTA-wide version (each
// chunk's sum selected into one of BT partials, BT-wide block reductions)
// spent 6.5 us of a batch-16 LayerNorm block staging 16 x 768 values, most
// of it in code that ran once.  Every load is issued before any is used; gc
// (and bc) are gamma (and beta) at the lane's chunk columns, read before the
// dependency wait.  LayerNorm: mean, then the variance about it (two warp
// reductions), (x - mean) * rstd * gamma + beta; RMSNorm: x * rsqrt(mean x^2
// + eps) * gamma; rounded once to bf16 into columns [c0, c0 + nch) of xs.
template <int BT, int MC, bool LN>
__device__ void stage_rows(const GemvParams& p, float* stats, uint16_t* xs, int c0, int nch,
                           int warp, int lane, const uint4 (&gc)[MC], const uint4 (&bc)[MC]) {
  static_assert(BT % kWarps == 0 || BT < kWarps, "whole rows per warp");
  constexpr int RPW = BT >= kWarps ? BT / kWarps : 1;  // below 8 rows: warps < BT, a row each
  if (BT < kWarps && warp >= BT) return;
  const int kch = p.K >> 3;
  uint4* xs4 = reinterpret_cast<uint4*>(xs);
  // LayerNorm keeps the bf16 words (widened at each use), RMSNorm the fp32
  // values it loaded
  uint4 u[LN ? RPW : 1][LN ? MC : 1];
  float4 f[LN ? 1 : RPW][LN ? 1 : 2 * MC];
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    const int b = warp + kWarps * j;
#pragma unroll
    for (int m = 0; m < MC; ++m) {
      const int c = lane + 32 * m;
      const bool ok = b < p.B && c < kch;
      if constexpr (LN) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x));
        u[j][m] = ok ? __ldcg(src + (size_t)b * kch + c) : make_uint4(0u, 0u, 0u, 0u);
      } else {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x)) +
                            2 * ((size_t)b * kch + c);
        f[j][2 * m] = ok ? __ldcg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
        f[j][2 * m + 1] = ok ? __ldcg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    const int b = warp + kWarps * j;
    if (b >= p.B) {  // batch rows the kernel computes past B read zeros
      for (int c = lane; c < nch; c += 32) xs4[b * nch + c] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    auto vals = [&](int m, float (&v)[8]) {
      if constexpr (LN) {
        const uint4 w = u[j][m];
        v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
        v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
      } else {
        const float4 a = f[j][2 * m], c = f[j][2 * m + 1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
      }
    };
    float mean = 0.f, scale;
    if constexpr (LN) {
      float t = 0.f;
#pragma unroll
      for (int m = 0; m < MC; ++m) {
        float v[8];
        vals(m, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) t += v[e];
      }
      mean = warp_sum(t) / (float)p.K;
      float q = 0.f;
#pragma unroll
      for (int m = 0; m < MC; ++m) {
        if (lane + 32 * m < kch) {
          float v[8];
          vals(m, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) q = fmaf(v[e] - mean, v[e] - mean, q);
        }
      }
      scale = rsqrtf(warp_sum(q) / (float)p.K + p.eps);
    } else {
      float q = 0.f;
#pragma unroll
      for (int m = 0; m < MC; ++m) {
        float v[8];
        vals(m, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) q = fmaf(v[e], v[e], q);
      }
      scale = rsqrtf(warp_sum(q) / (float)p.K + p.eps);
    }
    if (lane == 0) {
      stats[2 * b] = LN ? mean : scale;
      stats[2 * b + 1] = scale;
    }
#pragma unroll
    for (int m = 0; m < MC; ++m) {
      const int c = lane + 32 * m, cc = c - c0;
      if (c < kch && cc >= 0 && cc < nch) {
        float v[8];
        vals(m, v);
        const uint4 g = gc[m];
        const float gf[8] = {bf16lo(g.x), bf16hi(g.x), bf16lo(g.y), bf16hi(g.y),
                             bf16lo(g.z), bf16hi(g.z), bf16lo(g.w), bf16hi(g.w)};
        float bf[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if constexpr (LN) {
          const uint4 h = bc[m];
          bf[0] = bf16lo(h.x); bf[1] = bf16hi(h.x); bf[2] = bf16lo(h.y); bf[3] = bf16hi(h.y);
          bf[4] = bf16lo(h.z); bf[5] = bf16hi(h.z); bf[6] = bf16lo(h.w); bf[7] = bf16hi(h.w);
        }
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if constexpr (LN)
            w[e] = pack_bf16x2((v[2 * e] - mean) * scale * gf[2 * e] + bf[2 * e],
                               (v[2 * e + 1] - mean) * scale * gf[2 * e + 1] + bf[2 * e + 1]);
          else
            w[e] = pack_bf16x2(v[2 * e] * scale * gf[2 * e], v[2 * e + 1] * scale * gf[2 * e + 1]);
        }
        xs4[b * nch + cc] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// gamma (or beta) at a lane's chunk columns lane, lane + 32, ... (zeros past K).
template <int MC>
__device__ __forceinline__ void cols_preload(const uint16_t* g, int kch, int lane, uint4 (&out)[MC]) {
#pragma unroll
  for (int m = 0; m < MC; ++m) {
    const int c = lane + 32 * m;
    out[m] = c < kch ? *reinterpret_cast<const uint4*>(g + c * 8) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Staging without a prologue, bf16 activations: a copy into shared memory,
// with each thread's loads (up to eight 16-byte chunks) all in flight before
// its first store, so K = 8960 costs one round of latency, not five.
template <int BT>
__device__ void stage_copy_bf16(const GemvParams& p, uint16_t* xs, int c0, int nch, int tid) {
  const int n = BT * nch;
  uint4* xs4 = reinterpret_cast<uint4*>(xs);
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x));
  const int rs = p.K >> 3;  // chunks per activation row in global memory
  for (int base = tid; base < n; base += 8 * kThreads) {
    uint4 t[8];
    int b[8], c[8];
    chunk_coords<8, BT>(base, kThreads, nch, b, c);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      t[i] = (b[i] < BT && b[i] < p.B) ? __ldcg(src + (size_t)b[i] * rs + c0 + c[i])
                                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int o = base + i * kThreads;
      if (o < n) xs4[o] = t[i];
    }
  }
}

// Prologue and staging in one pass: every thread loads all of its chunks of
// the activations first (one round of memory latency), the CTA reduces the
// statistics from registers, and the normalised bf16 rows -- all K columns --
// go to shared memory [BT][K].  Takes at most kMaxChunks chunks per thread;
// returns false (having done nothing) otherwise.
constexpr int kMaxChunks = 6;

template <int BT>
__device__ bool prologue_stage_fused(const GemvParams& p, float* stats, float* red, uint16_t* xs,
                                     int tid) {
  const int nch = p.K >> 3;
  const int total = BT * nch;
  if (total > kMaxChunks * kThreads) return false;
  float v[kMaxChunks][8];
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int o = tid + i * kThreads;
    const int b = o / nch;
    if (o < total && b < p.B) {
      load_x8(p, b, o - b * nch, v[i]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[i][e] = 0.f;
    }
  }
  if (p.prologue != PRO_NONE) {
    float* tot = red + kWarps * BT;
    float s[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) s[b] = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxChunks; ++i) {
      const int o = tid + i * kThreads;
#pragma unroll
      for (int b = 0; b < BT; ++b)
        if (o / nch == b)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            s[b] = p.prologue == PRO_RMSNORM ? fmaf(v[i][e], v[i][e], s[b]) : s[b] + v[i][e];
    }
    block_sum<BT>(s, red, tot, p.B, tid);
    if (p.prologue == PRO_RMSNORM) {
      if (tid < p.B) stats[2 * tid] = rsqrtf(tot[tid] / (float)p.K + p.eps);
    } else {
      if (tid < p.B) stats[2 * tid] = tot[tid] / (float)p.K;
      consumer_sync(kThreads);
#pragma unroll
      for (int b = 0; b < BT; ++b) s[b] = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxChunks; ++i) {
        const int o = tid + i * kThreads;
#pragma unroll
        for (int b = 0; b < BT; ++b)
          if (o / nch == b && b < p.B) {
            const float mean = stats[2 * b];
#pragma unroll
            for (int e = 0; e < 8; ++e) s[b] = fmaf(v[i][e] - mean, v[i][e] - mean, s[b]);
          }
      }
      block_sum<BT>(s, red, tot, p.B, tid);
      if (tid < p.B) stats[2 * tid + 1] = rsqrtf(tot[tid] / (float)p.K + p.eps);
    }
    consumer_sync(kThreads);
  }
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int o = tid + i * kThreads;
    if (o < total) {
      const int b = o / nch;
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      if (b < p.B) out = normalise8(p, stats, b, o - b * nch, v[i]);
      reinterpret_cast<uint4*>(xs)[o] = out;
    }
  }
  return true;
}

// Stage `nch` chunks of 8 columns, from chunk c0 on, of the (normalised)
// activations as bf16 into shared memory, [BT][nch]; rows b >= B are zero.
// (General path: any column range and any number of chunks per thread.)
template <int BT>
__device__ void stage_x(const GemvParams& p, const float* stats, uint16_t* xs, int c0, int nch,
                        int tid) {
  for (int o = tid; o < BT * nch; o += kThreads) {
    const int b = o / nch;
    const int c = o - b * nch;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (b < p.B) {
      if (p.prologue == PRO_NONE && p.x_dtype == DT_BF16) {
        out = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) +
                                                    (size_t)b * p.K) + c0 + c);
      } else {
        float v[8];
        load_x8(p, b, c0 + c, v);
        const int k = (c0 + c) * 8;
        if (p.prologue == PRO_RMSNORM) {
          const float r = stats[2 * b];
          const uint4 g = *reinterpret_cast<const uint4*>(p.gamma + k);
          const float gf[8] = {bf16lo(g.x), bf16hi(g.x), bf16lo(g.y), bf16hi(g.y),
                               bf16lo(g.z), bf16hi(g.z), bf16lo(g.w), bf16hi(g.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = v[e] * r * gf[e];
        } else if (p.prologue == PRO_LAYERNORM) {
          const float mean = stats[2 * b], rstd = stats[2 * b + 1];
          const uint4 g = *reinterpret_cast<const uint4*>(p.gamma + k);
          const uint4 bt = *reinterpret_cast<const uint4*>(p.beta + k);
          const float gf[8] = {bf16lo(g.x), bf16hi(g.x), bf16lo(g.y), bf16hi(g.y),
                               bf16lo(g.z), bf16hi(g.z), bf16lo(g.w), bf16hi(g.w)};
          const float bf[8] = {bf16lo(bt.x), bf16hi(bt.x), bf16lo(bt.y), bf16hi(bt.y),
                               bf16lo(bt.z), bf16hi(bt.z), bf16lo(bt.w), bf16hi(bt.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = (v[e] - mean) * rstd * gf[e] + bf[e];
        }
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
        out = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    reinterpret_cast<uint4*>(xs)[(size_t)b * nch + c] = out;
  }
}

// Issue the bulk copies of piece j (columns [k0 + j*PC, ...)) of row group rg
// into ring slot `slot`.
// Dot products of one ring piece against the staged activations: the piece
// holds NMAT x RT rows of nc 8-column chunks, rows rs chunks apart; xs points
// at the activations' chunk matching the piece's first column, batch rows
// nchx chunks apart.  Lane l takes chunks l, l + 32, ...  Each output keeps
// ACC partial sums (word k of a chunk feeds partial k % ACC), so that a warp
// always has at least eight independent fma chains; the partials are folded
// into acc at the end of the piece.  Rows past the end of the matrix hold
// stale bytes; their sums are never written out.
template <int BT, int NMAT, int RT, int UNROLL = 2>
__device__ __forceinline__ void dot_piece(float (&acc)[2][4][BT], const uint4* st,
                                          const uint4* xs, int nc, int rs, int nchx, int lane) {
  constexpr int CH = NMAT * RT * BT;
  constexpr int kUnroll = UNROLL;
  constexpr int ACC = CH >= 8 ? 1 : (CH >= 4 ? 2 : 4);
  float part[ACC][NMAT][RT][BT];
#pragma unroll
  for (int a = 0; a < ACC; ++a)
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) part[a][m][r][b] = 0.f;
#pragma unroll kUnroll
  for (int c = lane; c < nc; c += 32) {
    uint4 w[NMAT][RT];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int m = 0; m < NMAT; ++m) w[m][r] = st[(m * RT + r) * rs + c];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const uint4 xv = xs[b * nchx + c];
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          part[0][m][r][b] = fma_bf16x2(w[m][r].x, xv.x, part[0][m][r][b]);
          part[1 % ACC][m][r][b] = fma_bf16x2(w[m][r].y, xv.y, part[1 % ACC][m][r][b]);
          part[2 % ACC][m][r][b] = fma_bf16x2(w[m][r].z, xv.z, part[2 % ACC][m][r][b]);
          part[3 % ACC][m][r][b] = fma_bf16x2(w[m][r].w, xv.w, part[3 % ACC][m][r][b]);
        }
    }
  }
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        float t = part[0][m][r][b];
#pragma unroll
        for (int a = 1; a < ACC; ++a) t += part[a][m][r][b];
        acc[m][r][b] += t;
      }
}

// Two 4-bit codes of a word (bits 4j.. and 16 + 4j..) as a bf16 pair 128 + q:
// 0x4300 is 128 in bf16 and the nibble lands in the low mantissa bits.
__device__ __forceinline__ uint32_t q4_pair(uint32_t w, int j) {
  return ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
}

// Dot products of one ring piece of 4-bit rows against the staged
// activations.  The piece holds NMAT x RT rows pst bytes apart, each len
// columns of whole super-groups.  Lane l takes 16-column chunks l, l + 32,
// ...: two code words (16 weights) and their group's (s, z) per row, two
// activation chunks and their sum X per batch row.  (16-column chunks keep
// every lane of a warp busy on a 1536-column row: 96 chunks, three a lane.)
// With t = sum (128 + q) x (mixed fma: bf16 operands, exact products, fp32
// sums), s t + (z - 136 s) X = sum (s (q - 8) + z) x.
template <int BT, int NMAT, int RT>
__device__ __forceinline__ void dot_piece_q4(float (&acc)[2][4][BT], const uint8_t* st, int pst,
                                             const uint4* xs, const float* xsum, int len,
                                             int nchx, int nx16, int lane) {
  const int nc = len >> 4, ngr = len >> 7;
  // batch 1: two chunks in flight per lane (measured: 4-bit step 677.5 ->
  // 671.8 us); at batch 4 the unrolled body is slower (1058 -> 1135 us)
  constexpr int kUnroll = BT == 1 ? 2 : 1;
#pragma unroll kUnroll
  for (int c = lane; c < nc; c += 32) {
    const int u = c >> 5, w = c & 31;    // super-group, 16-column chunk within it
    const int gu = min(4, ngr - 4 * u);  // groups of super-group u
    const int off = u * kQ4SuperBytes + w * 8;
    const int soff = u * kQ4SuperBytes + gu * 64 + (w >> 3) * 4;
    uint32_t qp[NMAT][RT][8];
    float sc[NMAT][RT], zc[NMAT][RT];
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const uint8_t* row = st + (size_t)(m * RT + r) * pst;
        const uint2 q = *reinterpret_cast<const uint2*>(row + off);
        const uint32_t sz = *reinterpret_cast<const uint32_t*>(row + soff);
        const uint32_t qw[2] = {q.x, q.y};
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) qp[m][r][4 * i + jj] = q4_pair(qw[i], jj);
        sc[m][r] = bf16lo(sz);
        zc[m][r] = fmaf(-136.f, bf16lo(sz), bf16hi(sz));
      }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const uint4* xb = xs + (size_t)b * nchx + 2 * c;
      const uint4 x0 = xb[0], x1 = xb[1];
      const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const float X = xsum[b * nx16 + c];
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          float t0 = 0.f, t1 = 0.f;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            t0 = fma_bf16x2(qp[m][r][e], xw[e], t0);
            t1 = fma_bf16x2(qp[m][r][e + 1], xw[e + 1], t1);
          }
          acc[m][r][b] = fmaf(sc[m][r], t0 + t1, acc[m][r][b]);
          acc[m][r][b] = fmaf(zc[m][r], X, acc[m][r][b]);
        }
    }
  }
}

// The last split of a row group: the sums over all splits, in split order,
// of the outputs o0 + 32 u (u < U) of this lane, n_out outputs in all.  The
// loads of U outputs and two splits are in flight together (the partials
// come from L2, one round trip each).
template <int NMAT, int U>
__device__ __forceinline__ void split_sums(const GemvParams& p, int rowg, int n_out, int o0,
                                           float (&v)[NMAT][U], int (&rr)[U], int (&bb)[U]) {
  bool ok[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int o = o0 + 32 * u;
    ok[u] = o < n_out;
    rr[u] = o / p.B;
    bb[u] = o - rr[u] * p.B;
#pragma unroll
    for (int m = 0; m < NMAT; ++m) v[m][u] = 0.f;
  }
#pragma unroll 2
  for (int s = 0; s < p.sc.S; ++s)
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u])
          v[m][u] += __ldcg(&p.part[((size_t)(s * NMAT + m) * p.B + bb[u]) * p.M_total + rowg + rr[u]]);
}

template <int NMAT, int RT, bool ONE_SEG, bool Q4 = false>
__device__ __forceinline__ void issue_piece(const GemvParams& p, int rg, int j, int slot, int k0,
                                            uint8_t* ring, uint64_t* full, uint64_t pol) {
  if constexpr (Q4) {
    // 4-bit rows: a piece is a run of whole super-groups (its columns start
    // at a multiple of 512), q4_prefix(PC) bytes apart in the ring
    const Sched& sc = p.sc;
    int seg = 0, rgl = rg;
    if (!ONE_SEG) decode_rg(p, rg, seg, rgl);
    const Seg& S = p.seg[seg];
    const int row0 = rgl * RT;
    const int rows = min(RT, S.M - row0);
    const int c0 = k0 + j * sc.PC;
    const int len = min(sc.PC, sc.KS - j * sc.PC);
    const int rb = q4_prefix(p.K), src0 = q4_prefix(c0);
    const int nb = q4_prefix(c0 + len) - src0, pst = q4_prefix(sc.PC);
    uint8_t* dst = ring + (size_t)slot * sc.piece_bytes;
    mbar_arrive_expect_tx(&full[slot], (uint32_t)(NMAT * rows * nb));
#pragma unroll
    for (int mat = 0; mat < NMAT; ++mat) {
      const uint8_t* W = reinterpret_cast<const uint8_t*>(mat == 0 ? S.W0 : S.W1);
      for (int r = 0; r < rows; ++r)
        bulk_copy_g2s(dst + ((size_t)mat * RT + r) * pst, W + (size_t)(row0 + r) * rb + src0,
                      (uint32_t)nb, &full[slot], pol);
    }
    return;
  }
  const Sched& sc = p.sc;
  int seg = 0, rgl = rg;
  if (!ONE_SEG) decode_rg(p, rg, seg, rgl);
  const Seg& S = p.seg[seg];
  const int row0 = rgl * RT;
  const int rows = min(RT, S.M - row0);
  const int c0 = k0 + j * sc.PC;
  const int len = min(sc.PC, sc.KS - j * sc.PC);
  uint8_t* dst = ring + (size_t)slot * sc.piece_bytes;
  const int K = p.K;
  mbar_arrive_expect_tx(&full[slot], (uint32_t)(NMAT * rows * len * 2));
#pragma unroll
  for (int mat = 0; mat < NMAT; ++mat) {
    const uint16_t* W = mat == 0 ? S.W0 : S.W1;
    // one copy per row (also for whole rows: one code path is shorter code)
    for (int r = 0; r < rows; ++r)
      bulk_copy_g2s(dst + ((size_t)mat * RT + r) * sc.PC * 2, W + (size_t)(row0 + r) * K + c0,
                    (uint32_t)(len * 2), &full[slot], pol);
  }
}

template <int BT, int NMAT, int RT, int F, bool Q4 = false>
__global__ void __launch_bounds__(kThreads, 1) k_stream_gemv(const __grid_constant__ GemvParams p) {
  using FT = FormTraits<F>;
  constexpr int EPI = FT::epi;
  const int epi = EPI >= 0 ? EPI : p.epilogue;
  unsigned long long* stamp =
      p.stamps ? p.stamps + (size_t)blockIdx.x * p.stamp_stride : nullptr;
  if (stamp && threadIdx.x == 0) stamp[0] = global_ns();
  extern __shared__ __align__(128) uint8_t smem[];
  const Sched& sc = p.sc;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sc.off_bar) + warp * kMaxStages;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + sc.off_flags);
  float* stats = reinterpret_cast<float*>(smem + sc.off_stats);
  float* red = reinterpret_cast<float*>(smem + sc.off_red);
  float* argv = reinterpret_cast<float*>(smem + sc.off_arg);
  int* argi = reinterpret_cast<int*>(argv + kWarps * 32);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + sc.off_xs);
  uint8_t* ring = smem + sc.off_ring + (size_t)warp * sc.NSW * sc.piece_bytes;

  int ks, rg0, rg1;
  cta_range(sc, blockIdx.x, ks, rg0, rg1);
  const int k0 = ks * sc.KS;
  const int NP = sc.NP, NSW = sc.NSW;
  const int npw = warp_tasks(rg0, rg1, warp) * NP;  // pieces of this warp
  const int rgw = rg0 + warp;                         // this warp's first row group

  // issue cursor (lane 0): next piece, its task, piece index and slot
  int iq = 0, iti = 0, ij = 0, islot = 0;
  uint64_t pol = 0;
  if (lane == 0) {
    for (int s = 0; s < NSW; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    pol = p.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
    // Weights do not depend on the previous kernel: fill the whole ring
    // before waiting for it.
    while (iq < NSW && iq < npw) {
      issue_piece<NMAT, RT, FT::one_seg, Q4>(p, rgw + iti * kWarps, ij, islot, k0, ring, full, pol);
      ++iq;
      if (++ij == NP) { ij = 0; ++iti; }
      if (++islot == NSW) islot = 0;
    }
  }
  // gamma does not depend on the previous op either
  const bool one_round = FT::rms1 || (!FT::copy_bf16 && !FT::ln1 && one_round_rms(p));
  constexpr int NR = (FT::rms1 || FT::ln1) ? form_round_chunks(BT) : kOneRound;
  // From batch tile 8 the normalising prologues stage whole rows per warp
  // (stage_rows) when a row has at most 32 * MC chunks, with gamma and beta
  // read per lane column here; otherwise the CTA-wide staging, which then
  // reads gamma and beta after its reductions.
  constexpr int NG = BT >= 8 ? 1 : NR;
  constexpr int MC = BT >= 16 ? 6 : 8;
  constexpr int NC = MC;
  // Below batch tile 8 only BT warps stage, a row each.  Measured: at batch
  // tile 4 that pays for the QKV form (QKV 6.2 -> 4.4 us a launch, the decode
  // step 975.5 -> 946.8 us) and the LayerNorm form (the 72-block chain 256.3
  // -> 223.3 us); at batch tile 2 the decode step lost (760.1 -> 778.5 us:
  // gate/up, next but one, 10.2 -> 12.1 us, with less of Wo's time left for
  // its ring fill) and so did the LayerNorm chain (209 -> 213 us); gate/up
  // itself loses, its few staging warps' loads queued behind its own 192 KB
  // ring fill; at batch 1 everything lost (the decode step 636 -> 698 us, the
  // LayerNorm chain 182 -> 227 us).
  constexpr bool kRowsSmall = BT == 4 && (F == F_RMS_F32 || F == F_LN_GELU);
  const bool by_rows = (BT >= kWarps || kRowsSmall) && (FT::rms1 || FT::ln1 || one_round) &&
                       (p.K >> 3) <= 32 * MC;
  uint4 gpre[NG];
  uint4 bpre[FT::ln1 ? NG : 1];
  uint4 gcol[NC], bcol[NC];
  if (by_rows) {
    if constexpr (BT >= kWarps || kRowsSmall) {
      if (BT >= kWarps || warp < BT) {
        cols_preload<NC>(p.gamma, p.K >> 3, lane, gcol);
        if constexpr (FT::ln1) cols_preload<NC>(p.beta, p.K >> 3, lane, bcol);
      }
    }
  } else if constexpr (NG == NR) {
    if (one_round || FT::ln1) gamma_preload<NR, BT>(p, tid, gpre);
    if constexpr (FT::ln1) beta_preload<NR, BT>(p, tid, bpre);
  }
  pdl_launch_dependents();
  pdl_wait();
  if (stamp && tid == 0) stamp[1] = global_ns();

  // the residual input of this CTA's rows, read while the activations stage
  float* res_s = (EPI < 0 || EPI == EPI_RESID) && sc.off_res
                     ? reinterpret_cast<float*>(smem + sc.off_res)
                     : nullptr;
  const int res_row0 = rg0 * RT;
  if (res_s) {
    const float* src = p.res_in ? p.res_in : static_cast<const float*>(p.seg[0].out);
    const int nr = min(rg1 * RT, p.seg[0].M) - res_row0;
#pragma unroll 1  // one pass when B x rows <= threads; compact code
    for (int i = tid; i < p.B * nr; i += kThreads) {
      const int b = i / nr, r = i - (i / nr) * nr;
      res_s[b * sc.res_rows + r] = __ldcg(src + (size_t)b * p.seg[0].M + res_row0 + r);
    }
  }
  // the activations of this CTA's split, [BT][KS].  Two passes (statistics,
  // then normalise and store) rather than the one-round fused path: the
  // fused code is 24 KB, and a launch of a chain starts with cold
  // instruction caches (measured: 817 vs 897 us per Qwen chain step).
  if (by_rows) {
    if constexpr (BT >= kWarps || kRowsSmall) {
      if constexpr (FT::ln1)
        stage_rows<BT, NC, true>(p, stats, xs, k0 >> 3, sc.KS >> 3, warp, lane, gcol, bcol);
      else
        stage_rows<BT, NC, false>(p, stats, xs, 0, p.K >> 3, warp, lane, gcol, bcol);
    }
  } else if constexpr (FT::rms1) {
    stage_rms_one_round<BT, NR>(p, stats, red, xs, tid, gpre);
  } else if constexpr (FT::ln1) {
    stage_ln_one_round<BT, NR>(p, stats, red, xs, k0 >> 3, sc.KS >> 3, tid, gpre, bpre);
  } else if constexpr (FT::copy_bf16) {
    stage_copy_bf16<BT>(p, xs, k0 >> 3, sc.KS >> 3, tid);
  } else if (one_round) {
    stage_rms_one_round<BT, NR>(p, stats, red, xs, tid, gpre);
  } else if (p.prologue == PRO_NONE && p.x_dtype == DT_BF16) {
    stage_copy_bf16<BT>(p, xs, k0 >> 3, sc.KS >> 3, tid);
  } else {
    prologue_stats<BT>(p, stats, red, tid);
    stage_x<BT>(p, stats, xs, k0 >> 3, sc.KS >> 3, tid);
  }
  __syncthreads();
  if (stamp && tid == 0) stamp[2] = global_ns();
  if constexpr (FT::ln1 || F == F_ANY) {
    // training forward: the LayerNorm statistics of every batch row, and the
    // normalised rows (the first CTA of each K split writes its columns)
    if (p.prologue == PRO_LAYERNORM) {
      if (p.ln_stats && blockIdx.x == 0 && tid < p.B) {
        p.ln_stats[2 * tid] = stats[2 * tid];
        p.ln_stats[2 * tid + 1] = stats[2 * tid + 1];
      }
      if (p.ln_out && (int)blockIdx.x == ks * sc.Gs) {
        const int nch = sc.KS >> 3;
        for (int o = tid; o < p.B * nch; o += kThreads) {
          const int b = o / nch, c = o - b * nch;
          reinterpret_cast<uint4*>(p.ln_out + (size_t)b * p.K + k0)[c] =
              reinterpret_cast<const uint4*>(xs)[o];
        }
      }
    }
  }

  const int nchx = sc.KS >> 3;  // chunks of x in shared memory
  const int ncp = sc.PC >> 3;   // chunk stride of one row of a piece
  const uint4* xs4 = reinterpret_cast<const uint4*>(xs);
  float* xsum = Q4 ? reinterpret_cast<float*>(smem + sc.off_xsum) : nullptr;
  if constexpr (Q4) {
    // per batch row the sum of every 16 staged (rounded) activations, in
    // column order
    const int n16 = sc.KS >> 4;
    for (int o = tid; o < BT * n16; o += kThreads) {
      const int b = o / n16, c = o - b * n16;
      const uint4* src = xs4 + (size_t)b * nchx + 2 * c;
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 v = src[i];
        sum += bf16lo(v.x) + bf16hi(v.x) + bf16lo(v.y) + bf16hi(v.y);
        sum += bf16lo(v.z) + bf16hi(v.z) + bf16lo(v.w) + bf16hi(v.w);
      }
      xsum[o] = sum;
    }
    __syncthreads();
  }
  float best_v = -INFINITY;
  int best_i = 0x7fffffff;
  bool abort = false;

  float acc[2][4][BT];  // [matrix][row][batch]; NMAT x RT used
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[m][r][b] = 0.f;

  // consume cursor: piece q of task ti, piece index j, ring slot and phase
  int ti = 0, j = 0, slot = 0;
  uint32_t phase = 0;
  for (int q = 0; q < npw; ++q) {
    const int rg = rgw + ti * kWarps;
    int seg = 0, rgl = rg;
    if (!FT::one_seg) decode_rg(p, rg, seg, rgl);
    const int row0 = rgl * RT;
    const int rows = min(RT, p.seg[seg].M - row0);
    const int len = min(sc.PC, sc.KS - j * sc.PC);
    const bool ok = abort || mbar_wait_bounded(&full[slot], phase, p.timeout_ns);
    if (__any_sync(0xffffffffu, !ok) && !abort) {
      abort = true;
      if (lane == 0) raise_device_error(p.err, DERR_TIMEOUT);
    }

    // a piece's rows sit PC columns apart, also in a task's shorter last piece
    const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)slot * sc.piece_bytes);
    // batch 1 in a chain form keeps the loop rolled: shorter code, and one
    // iteration per 16-byte chunk is far from the issue limit (measured: it
    // is not at batch 4).  From batch 8 one iteration already holds 256-512
    // independent fmas and its code overflows the instruction cache when
    // unrolled (ncu at batch 16: "no instruction" the top stall)
    if constexpr (Q4) {
      dot_piece_q4<BT, NMAT, RT>(acc, reinterpret_cast<const uint8_t*>(st), q4_prefix(sc.PC),
                                 xs4 + j * ncp, xsum + j * (sc.PC >> 4), len, nchx, sc.KS >> 4,
                                 lane);
    } else {
      dot_piece<BT, NMAT, RT, ((F != F_ANY && BT == 1) || BT >= 8) ? 1 : 2>(
          acc, st, xs4 + j * ncp, len >> 3, ncp, nchx, lane);
    }
    // Every lane's shared-memory reads of this slot have returned (their
    // values fed the FMAs above, and issue is in order): refill the slot.
    __syncwarp();
    if (lane == 0 && !abort && iq < npw) {
      issue_piece<NMAT, RT, FT::one_seg, Q4>(p, rgw + iti * kWarps, ij, islot, k0, ring, full, pol);
      ++iq;
      if (++ij == NP) { ij = 0; ++iti; }
      if (++islot == NSW) islot = 0;
    }

    if (j == NP - 1) {
      // task complete: sum over lanes; output o = r * BT + b ends in the
      // lanes of group o, whose first lane runs its epilogue
      constexpr int V = RT * BT, G = 32 / V;
      float v[NMAT][V];
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int b = 0; b < BT; ++b) v[m][r * BT + b] = acc[m][r][b];
      warp_reduce_scatter<NMAT, V>(v, lane);
      const int o = lane / G, r = o / BT, b = o - (o / BT) * BT;
      const bool mine = lane % G == 0 && r < rows && b < p.B;
      const int rowg = p.seg[seg].row_base + row0;
      if (FT::no_split || sc.S == 1) {
        if (mine)
          apply_epilogue<EPI>(p, seg, row0 + r, b, v[0][0], v[NMAT - 1][0], best_v, best_i, res_s,
                         res_row0, sc.res_rows);
      } else {
        // split-K: write this split's partials; the last split of the row
        // group adds all splits in split order and runs the epilogue
        if (mine) {
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
            p.part[((size_t)(ks * NMAT + m) * p.B + b) * p.M_total + rowg + r] = v[m][0];
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          const unsigned old = atomicAdd(&p.tickets[rg], 1u);
          last = old == (unsigned)(sc.S - 1);
          if (last) atomicExch(&p.tickets[rg], 0u);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          constexpr int U = 4;
          for (int o0 = lane; o0 < rows * p.B; o0 += 32 * U) {
            float v[NMAT][U];
            int rr[U], bb[U];
            split_sums<NMAT, U>(p, rowg, rows * p.B, o0, v, rr, bb);
#pragma unroll
            for (int u = 0; u < U; ++u)
              if (o0 + 32 * u < rows * p.B) {
                float dv = -INFINITY;
                int di = 0x7fffffff;
                apply_epilogue<EPI>(p, seg, row0 + rr[u], bb[u], v[0][u], v[NMAT - 1][u], dv, di,
                                    res_s, res_row0, sc.res_rows);
              }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int b = 0; b < BT; ++b) acc[m][r][b] = 0.f;
    }
    if (++j == NP) { j = 0; ++ti; }
    if (++slot == NSW) { slot = 0; phase ^= 1u; }
  }

  if (abort && lane == 0) {
    // a wait ran out: no copy may still be landing when the CTA exits; the
    // last NSW pieces issued are the only ones that can be in flight
    for (int q = iq - NSW; q < iq; ++q)
      if (q >= 0) mbar_wait_bounded(&full[q % NSW], (q / NSW) & 1, p.timeout_ns);
  }

  if (stamp) {  // the same for every thread of the grid
    __syncthreads();
    if (tid == 0) stamp[3] = global_ns();
  }

  if (epi == EPI_ARGMAX) {
    // per batch row b the lanes of output groups r*BT + b hold a running
    // best: a warp butterfly per batch row, then thread b combines the warps,
    // then the last CTA (ticket) combines all CTAs with a warp per batch row
    constexpr int G = 32 / (RT * BT);
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const bool has = (lane / G) % BT == b;
      float v = has ? best_v : -INFINITY;
      int i = has ? best_i : 0x7fffffff;
      warp_argmax(v, i);
      if (lane == 0) {
        argv[warp * BT + b] = v;
        argi[warp * BT + b] = i;
      }
    }
    __syncthreads();
    if (tid < p.B) {
      float bv = argv[tid];
      int bi = argi[tid];
#pragma unroll
      for (int w = 1; w < kWarps; ++w)
        if (arg_better(argv[w * BT + tid], argi[w * BT + tid], bv, bi)) {
          bv = argv[w * BT + tid];
          bi = argi[w * BT + tid];
        }
      p.arg_val[(size_t)blockIdx.x * p.B + tid] = bv;
      p.arg_idx[(size_t)blockIdx.x * p.B + tid] = bi;
      __threadfence();
    }
    __syncthreads();
    if (tid == 0) {
      const unsigned old = atomicAdd(p.arg_ticket, 1u);
      const int last = old == gridDim.x - 1;
      if (last) atomicExch(p.arg_ticket, 0u);
      flags[0] = last;
    }
    __syncthreads();
    if (flags[0]) {
      __threadfence();
      for (int b = warp; b < p.B; b += kWarps) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int c = lane; c < (int)gridDim.x; c += 32) {
          const float v = __ldcg(&p.arg_val[(size_t)c * p.B + b]);
          const int ix = __ldcg(&p.arg_idx[(size_t)c * p.B + b]);
          if (arg_better(v, ix, bv, bi)) {
            bv = v;
            bi = ix;
          }
        }
        warp_argmax(bv, bi);
        if (lane == 0) p.argmax_idx[b] = bi;
      }
    }
  }
}

// Instantiation tables, one per translation unit (compiled in parallel):
// the F_ANY kernels per batch tile, and the chain forms per batch tile.
GemvKernel pick_kernel_b12(int BT, int nmat, int RT);
GemvKernel pick_kernel_b4(int BT, int nmat, int RT);
GemvKernel pick_kernel_b816(int BT, int nmat, int RT);
GemvKernel pick_kernel_b16(int BT, int nmat, int RT);
GemvKernel pick_form_b1(int BT, int nmat, int RT, int F);
GemvKernel pick_form_b24(int BT, int nmat, int RT, int F);
GemvKernel pick_form_b8(int BT, int nmat, int RT, int F);
GemvKernel pick_form_b16(int BT, int nmat, int RT, int F);
GemvKernel pick_kernel_mma(int BT, int nmat, int F);
GemvKernel pick_kernel_q4(int BT, int nmat, int RT, int F);
GemvKernel pick_kernel_q4mma(int nmat, int F);

}  // namespace ws
