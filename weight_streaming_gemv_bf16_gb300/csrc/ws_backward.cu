// ws_backward.cu -- training: the backward pass of a chain of LayerNorm ->
// Linear(+bias) -> GELU blocks, one launch per block, with the L2 prefetch of
// the next launch's weight on a side branch ("Making small PyTorch ops faster
// on a laptop GPU", "It works in training too": the gradient of block i reads
// W_i again, so while it runs the prefetch fetches W_(i-1)).
//
// What a block's backward computes (module by module, bf16 like the forward;
// every gradient a module hands on or keeps is rounded to bf16 once):
//   dlin = bf16(dz * gelu'(t))           t the GELU's input, saved by the forward
//   dln  = bf16(dlin . W)                 dln[b][k] = sum_m dlin[b][m] W[m][k]
//   dW   = bf16(dlin^T . ln)              dW[m][k]  = sum_b dlin[b][m] ln[b][k]
//   db   = bf16(sum_b dlin)
//   LayerNorm, xh = (x - mean) rstd, g = dln * gamma:
//   dx   = bf16(rstd (g - mean_k g - xh mean_k(g xh)))
//   dgamma = bf16(sum_b dln xh), dbeta = bf16(sum_b dln)
// and dx of block i is dz of block i - 1.
//
// Launch s (s = 0 .. L-1) runs the first five lines for block j = L-1-s (its
// "front") and, first, the LayerNorm lines for block j+1 (its "tail"), whose
// dx is block j's dz; launch L runs the tail of block 0 alone.  CTA c of a
// launch owns the 8 columns k0 = 8c .. 8c+7 of the block's [w][w] weight:
//  * before waiting for the previous launch it loads W[:, k0:k0+8] with 2-D
//    TMA boxes (8 columns x up to 256 rows) and, with 1-D bulk copies, the
//    forward's saved tensors it needs whole (x of block j+1, gelu'(t) of
//    block j); the weight does not depend on the previous launch;
//  * every CTA then computes the tail and dlin for the whole [B][w] (a few
//    thousand elements, cheaper than meeting the other CTAs at a barrier),
//    and writes the tail's outputs for its own columns;
//  * dln[:, k0:k0+8] is the transposed product over its slab: lane (k, q) of
//    warp v sums W[m][k] dlin[b][m] over a quarter of the warp's rows m for
//    four batch rows, the warps' partials are added in warp order;
//  * dW[:, k0:k0+8] takes the saved ln[:, k0:k0+8]: each thread forms whole
//    16-byte rows of the slab, one per weight row m it owns;
//  * db for the rows m = k0 .. k0+7 (the same index range as its columns).
// Sums run in a fixed order, so the result does not depend on timing, and a
// prefetch (which only reads) leaves every bit unchanged.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "wsgemv.h"
#include "ws_common.cuh"
#include "ws_device.cuh"

namespace ws {

constexpr int kBwdThreads = 512;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kSlab = 8;         // columns per CTA (16 bytes of bf16: one TMA box row)
constexpr int kBwdMaxWidth = 1024;
constexpr int kBwdWidthUnit = 64;  // widths are multiples of this
// The transposed product gives each warp w / kBwdWarps rows of dlin, read
// four rows at a time as aligned float4: every allowed width must give each
// warp a multiple of four rows.
static_assert(kBwdWidthUnit % (4 * kBwdWarps) == 0,
              "each warp's rows of the transposed product must be a multiple of four");

struct alignas(64) BwdParams {
  CUtensorMap tmW;  // the block's W [w rows][w columns] bf16, box {8, R}
  int B, w, R, nbox;
  // the tail: block j+1's LayerNorm backward (t_dln null: none)
  const uint16_t* t_dln;    // dln of block j+1 [B][w] bf16 (the previous launch's)
  const uint16_t* t_x;      // x of block j+1 [B][w] bf16 (forward)
  const float* t_stats;     // its mean, rstd [B][2] (forward)
  const uint16_t* t_gamma;  // [w]
  uint16_t* t_dx;           // dx of block j+1 [B][w] (this CTA's columns), or null
  uint16_t* t_dx2;          // a second copy of it, or null
  uint16_t* t_dgamma;       // [w]
  uint16_t* t_dbeta;        // [w]
  // the front: block j (has_front 0: the last launch)
  int has_front;
  const uint16_t* dz;       // the first launch: the loss gradient [B][w] bf16, or null:
  const uint16_t* z_loss;   //   dz = bf16(loss_scale * z) of the chain output z
  float loss_scale;
  uint16_t* dz_out;         // the first launch: dz written back (this CTA's columns), or null
  const float* f_gelu;      // gelu'(t) of block j [B][w] fp32 (forward)
  uint16_t* f_dlin;         // dlin of block j [B][w] (this CTA's columns)
  uint16_t* f_dln;          // dln of block j [B][w] (this CTA's columns)
  int* err;
  unsigned long long timeout_ns;
  // shared-memory layout (bytes)
  int off_slab, off_x, off_g, off_dl, off_dln, off_red, off_misc, smem_bytes, dl_stride;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Per batch row b < B, the sums over the CTA of a[b] and c[b] (BT values per
// thread each); totals in tot[2 b] and tot[2 b + 1].
template <int BT>
__device__ __forceinline__ void bwd_block_sum2(float (&a)[BT], float (&c)[BT], float* red,
                                               float* tot, int B, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    const float x = warp_sum(a[b]), y = warp_sum(c[b]);
    if (lane == 0) {
      red[(warp * BT + b) * 2] = x;
      red[(warp * BT + b) * 2 + 1] = y;
    }
  }
  __syncthreads();
  if (tid < 2 * B) {
    float t = 0.f;
    for (int v = 0; v < kBwdWarps; ++v) t += red[(v * BT + (tid >> 1)) * 2 + (tid & 1)];
    tot[tid] = t;
  }
  __syncthreads();
}

template <int BT>
__global__ void __launch_bounds__(kBwdThreads, 1) k_mlp_backward(const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  const uint4* slab = reinterpret_cast<const uint4*>(smem + p.off_slab);  // [w] rows of 8 bf16
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + p.off_x);  // [B][w] x of block j+1
  const float* gs = reinterpret_cast<const float*>(smem + p.off_g);        // [B][w] gelu'
  float* dl = reinterpret_cast<float*>(smem + p.off_dl);                   // [BT][dl_stride] dlin
  uint16_t* dlns = reinterpret_cast<uint16_t*>(smem + p.off_dln);          // [B][w] tail dln
  float* red = reinterpret_cast<float*>(smem + p.off_red);
  float* misc = reinterpret_cast<float*>(smem + p.off_misc);
  float* tot = misc;             // [2 BT] tail sums
  float* st = misc + 2 * BT;     // [2 BT] tail mean, rstd
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, w = p.w, nch = w >> 3;
  const int k0 = blockIdx.x * kSlab;
  const bool tail = p.t_dln != nullptr;

  // weights and the forward's saved tensors do not depend on the previous
  // launch: ask for them before waiting on it
  uint32_t tx = 0;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    if (p.has_front) tx += (uint32_t)p.nbox * p.R * 16;
    if (tail) tx += (uint32_t)B * w * 2;
    if (p.has_front) tx += (uint32_t)B * w * 4;
    mbar_arrive_expect_tx(bar, tx);
    if (p.has_front)
      for (int i = 0; i < p.nbox; ++i)
        tma_load_2d(smem + p.off_slab + (size_t)i * p.R * 16, &p.tmW, k0, i * p.R, bar);
    const uint64_t pol = l2_policy_evict_normal();
    // 1-D bulk copies of at most 16 KiB each
    auto copy = [&](uint8_t* dst, const void* src, uint32_t bytes) {
      for (uint32_t off = 0; off < bytes; off += 16384u) {
        const uint32_t nb = bytes - off < 16384u ? bytes - off : 16384u;
        bulk_copy_g2s(dst + off, static_cast<const uint8_t*>(src) + off, nb, bar, pol);
      }
    };
    if (tail) copy(smem + p.off_x, p.t_x, (uint32_t)B * w * 2);
    if (p.has_front) copy(smem + p.off_g, p.f_gelu, (uint32_t)B * w * 4);
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  const bool ok = mbar_wait_bounded(bar, 0, p.timeout_ns);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) {
      if (p.err) atomicExch(p.err, DERR_TIMEOUT);
      mbar_wait_bounded(bar, 0, p.timeout_ns);  // no copy may land after the CTA exits
    }
    return;
  }

  // ---- the tail (block j+1's LayerNorm backward) and dz of block j ----
  constexpr int NCH = (BT * kBwdMaxWidth / 8 + kBwdThreads - 1) / kBwdThreads;  // chunks per thread
  const int n = B * nch;
  if (tail) {
    if (tid < B) {
      st[2 * tid] = __ldg(p.t_stats + 2 * tid);
      st[2 * tid + 1] = __ldg(p.t_stats + 2 * tid + 1);
    }
    float s1[BT], s2[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) s1[b] = s2[b] = 0.f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int o = tid + i * kBwdThreads;
      if (o < n) {
        const int b = o / nch, c = o - b * nch;
        const uint4 d = __ldcg(reinterpret_cast<const uint4*>(p.t_dln) + o);
        reinterpret_cast<uint4*>(dlns)[o] = d;
        const uint4 xv = reinterpret_cast<const uint4*>(xs)[o];
        const uint4 gv = __ldg(reinterpret_cast<const uint4*>(p.t_gamma) + c);
        const uint32_t dw[4] = {d.x, d.y, d.z, d.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w},
                       gw[4] = {gv.x, gv.y, gv.z, gv.w};
        const float mean = st[2 * b], rstd = st[2 * b + 1];
        float a = 0.f, e = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float g0 = bf16lo(dw[q]) * bf16lo(gw[q]), g1 = bf16hi(dw[q]) * bf16hi(gw[q]);
          const float h0 = (bf16lo(xw[q]) - mean) * rstd, h1 = (bf16hi(xw[q]) - mean) * rstd;
          a += g0 + g1;
          e += g0 * h0 + g1 * h1;
        }
#pragma unroll
        for (int bb = 0; bb < BT; ++bb)
          if (bb == b) {
            s1[bb] += a;
            s2[bb] += e;
          }
      }
    }
    bwd_block_sum2<BT>(s1, s2, red, tot, B, tid);
  }
  // dz (the tail's dx, or the loss gradient) and dlin = bf16(dz * gelu'), for
  // all of [B][w]
  const float inv_w = 1.0f / (float)w;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int o = tid + i * kBwdThreads;
    if (o < n) {
      const int b = o / nch, c = o - b * nch;
      float dz[8];
      if (tail) {
        const uint4 d = reinterpret_cast<const uint4*>(dlns)[o];
        const uint4 xv = reinterpret_cast<const uint4*>(xs)[o];
        const uint4 gv = __ldg(reinterpret_cast<const uint4*>(p.t_gamma) + c);
        const uint32_t dw[4] = {d.x, d.y, d.z, d.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w},
                       gw[4] = {gv.x, gv.y, gv.z, gv.w};
        const float mean = st[2 * b], rstd = st[2 * b + 1];
        const float m1 = tot[2 * b] * inv_w, m2 = tot[2 * b + 1] * inv_w;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float g0 = bf16lo(dw[q]) * bf16lo(gw[q]), g1 = bf16hi(dw[q]) * bf16hi(gw[q]);
          const float h0 = (bf16lo(xw[q]) - mean) * rstd, h1 = (bf16hi(xw[q]) - mean) * rstd;
          dz[2 * q] = round_bf16(rstd * (g0 - m1 - h0 * m2));
          dz[2 * q + 1] = round_bf16(rstd * (g1 - m1 - h1 * m2));
        }
      } else {
        const uint4 v = p.dz ? __ldcg(reinterpret_cast<const uint4*>(p.dz) + o)
                             : __ldcg(reinterpret_cast<const uint4*>(p.z_loss) + o);
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dz[2 * q] = bf16lo(vw[q]);
          dz[2 * q + 1] = bf16hi(vw[q]);
        }
        if (!p.dz)
#pragma unroll
          for (int e = 0; e < 8; ++e) dz[e] = round_bf16(p.loss_scale * dz[e]);
      }
      // this CTA's columns of dz: the tail's dx (or the loss gradient)
      if (c == (k0 >> 3)) {
        const uint4 pk = make_uint4(pack2_bf16(dz[0], dz[1]), pack2_bf16(dz[2], dz[3]),
                                    pack2_bf16(dz[4], dz[5]), pack2_bf16(dz[6], dz[7]));
        uint16_t* d1 = tail ? p.t_dx : p.dz_out;
        uint16_t* d2 = tail ? p.t_dx2 : nullptr;
        if (d1) reinterpret_cast<uint4*>(d1)[o] = pk;
        if (d2) reinterpret_cast<uint4*>(d2)[o] = pk;
      }
      if (p.has_front) {
        const float4* g4 = reinterpret_cast<const float4*>(gs + (size_t)b * w + 8 * c);
        const float4 ga = g4[0], gb = g4[1];
        const float gd[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = round_bf16(dz[e] * gd[e]);
        float4* d4 = reinterpret_cast<float4*>(dl + (size_t)b * p.dl_stride + 8 * c);
        d4[0] = make_float4(v[0], v[1], v[2], v[3]);
        d4[1] = make_float4(v[4], v[5], v[6], v[7]);
        if (c == (k0 >> 3))
          reinterpret_cast<uint4*>(p.f_dlin)[o] =
              make_uint4(pack2_bf16(v[0], v[1]), pack2_bf16(v[2], v[3]),
                         pack2_bf16(v[4], v[5]), pack2_bf16(v[6], v[7]));
      }
    }
  }
  // the tail's dgamma and dbeta for this CTA's columns
  if (tail && tid < kSlab) {
    const int k = k0 + tid;
    float dg = 0.f, dbt = 0.f;
    for (int b = 0; b < B; ++b) {
      const float d = __uint_as_float((uint32_t)dlns[(size_t)b * w + k] << 16);
      const float xh = (__uint_as_float((uint32_t)xs[(size_t)b * w + k] << 16) - st[2 * b]) *
                       st[2 * b + 1];
      dg += d * xh;
      dbt += d;
    }
    reinterpret_cast<__nv_bfloat16*>(p.t_dgamma)[k] = __float2bfloat16_rn(dg);
    reinterpret_cast<__nv_bfloat16*>(p.t_dbeta)[k] = __float2bfloat16_rn(dbt);
  }
  if (!p.has_front) return;
  __syncthreads();

  // ---- dln[:, slab] = dlin . W[:, slab] ----
  {
    constexpr int NBQ = BT / 4;      // batch groups of four rows
    constexpr int MQ = 4 / NBQ;      // lane groups that split the rows m instead
    const int k = lane & 7, q = lane >> 3;
    const int bq = q % NBQ, mq = q / NBQ;
    const int rows = w / kBwdWarps;  // rows m of this warp (a multiple of 4)
    const int m0 = warp * rows;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint16_t* sl = reinterpret_cast<const uint16_t*>(slab);
#pragma unroll 2
    for (int m = m0 + 4 * mq; m < m0 + rows; m += 4 * MQ) {
      float wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) wv[u] = __uint_as_float((uint32_t)sl[(m + u) * kSlab + k] << 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 d = *reinterpret_cast<const float4*>(dl + (size_t)(bq + NBQ * i) * p.dl_stride + m);
        acc[i] = fmaf(wv[0], d.x, acc[i]);
        acc[i] = fmaf(wv[1], d.y, acc[i]);
        acc[i] = fmaf(wv[2], d.z, acc[i]);
        acc[i] = fmaf(wv[3], d.w, acc[i]);
      }
    }
    if (MQ > 1) {  // lanes of the same k and batch rows, different rows m
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 8);
        if (MQ > 2) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 16);
      }
    }
    if (mq == 0)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[(warp * BT + bq + NBQ * i) * kSlab + k] = acc[i];
    __syncthreads();
    if (tid < B * kSlab) {
      const int b = tid / kSlab, kk = tid - b * kSlab;
      float t = 0.f;
      for (int v = 0; v < kBwdWarps; ++v) t += red[(v * BT + b) * kSlab + kk];
      reinterpret_cast<__nv_bfloat16*>(p.f_dln)[(size_t)b * w + k0 + kk] = __float2bfloat16_rn(t);
    }
  }

}

// dW and db of every block, after the chain: dW_j[m][k] = bf16(sum_b
// dlin_j[b][m] ln_j[b][k]), db_j[m] = bf16(sum_b dlin_j[b][m]).  Nothing
// downstream of a block's backward reads them, so they are kept off the
// chain of launches (each of which waits for all of the previous one's
// stores) and written here in one pass at the HBM rate.  CTA (j, t) takes
// rows m0 = t*kDwRows .. m0+kDwRows-1 of block j; a thread forms whole
// 16-byte row chunks.  The sums run over b in order, as in the forward of
// the reading.
constexpr int kDwRows = 32;

struct DwParams {
  const uint16_t* dlin;  // [L][B][w] bf16
  const uint16_t* ln;    // [L][B][w] bf16
  uint16_t* const* dW;   // [L] pointers to [w][w] bf16
  uint16_t* const* db;   // [L] pointers to [w] bf16
  int B, w, tiles;       // tiles = w / kDwRows per block
};

__global__ void __launch_bounds__(kBwdThreads) k_mlp_dw(const __grid_constant__ DwParams p) {
  extern __shared__ __align__(16) float dws[];
  const int B = p.B, w = p.w;
  const int j = blockIdx.x / p.tiles, m0 = (blockIdx.x - j * p.tiles) * kDwRows;
  float* lnf = dws;                   // [B][w]
  float* dlf = dws + (size_t)B * w;   // [B][kDwRows]
  pdl_launch_dependents();
  pdl_wait();
  const size_t bw = (size_t)B * w;
  const uint16_t* lnj = p.ln + (size_t)j * bw;
  const uint16_t* dlj = p.dlin + (size_t)j * bw;
  for (int i = threadIdx.x; i < B * w / 8; i += kBwdThreads) {
    const uint4 v = __ldcg(reinterpret_cast<const uint4*>(lnj) + i);
    float4* d = reinterpret_cast<float4*>(lnf + 8 * i);
    d[0] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
    d[1] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
  }
  for (int i = threadIdx.x; i < B * kDwRows; i += kBwdThreads) {
    const int b = i / kDwRows, r = i - b * kDwRows;
    dlf[i] = __uint_as_float((uint32_t)__ldcg(dlj + (size_t)b * w + m0 + r) << 16);
  }
  __syncthreads();
  const int nch = w / kSlab;
  uint16_t* dW = p.dW[j];
  for (int i = threadIdx.x; i < kDwRows * nch; i += kBwdThreads) {
    const int r = i / nch, c = i - r * nch;
    float a[kSlab];
#pragma unroll
    for (int e = 0; e < kSlab; ++e) a[e] = 0.f;
    for (int b = 0; b < B; ++b) {
      const float d = dlf[b * kDwRows + r];
      const float4 l0 = *reinterpret_cast<const float4*>(lnf + (size_t)b * w + kSlab * c);
      const float4 l1 = *reinterpret_cast<const float4*>(lnf + (size_t)b * w + kSlab * c + 4);
      a[0] = fmaf(d, l0.x, a[0]);
      a[1] = fmaf(d, l0.y, a[1]);
      a[2] = fmaf(d, l0.z, a[2]);
      a[3] = fmaf(d, l0.w, a[3]);
      a[4] = fmaf(d, l1.x, a[4]);
      a[5] = fmaf(d, l1.y, a[5]);
      a[6] = fmaf(d, l1.z, a[6]);
      a[7] = fmaf(d, l1.w, a[7]);
    }
    reinterpret_cast<uint4*>(dW + (size_t)(m0 + r) * w)[c] =
        make_uint4(pack2_bf16(a[0], a[1]), pack2_bf16(a[2], a[3]), pack2_bf16(a[4], a[5]),
                   pack2_bf16(a[6], a[7]));
  }
  if (threadIdx.x < kDwRows) {
    float t = 0.f;
    for (int b = 0; b < B; ++b) t += dlf[b * kDwRows + threadIdx.x];
    reinterpret_cast<__nv_bfloat16*>(p.db[j])[m0 + threadIdx.x] = __float2bfloat16_rn(t);
  }
}

// -------------------------------------------------------------------------
// host side
// -------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static std::mutex mu;
  static EncodeTiledFn fn = nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  }
  return fn;
}

// The shared-memory layout of a launch at batch tile BT.
static void bwd_layout(BwdParams& p, int BT) {
  const int w = p.w, B = p.B;
  auto up = [](int v, int a) { return (v + a - 1) / a * a; };
  int off = 128;  // the mbarrier
  p.off_slab = off;
  off += up(p.nbox * p.R * 16, 128);
  p.off_x = off;
  off += up(B * w * 2, 128);
  p.off_g = off;
  off += up(B * w * 4, 128);
  // dlin rows w + 4 floats apart: the four batch rows lanes read together
  // (rows bq + NBQ i) fall in different bank groups
  p.dl_stride = w + 4;
  p.off_dl = off;
  off += up(BT * p.dl_stride * 4, 128);
  p.off_dln = off;
  off += up(B * w * 2, 128);
  p.off_red = off;
  off += up(kBwdWarps * BT * kSlab * 4 > 2 * kBwdWarps * BT * 4 ? kBwdWarps * BT * kSlab * 4
                                                                 : 2 * kBwdWarps * BT * 4,
            128);
  p.off_misc = off;
  off += up((4 * BT + BT * kSlab) * 4, 128);
  p.smem_bytes = off;
}

static bool bwd_prepare(int BT, int smem) {
  static std::mutex mu;
  static int done[64][2] = {{0}};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  int& d = done[dev][BT == 16];
  if (d >= smem) return true;
  const cudaError_t e =
      BT == 16 ? cudaFuncSetAttribute(k_mlp_backward<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
               : cudaFuncSetAttribute(k_mlp_backward<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return false;
  d = smem;
  return true;
}

static cudaError_t bwd_launch(const BwdParams& p, int BT, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.w / kSlab);
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return BT == 16 ? cudaLaunchKernelEx(&cfg, k_mlp_backward<16>, p)
                  : cudaLaunchKernelEx(&cfg, k_mlp_backward<4>, p);
}

// Two-sided 95% Student t quantile, rounded up for df between tabulated values.
static double t975_bwd(int df) {
  static const int dfs[] = {1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 12, 15, 20, 25, 30, 40, 60, 120};
  static const double ts[] = {12.706, 4.303, 3.182, 2.776, 2.571, 2.447, 2.365, 2.306, 2.262,
                              2.228,  2.179, 2.131, 2.086, 2.060, 2.042, 2.021, 2.000, 1.980};
  if (df < 1) return 1e30;
  double t = 1.960;
  for (int i = (int)(sizeof dfs / sizeof dfs[0]) - 1; i >= 0; --i)
    if (dfs[i] <= df) {
      t = ts[i];
      break;
    }
  return t;
}

}  // namespace ws

using namespace ws;

struct ws_mlp_backward {
  ws_mlp_backward_opts o;
  int L = 0, BT = 4;
  std::vector<BwdParams> launches;
  std::vector<std::pair<const void*, size_t>> reads;  // weight each launch reads (or empty)
  void* dln[2] = {nullptr, nullptr};
  void* dlin_buf = nullptr;       // every block's dlin when no trace is given
  uint16_t** d_tabs = nullptr;    // device tables: dW pointers, then db pointers
  DwParams dw;
  int dw_smem = 0;
  cudaStream_t cap = nullptr, side = nullptr;
  std::vector<cudaEvent_t> fork;
  cudaEvent_t join = nullptr;
  cudaGraphExec_t exec = nullptr;
  ws_prefetch_plan plan = {0, 0, 0, WS_PREFETCH_NONE};
  float gain_lo = 0.f, gain_mean = 0.f;
};

static void bwd_free(ws_mlp_backward* c) {
  if (!c) return;
  if (c->exec) cudaGraphExecDestroy(c->exec);
  for (cudaEvent_t e : c->fork) cudaEventDestroy(e);
  if (c->join) cudaEventDestroy(c->join);
  if (c->cap) cudaStreamDestroy(c->cap);
  if (c->side) cudaStreamDestroy(c->side);
  for (void* d : c->dln)
    if (d) cudaFree(d);
  if (c->dlin_buf) cudaFree(c->dlin_buf);
  if (c->d_tabs) cudaFree(c->d_tabs);
  delete c;
}

// Enqueue every launch on `st` with prefetch plan `pl` (mode NONE: none);
// used inside capture.
static ws_status bwd_enqueue(ws_mlp_backward* c, const ws_prefetch_plan& pl, bool decoy,
                             cudaStream_t st) {
  const int n = (int)c->launches.size();
  bool forked = false;
  for (int s = 0; s < n; ++s) {
    const int t = s + c->o.distance;
    if (pl.mode != WS_PREFETCH_NONE && t < n && c->reads[t].first) {
      // the decoy aims at the weight of the launch half a chain away
      int tg = t;
      if (decoy) {
        tg = (t + n / 2) % n;
        if (!c->reads[tg].first) tg = (tg + 1) % n;
      }
      if (cudaEventRecord(c->fork[s], st) != cudaSuccess ||
          cudaStreamWaitEvent(c->side, c->fork[s], 0) != cudaSuccess)
        return WS_ERR_CUDA;
      const ws_status r = ws_l2_prefetch(c->reads[tg].first, c->reads[tg].second, pl, c->side);
      if (r != WS_OK) return r;
      forked = true;
    }
    const cudaError_t e = bwd_launch(c->launches[s], c->BT, st, c->o.use_pdl && s > 0);
    if (e != cudaSuccess) {
      set_error("backward launch %d failed: %s", s, cudaGetErrorString(e));
      return WS_ERR_CUDA;
    }
  }
  // dW and db of every block, once every dlin is written
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c->L * c->dw.tiles);
    cfg.blockDim = dim3(kBwdThreads);
    cfg.dynamicSmemBytes = c->dw_smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = c->o.use_pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_mlp_dw, c->dw);
    if (e != cudaSuccess) {
      set_error("dW launch failed: %s", cudaGetErrorString(e));
      return WS_ERR_CUDA;
    }
  }
  if (forked) {
    if (cudaEventRecord(c->join, c->side) != cudaSuccess ||
        cudaStreamWaitEvent(st, c->join, 0) != cudaSuccess)
      return WS_ERR_CUDA;
  }
  return WS_OK;
}

static ws_status bwd_capture(ws_mlp_backward* c, const ws_prefetch_plan& pl, bool decoy,
                             cudaGraphExec_t* out) {
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    set_error("cudaStreamBeginCapture failed");
    return WS_ERR_CUDA;
  }
  const ws_status s = bwd_enqueue(c, pl, decoy, c->cap);
  const cudaError_t e = cudaStreamEndCapture(c->cap, &g);
  if (s != WS_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    if (s == WS_OK) set_error("capture failed: %s", cudaGetErrorString(e));
    cudaGetLastError();
    return s != WS_OK ? s : WS_ERR_CUDA;
  }
  const cudaError_t ie = cudaGraphInstantiate(out, g, 0);
  cudaGraphDestroy(g);
  if (ie != cudaSuccess) {
    set_error("graph instantiation failed: %s", cudaGetErrorString(ie));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

static bool al16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

extern "C" {

ws_status ws_mlp_backward_create(const ws_mlp_block* blocks, const ws_mlp_grads* grads, int n,
                                 const ws_mlp_backward_opts* opts, ws_mlp_backward** out) {
  if (!blocks || !grads || n <= 0 || !opts || !out) {
    set_error("bad arguments");
    return WS_ERR_ARG;
  }
  *out = nullptr;
  const ws_mlp_backward_opts& o = *opts;
  const int B = o.batch, w = o.width;
  if (B < 1 || B > kMaxBatch || w < kBwdWidthUnit || w > kBwdMaxWidth || w % kBwdWidthUnit != 0) {
    set_error("bad shape B=%d w=%d (need 1<=B<=16, %d<=w<=%d, w a multiple of %d)", B, w,
              kBwdWidthUnit, kBwdMaxWidth, kBwdWidthUnit);
    return WS_ERR_SHAPE;
  }
  if (o.distance < 1) {
    set_error("distance must be >= 1");
    return WS_ERR_ARG;
  }
  const void* need[] = {o.x_in, o.acts, o.ln, o.gelu_grad, o.ln_stats, o.dx};
  for (const void* q : need)
    if (!q || !al16(q)) {
      set_error("x_in, acts, ln, gelu_grad, ln_stats and dx must be 16-byte aligned device "
                "pointers");
      return WS_ERR_ALIGN;
    }
  if ((o.dz && !al16(o.dz)) || (o.dx_trace && !al16(o.dx_trace)) ||
      (o.dlin_trace && !al16(o.dlin_trace)) || (o.dln_trace && !al16(o.dln_trace))) {
    set_error("dz and the traces must be 16-byte aligned");
    return WS_ERR_ALIGN;
  }
  for (int i = 0; i < n; ++i) {
    const void* q[] = {blocks[i].gamma, blocks[i].W, grads[i].dW, grads[i].db, grads[i].dgamma,
                       grads[i].dbeta};
    for (const void* v : q)
      if (!v || !al16(v)) {
        set_error("block %d: weights and gradients must be 16-byte aligned", i);
        return WS_ERR_ALIGN;
      }
  }
  EncodeTiledFn enc = encode_tiled();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return WS_ERR_CUDA;
  }
  ws_mlp_backward* c = new ws_mlp_backward();
  c->o = o;
  c->L = n;
  c->BT = B <= 4 ? 4 : 16;
  const size_t bw = (size_t)B * w;
  auto bf = [](const void* base, size_t off) {
    return static_cast<const uint16_t*>(base) + off;
  };
  auto bfw = [](void* base, size_t off) { return base ? static_cast<uint16_t*>(base) + off : nullptr; };
  if (!o.dln_trace)
    for (int i = 0; i < 2; ++i)
      if (cudaMalloc(&c->dln[i], bw * 2) != cudaSuccess) {
        bwd_free(c);
        return WS_ERR_NOMEM;
      }
  auto dln_of = [&](int j) -> uint16_t* {
    return o.dln_trace ? static_cast<uint16_t*>(o.dln_trace) + (size_t)j * bw
                       : static_cast<uint16_t*>(c->dln[j % 2]);
  };
  // every block's dlin (the trace, or the handle's own rows) for the dW pass
  void* dlin_base = o.dlin_trace;
  if (!dlin_base) {
    if (cudaMalloc(&c->dlin_buf, (size_t)n * bw * 2) != cudaSuccess) {
      bwd_free(c);
      return WS_ERR_NOMEM;
    }
    dlin_base = c->dlin_buf;
  }
  {
    std::vector<uint16_t*> tw(n), tb(n);
    for (int i = 0; i < n; ++i) {
      tw[i] = static_cast<uint16_t*>(grads[i].dW);
      tb[i] = static_cast<uint16_t*>(grads[i].db);
    }
    if (cudaMalloc((void**)&c->d_tabs, sizeof(uint16_t*) * 2 * n) != cudaSuccess) {
      bwd_free(c);
      return WS_ERR_NOMEM;
    }
    if (cudaMemcpy(c->d_tabs, tw.data(), sizeof(uint16_t*) * n, cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(c->d_tabs + n, tb.data(), sizeof(uint16_t*) * n, cudaMemcpyHostToDevice) !=
            cudaSuccess) {
      bwd_free(c);
      return WS_ERR_CUDA;
    }
    c->dw.dlin = static_cast<const uint16_t*>(dlin_base);
    c->dw.ln = static_cast<const uint16_t*>(o.ln);
    c->dw.dW = c->d_tabs;
    c->dw.db = c->d_tabs + n;
    c->dw.B = B;
    c->dw.w = w;
    c->dw.tiles = w / kDwRows;
    c->dw_smem = (int)(((size_t)B * w + (size_t)B * kDwRows) * 4);
    if (cudaFuncSetAttribute(k_mlp_dw, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             c->dw_smem) != cudaSuccess) {
      set_error("could not configure the dW kernel");
      bwd_free(c);
      return WS_ERR_CUDA;
    }
  }
  const int R = w < 256 ? w : 256, nbox = (w + R - 1) / R;
  for (int s = 0; s <= n; ++s) {
    BwdParams p;
    memset(&p, 0, sizeof p);
    p.B = B;
    p.w = w;
    p.R = R;
    p.nbox = nbox;
    p.err = device_error_ptr();
    p.timeout_ns = tuning().timeout_ns;
    const int j = n - 1 - s;  // front block (-1: none)
    if (s > 0) {              // tail of block j + 1
      const int t = j + 1;
      p.t_dln = dln_of(t);
      p.t_x = t == 0 ? static_cast<const uint16_t*>(o.x_in) : bf(o.acts, (size_t)(t - 1) * bw);
      p.t_stats = o.ln_stats + (size_t)t * B * 2;
      p.t_gamma = static_cast<const uint16_t*>(blocks[t].gamma);
      p.t_dx = t == 0 ? static_cast<uint16_t*>(o.dx) : bfw(o.dx_trace, (size_t)t * bw);
      p.t_dx2 = t == 0 ? bfw(o.dx_trace, 0) : nullptr;
      p.t_dgamma = static_cast<uint16_t*>(grads[t].dgamma);
      p.t_dbeta = static_cast<uint16_t*>(grads[t].dbeta);
    }
    if (j >= 0) {
      p.has_front = 1;
      if (s == 0) {
        p.dz = static_cast<const uint16_t*>(o.dz);
        p.z_loss = bf(o.acts, (size_t)(n - 1) * bw);
        p.loss_scale = 2.0f / (float)(B * w);
        p.dz_out = bfw(o.dx_trace, (size_t)n * bw);
      }
      p.f_gelu = o.gelu_grad + (size_t)j * bw;
      p.f_dlin = static_cast<uint16_t*>(dlin_base) + (size_t)j * bw;
      p.f_dln = dln_of(j);
      const cuuint64_t dims[2] = {(cuuint64_t)w, (cuuint64_t)w};
      const cuuint64_t strides[1] = {(cuuint64_t)w * 2};
      const cuuint32_t box[2] = {(cuuint32_t)kSlab, (cuuint32_t)R};
      const cuuint32_t es[2] = {1, 1};
      const CUresult r = enc(&p.tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                             const_cast<void*>(blocks[j].W), dims, strides, box, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) {
        set_error("tensor map of block %d's weight failed (%d)", j, (int)r);
        bwd_free(c);
        return WS_ERR_CUDA;
      }
      c->reads.push_back({blocks[j].W, (size_t)w * w * 2});
    } else {
      c->reads.push_back({nullptr, 0});
    }
    bwd_layout(p, c->BT);
    c->launches.push_back(p);
  }
  const int smem = c->launches[0].smem_bytes;
  if (!bwd_prepare(c->BT, smem)) {
    set_error("could not configure the backward kernel (%d bytes of shared memory)", smem);
    bwd_free(c);
    return WS_ERR_CUDA;
  }
  c->fork.resize(c->launches.size(), nullptr);
  bool ok = cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&c->join, cudaEventDisableTiming) == cudaSuccess;
  for (auto& e : c->fork) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    set_error("could not create streams or events");
    bwd_free(c);
    return WS_ERR_CUDA;
  }
  if (o.prefetch == 2) c->plan = o.fixed_plan;
  *out = c;
  return WS_OK;
}

ws_status ws_mlp_backward_tune(ws_mlp_backward* c, ws_stream_t stream) {
  if (!c) {
    set_error("null handle");
    return WS_ERR_ARG;
  }
  (void)stream;
  if (c->o.prefetch != 1) return WS_OK;
  const int pairs = c->o.tune_pairs < 8 ? 8 : c->o.tune_pairs;
  const ws_prefetch_plan none = {0, 0, 0, WS_PREFETCH_NONE};
  std::vector<ws_prefetch_plan> cands;
  for (int blocks : {4, 16, 64}) {
    cands.push_back({blocks, 256, 128, WS_PREFETCH_L2});
    cands.push_back({blocks, 256, 16384, WS_PREFETCH_BULK});
  }
  cudaGraphExec_t g0 = nullptr;
  ws_status st = bwd_capture(c, none, false, &g0);
  if (st != WS_OK) return st;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaGraphExecDestroy(g0);
    return WS_ERR_CUDA;
  }
  auto time_one = [&](cudaGraphExec_t g, float* ms) -> bool {
    return cudaEventRecord(e0, c->cap) == cudaSuccess && cudaGraphLaunch(g, c->cap) == cudaSuccess &&
           cudaEventRecord(e1, c->cap) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
           cudaEventElapsedTime(ms, e0, e1) == cudaSuccess;
  };
  ws_prefetch_plan best = none;
  double best_lo = -1e30, best_mean = 0.0;
  for (const ws_prefetch_plan& pl : cands) {
    cudaGraphExec_t g1 = nullptr;
    st = bwd_capture(c, pl, false, &g1);
    if (st != WS_OK) break;
    float t;
    for (int wu = 0; wu < 3; ++wu) {  // warm-up
      time_one(g0, &t);
      time_one(g1, &t);
    }
    std::vector<double> gains;
    for (int i = 0; i < pairs && st == WS_OK; ++i) {
      float a = 0.f, b = 0.f;
      const bool ok = (i & 1) ? (time_one(g1, &b) && time_one(g0, &a))
                              : (time_one(g0, &a) && time_one(g1, &b));
      if (!ok) st = WS_ERR_CUDA;
      else gains.push_back((a - b) / a);
    }
    cudaGraphExecDestroy(g1);
    if (st != WS_OK) break;
    double mean = 0.0, var = 0.0;
    for (double g : gains) mean += g;
    mean /= gains.size();
    for (double g : gains) var += (g - mean) * (g - mean);
    var /= gains.size() > 1 ? gains.size() - 1 : 1;
    const double lo = mean - t975_bwd((int)gains.size() - 1) * std::sqrt(var / gains.size());
    if (lo > best_lo) {
      best_lo = lo;
      best_mean = mean;
      best = pl;
    }
  }
  cudaGraphExecDestroy(g0);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st != WS_OK) return st;
  c->gain_lo = (float)best_lo;
  c->gain_mean = (float)best_mean;
  c->plan = best_lo > c->o.tune_min_gain ? best : none;
  return WS_OK;
}

ws_status ws_mlp_backward_capture(ws_mlp_backward* c, ws_stream_t stream) {
  if (!c) {
    set_error("null handle");
    return WS_ERR_ARG;
  }
  (void)stream;
  if (c->exec) {
    cudaGraphExecDestroy(c->exec);
    c->exec = nullptr;
  }
  const ws_prefetch_plan none = {0, 0, 0, WS_PREFETCH_NONE};
  return bwd_capture(c, c->o.prefetch ? c->plan : none, c->o.decoy != 0, &c->exec);
}

ws_status ws_mlp_backward_run(ws_mlp_backward* c, ws_stream_t stream) {
  if (!c) {
    set_error("null handle");
    return WS_ERR_ARG;
  }
  if (!c->exec) {
    set_error("backward not captured");
    return WS_ERR_STATE;
  }
  const cudaError_t e = cudaGraphLaunch(c->exec, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    set_error("graph launch failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

ws_status ws_mlp_backward_plan(const ws_mlp_backward* c, ws_prefetch_plan* plan, float* gain_lo,
                               float* gain_mean) {
  if (!c) {
    set_error("null handle");
    return WS_ERR_ARG;
  }
  if (plan) *plan = c->plan;
  if (gain_lo) *gain_lo = c->gain_lo;
  if (gain_mean) *gain_mean = c->gain_mean;
  return WS_OK;
}

int ws_mlp_backward_num_launches(const ws_mlp_backward* c) {
  return c ? (int)c->launches.size() + 1 : 0;
}

void ws_mlp_backward_destroy(ws_mlp_backward* c) { bwd_free(c); }

}  // extern "C"
