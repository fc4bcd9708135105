// ws_attention.cu -- decode attention over a key-value cache, one new token
// per batch row ("Making small PyTorch ops faster on a laptop GPU", "A full
// decode step is a different story": append the new key and value, an FP32
// softmax, the cache split across blocks, the last block to finish merging
// the partial results; "One Token, Kernel by Kernel", "The fix: Part 10's
// split-KV kernel": the (batch, head, slot, dimension) cache layout, the
// valid length read on the GPU at run time so that a CUDA graph can be
// replayed, one key-value head read once for all of its query heads).
//
// Design for GB300: the group's G <= 8 query heads make the scores a
// product [16 slots x 128] x [128 x 8 heads] and the output a product
// [128 x 16 slots] x [16 slots x 8 heads] per tile of 16 cached slots, done
// with warp-level bf16 tensor-core MMAs (m16n8k16, fp32 accumulators).  The
// fp32 queries and probabilities enter as a pair of bf16 terms (hi + lo,
// relative error 2^-17), the keys and values are bf16 already, so the
// products match an fp32 computation to well under the fp32 test bound.
// Softmax is online and in fp32, per warp, over its tiles.
//
// One CTA of four warps per (split, key-value head, batch row).  A split is a
// run of tiles sized on the device from the actual length so that the grid's
// CTAs share the cache evenly; warp w takes tiles w, w + 4, ... of its split.
// Each warp streams its tiles through its own two-stage ring: 32 row copies
// of 256 bytes (16 key rows, 16 value rows, one 1-D bulk async copy per lane)
// into rows of 272 bytes, so the ldmatrix reads of 8 rows hit 8 different
// bank groups.  The new token's row is written to the cache and to the ring
// by the warp whose tile holds it (the copies stop short of it); rows past it
// are zero-filled, so a tile never reads a slot it does not own.  At the end
// the four warps' (max, sum, acc) are combined in shared memory; a single
// split writes the output, otherwise the split writes a partial result, the
// last split of each group of 16 (an atomic ticket, reset by that split for
// the next replay) merges the group in split order, and with more than one
// group the last group merges the groups.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include <cstdint>
#include <cstring>

#include "wsgemv.h"
#include "ws_common.cuh"
#include "ws_device.cuh"

namespace ws {

constexpr int kAttnDim = 128;              // head dimension
constexpr int kAttnTile = 16;              // slots per tile (one MMA's rows)
constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kAttnStages = 2;             // ring stages per warp
constexpr int kAttnPitch = kAttnDim * 2 + 16;  // bytes per staged row
constexpr int kAttnStageBytes = 2 * kAttnTile * kAttnPitch;  // keys then values
constexpr int kAttnMaxG = 8;               // query heads per key-value head (MMA columns)
constexpr int kAttnGroup = 16;             // splits merged by one first-level merge
constexpr int kPartStride = kAttnDim + 2;  // one partial result: acc[128], max, sum
constexpr int kDerrBadPos = 2;             // device error flag: a position outside the cache

// ring, then per barrier one mbarrier per (warp, stage)
constexpr int kAttnSmem = kAttnWarps * kAttnStages * kAttnStageBytes;
static_assert(kAttnSmem >= kAttnWarps * kAttnMaxG * kAttnDim * 4 + 256 * kAttnMaxG * 4,
              "combine area and merge weights fit the ring");

struct AttnParams {
  const float* q;      // [B][nh * 128]
  const float* k_new;  // [B][nkv * 128]
  const float* v_new;
  uint16_t* k_cache;   // bf16 [B][nkv][S][128]
  uint16_t* v_cache;
  const int* pos;      // [B]: slot of the new token
  float* out_f32;      // optional [B][nh * 128]
  uint16_t* out_bf16;  // optional bf16 [B][nh * 128]
  int nh, nkv, S, G;
  float scale;         // 1 / sqrt(128)
  float* part0;        // [B][nkv][max splits][G][130]: per split
  float* part1;        // [B][nkv][groups][G][130]: per group of 16 splits
  unsigned* tick0;     // [B][nkv][groups]
  unsigned* tick1;     // [B][nkv]
  int* err;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi), two values per word
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = bf16x2_bits(a - __low2float(h), b - __high2float(h));
}

// Ticket of a merge: the CTA's writes precede thread 0's release (they come
// before a CTA barrier), and the last arrival's acquire precedes the merge's
// reads (they come after the next barrier), so one thread fences, not all.
__device__ __forceinline__ unsigned ticket_acq_rel(unsigned* p) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Merge of n partial results (acc, max, sum) for the G heads, by the whole
// CTA, thread t = dimension t: M = max m_c, L = sum e^(m_c - M) l_c,
// O = sum e^(m_c - M) acc_c.  Warp 0 forms M, L and the weights e^(m_c - M)
// from one pass of loads (each lane an online max and sum over its entries,
// combined across the warp) while every thread already has its first eight
// entries' values in flight.  wsm holds n x 8 weights, hsm M then L per head.
constexpr int kMergeBatch = 8;
constexpr int kMergeMax = 256;  // entries one merge takes (weights buffer)

__device__ __forceinline__ void merge_cta(const float* src, int n, int G, int t, float* wsm,
                                          float* hsm, float (&O)[kAttnMaxG]) {
  // every load is unconditional (entry and head indices clamped into range,
  // the extra values unused), so a thread's loads are all in flight at once
  const int lane = t & 31;
  int hc[kAttnMaxG];
#pragma unroll
  for (int h = 0; h < kAttnMaxG; ++h) hc[h] = min(h, G - 1);
  float x[kMergeBatch][kAttnMaxG];
#pragma unroll
  for (int c = 0; c < kMergeBatch; ++c)
#pragma unroll
    for (int h = 0; h < kAttnMaxG; ++h)
      x[c][h] = __ldcg(src + ((size_t)min(c, n - 1) * G + hc[h]) * kPartStride + t);
  if (t < 32) {
    float mr[kAttnMaxG], lr[kAttnMaxG];
#pragma unroll
    for (int h = 0; h < kAttnMaxG; ++h) {
      mr[h] = -INFINITY;
      lr[h] = 0.f;
    }
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int c = c0 + lane;
      float m[kAttnMaxG], l[kAttnMaxG];
#pragma unroll
      for (int h = 0; h < kAttnMaxG; ++h) {
        const float* e = src + ((size_t)min(c, n - 1) * G + hc[h]) * kPartStride + kAttnDim;
        m[h] = __ldcg(e);
        l[h] = __ldcg(e + 1);
      }
      if (c < n) {
#pragma unroll
        for (int h = 0; h < kAttnMaxG; ++h) {
          wsm[c * kAttnMaxG + h] = m[h];
          const float mn = fmaxf(mr[h], m[h]);
          lr[h] = fmaf(lr[h], expf(mr[h] - mn), l[h] * expf(m[h] - mn));
          mr[h] = mn;
        }
      }
    }
    float M[kAttnMaxG], L[kAttnMaxG];
#pragma unroll
    for (int h = 0; h < kAttnMaxG; ++h) M[h] = mr[h];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int h = 0; h < kAttnMaxG; ++h) M[h] = fmaxf(M[h], __shfl_xor_sync(0xffffffffu, M[h], off));
#pragma unroll
    for (int h = 0; h < kAttnMaxG; ++h) L[h] = lr[h] * expf(mr[h] - M[h]);  // 0 without entries
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int h = 0; h < kAttnMaxG; ++h) L[h] += __shfl_xor_sync(0xffffffffu, L[h], off);
    if (lane < kAttnMaxG) {
      hsm[lane] = M[0];
      hsm[kAttnMaxG + lane] = L[0];
#pragma unroll
      for (int h = 1; h < kAttnMaxG; ++h)
        if (lane == h) {
          hsm[lane] = M[h];
          hsm[kAttnMaxG + lane] = L[h];
        }
    }
    for (int c = lane; c < n; c += 32)
#pragma unroll
      for (int h = 0; h < kAttnMaxG; ++h)
        wsm[c * kAttnMaxG + h] = expf(wsm[c * kAttnMaxG + h] - M[h]);
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < kAttnMaxG; ++h) O[h] = 0.f;
  for (int c0 = 0; c0 < n; c0 += kMergeBatch) {
    if (c0 > 0) {
#pragma unroll
      for (int c = 0; c < kMergeBatch; ++c)
#pragma unroll
        for (int h = 0; h < kAttnMaxG; ++h)
          x[c][h] = __ldcg(src + ((size_t)min(c0 + c, n - 1) * G + hc[h]) * kPartStride + t);
    }
#pragma unroll
    for (int c = 0; c < kMergeBatch; ++c)
      if (c0 + c < n)
#pragma unroll
        for (int h = 0; h < kAttnMaxG; ++h) O[h] = fmaf(wsm[(c0 + c) * kAttnMaxG + h], x[c][h], O[h]);
  }
}

// The new token's key and value (the whole warp, 4 dimensions a lane), rounded
// to bf16, into row pos - 16 tile of a ring stage and into slot pos of the
// cache.
__device__ __forceinline__ void stage_new_row(const AttnParams& a, size_t row0, size_t kvn,
                                              int tile, int pos, unsigned char* st, int lane) {
  const int rp = pos - tile * kAttnTile;
  const float4 kf = *reinterpret_cast<const float4*>(a.k_new + kvn + lane * 4);
  const float4 vf = *reinterpret_cast<const float4*>(a.v_new + kvn + lane * 4);
  const uint2 ku = make_uint2(bf16x2_bits(kf.x, kf.y), bf16x2_bits(kf.z, kf.w));
  const uint2 vu = make_uint2(bf16x2_bits(vf.x, vf.y), bf16x2_bits(vf.z, vf.w));
  *reinterpret_cast<uint2*>(st + rp * kAttnPitch + lane * 8) = ku;
  *reinterpret_cast<uint2*>(st + (kAttnTile + rp) * kAttnPitch + lane * 8) = vu;
  *reinterpret_cast<uint2*>(a.k_cache + (row0 + pos) * kAttnDim + lane * 4) = ku;
  *reinterpret_cast<uint2*>(a.v_cache + (row0 + pos) * kAttnDim + lane * 4) = vu;
}

// Stage tile `tile` (slots 16 tile .. 16 tile + 15) of one (row, head) into a
// warp's ring stage: lane l copies key row l (l < 16) or value row l - 16 of
// the slots before pos; later slots are zero; the slot pos comes from the new
// key and value (stage_new_row), here unless with_new is false (the tiles
// staged before the dependency wait: the new key and value come from the
// previous kernel).
__device__ __forceinline__ void stage_tile(const AttnParams& a, size_t row0, size_t kvn, int tile,
                                           int pos, unsigned char* st, uint64_t* bar, int lane,
                                           uint64_t pol, bool with_new) {
  const int slot0 = tile * kAttnTile;
  const int ncopy = max(0, min(kAttnTile, pos - slot0));  // cached rows of this tile
  if (lane == 0) mbar_arrive_expect_tx(bar, 2u * ncopy * kAttnDim * 2);
  __syncwarp();
  const int r = lane & (kAttnTile - 1);
  const bool is_v = lane >= kAttnTile;
  unsigned char* dst = st + (is_v ? kAttnTile * kAttnPitch : 0) + r * kAttnPitch;
  if (r < ncopy) {
    fence_proxy_async_smem();  // earlier generic writes of this stage before the copy
    const uint16_t* src = (is_v ? a.v_cache : a.k_cache) + (row0 + slot0 + r) * kAttnDim;
    bulk_copy_g2s(dst, src, kAttnDim * 2, bar, pol);
  } else if (slot0 + r > pos) {
    uint4* z = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < kAttnDim * 2 / 16; ++i) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (with_new && pos >= slot0 && pos < slot0 + kAttnTile)
    stage_new_row(a, row0, kvn, tile, pos, st, lane);
  __syncwarp();  // generic rows visible to the warp's ldmatrix
}

// out[h][d] = O[h] / L[h] for the G heads of key-value head g (L in hsm[8..15])
__device__ __forceinline__ void write_heads(const AttnParams& a, int b, int g, int d,
                                            const float (&O)[kAttnMaxG], const float* hsm) {
#pragma unroll
  for (int h = 0; h < kAttnMaxG; ++h) {
    if (h < a.G) {
      const float v = O[h] / hsm[kAttnMaxG + h];
      const size_t oi = ((size_t)b * a.nh + (size_t)g * a.G + h) * kAttnDim + d;
      if (a.out_f32) a.out_f32[oi] = v;
      if (a.out_bf16) a.out_bf16[oi] = to_bf16_bits(v);
    }
  }
}

__global__ void __launch_bounds__(kAttnThreads)
    k_decode_attention(const __grid_constant__ AttnParams a) {
  const int g = blockIdx.y, b = blockIdx.z, G = a.G;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // inside a chain (programmatic dependent launch) the next op may start its
  // prologue now; the cached rows stream in before the wait on the previous
  // op (the QKV product), which only q and the new key and value need
  pdl_launch_dependents();
  const int pos = a.pos[b];
  if (pos < 0 || pos >= a.S) {  // no access outside the cache
    if (t == 0 && blockIdx.x == 0) atomicExch(a.err, kDerrBadPos);
    return;
  }
  // splits: tiles per split a multiple of the warps, at most gridDim.x
  // splits; at most one merge group (16 splits) while that keeps a split at
  // 32 tiles or fewer, since a second merge level costs more (three more
  // round trips to L2) than the longer splits
  const int ntiles = (pos + kAttnTile) / kAttnTile;
  int tps = (ntiles + gridDim.x - 1) / gridDim.x;
  tps = (tps + kAttnWarps - 1) / kAttnWarps * kAttnWarps;
  int tps_one = (ntiles + kAttnGroup - 1) / kAttnGroup;
  tps_one = (tps_one + kAttnWarps - 1) / kAttnWarps * kAttnWarps;
  if (tps_one <= 8 * kAttnWarps && tps_one > tps) tps = tps_one;
  const int nsplits = (ntiles + tps - 1) / tps;
  const int split = blockIdx.x;
  if (split >= nsplits) return;
  const int t0 = split * tps, t1 = min(t0 + tps, ntiles);
  const int nt = t1 - t0 > warp ? (t1 - t0 - warp + kAttnWarps - 1) / kAttnWarps : 0;

  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t full[kAttnWarps][kAttnStages];
  __shared__ float cm[kAttnWarps][kAttnMaxG], cl[kAttnWarps][kAttnMaxG];
  __shared__ int last;
  unsigned char* ring = smem + warp * kAttnStages * kAttnStageBytes;

  const size_t bg = (size_t)b * a.nkv + g;
  const size_t row0 = bg * a.S;           // slot 0 of this head's cache
  const size_t kvn = bg * kAttnDim;       // this head's new key and value
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kAttnStages; ++s) mbar_init(&full[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t pol = l2_policy_evict_normal();
#pragma unroll
  for (int s = 0; s < kAttnStages; ++s)
    if (s < nt)
      stage_tile(a, row0, kvn, t0 + warp + s * kAttnWarps, pos, ring + s * kAttnStageBytes,
                 &full[warp][s], lane, pol, false);
  pdl_wait();
#pragma unroll
  for (int s = 0; s < kAttnStages; ++s) {
    const int tile = t0 + warp + s * kAttnWarps;
    if (s < nt && pos >= tile * kAttnTile && pos < (tile + 1) * kAttnTile) {
      stage_new_row(a, row0, kvn, tile, pos, ring + s * kAttnStageBytes, lane);
      __syncwarp();
    }
  }
  // the queries as the MMA's B operand: lane holds head lane / 4, dimensions
  // 16 k + 2 (lane % 4) + {0, 1} and + 8, as hi and lo bf16 terms
  uint32_t qh[8][2], ql[8][2];
  {
    // heads past G read head 0's row (all loads unconditional, in flight
    // together) and are zeroed
    const int h = lane >> 2, c = (lane & 3) * 2;
    const float* qr = a.q + ((size_t)b * a.nh + (size_t)g * G + (h < G ? h : 0)) * kAttnDim;
    float2 x0[8], x1[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x0[k] = *reinterpret_cast<const float2*>(qr + k * 16 + c);
      x1[k] = *reinterpret_cast<const float2*>(qr + k * 16 + 8 + c);
    }
    const float z = h < G ? 1.f : 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      split_bf16x2(x0[k].x * z, x0[k].y * z, qh[k][0], ql[k][0]);
      split_bf16x2(x1[k].x * z, x1[k].y * z, qh[k][1], ql[k][1]);
    }
  }


  // per lane: heads c, c + 1 of the accumulators (c = 2 (lane % 4)), dims
  // 16 mt + lane / 4 and + 8
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool abort = false;
  const int rq = lane >> 2;  // this lane's slot rows rq, rq + 8 of a tile

  for (int i = 0; i < nt; ++i) {
    const int s = i % kAttnStages;
    const uint32_t par = (i / kAttnStages) & 1;
    const bool ok = abort || mbar_wait_bounded(&full[warp][s], par, a.timeout_ns);
    if (__any_sync(0xffffffffu, !ok) && !abort) {
      abort = true;
      if (lane == 0) atomicExch(a.err, (int)DERR_TIMEOUT);
    }
    if (abort) continue;
    const int tile = t0 + warp + i * kAttnWarps;
    const unsigned char* st = ring + s * kAttnStageBytes;
    const uint32_t sK = smem_addr(st), sV = sK + kAttnTile * kAttnPitch;

    // scores S[slot][head] over the 8 k-steps of 16 dimensions
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const uint32_t base = sK + ((lane & 7) + ((lane >> 3) & 1) * 8) * kAttnPitch + (lane >> 4) * 16;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(base + k * 32, a0, a1, a2, a3);
        mma_bf16_16816(sc, a0, a1, a2, a3, qh[k][0], qh[k][1]);
        mma_bf16_16816(sc, a0, a1, a2, a3, ql[k][0], ql[k][1]);
      }
    }
    const int sl = tile * kAttnTile + rq;
    const bool v0 = sl <= pos, v1 = sl + 8 <= pos;
    sc[0] = v0 ? sc[0] * a.scale : -INFINITY;
    sc[1] = v0 ? sc[1] * a.scale : -INFINITY;
    sc[2] = v1 ? sc[2] * a.scale : -INFINITY;
    sc[3] = v1 ? sc[3] * a.scale : -INFINITY;
    float t0m = fmaxf(sc[0], sc[2]), t1m = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      t0m = fmaxf(t0m, __shfl_xor_sync(0xffffffffu, t0m, off));
      t1m = fmaxf(t1m, __shfl_xor_sync(0xffffffffu, t1m, off));
    }
    const float n0 = fmaxf(m0, t0m), n1 = fmaxf(m1, t1m);
    const float r0 = expf(m0 - n0), r1 = expf(m1 - n1);
    m0 = n0;
    m1 = n1;
    const float p0 = expf(sc[0] - n0), p1 = expf(sc[1] - n1);
    const float p2 = expf(sc[2] - n0), p3 = expf(sc[3] - n1);
    l0 = fmaf(l0, r0, p0 + p2);
    l1 = fmaf(l1, r1, p1 + p3);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= r0;
      o[mt][1] *= r1;
      o[mt][2] *= r0;
      o[mt][3] *= r1;
    }
    // P as the B operand [16 slots][8 heads]: the score fragment transposed
    uint32_t h01, l01, h23, l23;
    split_bf16x2(p0, p1, h01, l01);
    split_bf16x2(p2, p3, h23, l23);
    const uint32_t bh0 = movmatrix_t(h01), bh1 = movmatrix_t(h23);
    const uint32_t bl0 = movmatrix_t(l01), bl1 = movmatrix_t(l23);
    {
      const uint32_t base = sV + ((lane & 7) + (lane >> 4) * 8) * kAttnPitch + ((lane >> 3) & 1) * 16;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(base + mt * 32, a0, a1, a2, a3);
        mma_bf16_16816(o[mt], a0, a1, a2, a3, bh0, bh1);
        mma_bf16_16816(o[mt], a0, a1, a2, a3, bl0, bl1);
      }
    }
    // every lane's reads of this stage fed the MMAs above: refill it
    __syncwarp();
    if (i + kAttnStages < nt)
      stage_tile(a, row0, kvn, tile + kAttnStages * kAttnWarps, pos, ring + s * kAttnStageBytes,
                 &full[warp][s], lane, pol, true);
  }
  if (abort && lane == 0) {
    // no copy may land after the CTA exits: wait (bounded) for the stages
    for (int i = max(0, nt - kAttnStages); i < nt; ++i)
      mbar_wait_bounded(&full[warp][i % kAttnStages], (i / kAttnStages) & 1, a.timeout_ns);
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  if (__syncthreads_or(abort)) return;

  // the four warps' results through the ring (no longer read)
  float* co = reinterpret_cast<float*>(smem);  // [warp][head][128]
  {
    const int c = (lane & 3) * 2;
    if (lane < 4) {
      cm[warp][c] = m0;
      cm[warp][c + 1] = m1;
      cl[warp][c] = l0;
      cl[warp][c + 1] = l1;
    }
    float* cw = co + (size_t)warp * kAttnMaxG * kAttnDim;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d = mt * 16 + rq;
      cw[c * kAttnDim + d] = o[mt][0];
      cw[(c + 1) * kAttnDim + d] = o[mt][1];
      cw[c * kAttnDim + d + 8] = o[mt][2];
      cw[(c + 1) * kAttnDim + d + 8] = o[mt][3];
    }
  }
  __syncthreads();
  const int d = t;  // one dimension per thread
  const bool single = nsplits == 1;
  const int maxs = a.S / (kAttnTile * kAttnWarps);
  const int maxg = (maxs + kAttnGroup - 1) / kAttnGroup;
  float* dst0 = a.part0 + (bg * maxs + split) * G * kPartStride;
  // all heads at once (unrolled over 8, heads past G unused): the shared
  // memory reads and exponentials of different heads overlap
  float Mh[kAttnMaxG], Lh[kAttnMaxG], Oh[kAttnMaxG];
#pragma unroll
  for (int h = 0; h < kAttnMaxG; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, cm[w][h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float e = expf(cm[w][h] - M);  // 0 for a warp without tiles
      L = fmaf(e, cl[w][h], L);
      O = fmaf(e, co[((size_t)w * kAttnMaxG + h) * kAttnDim + d], O);
    }
    Mh[h] = M;
    Lh[h] = L;
    Oh[h] = O;
  }
#pragma unroll
  for (int h = 0; h < kAttnMaxG; ++h) {
    if (h < G) {
      if (single) {
        const float v = Oh[h] / Lh[h];
        const size_t oi = ((size_t)b * a.nh + (size_t)g * G + h) * kAttnDim + d;
        if (a.out_f32) a.out_f32[oi] = v;
        if (a.out_bf16) a.out_bf16[oi] = to_bf16_bits(v);
      } else {
        dst0[h * kPartStride + d] = Oh[h];
        if (d == 0) {
          dst0[h * kPartStride + kAttnDim] = Mh[h];
          dst0[h * kPartStride + kAttnDim + 1] = Lh[h];
        }
      }
    }
  }
  if (single) return;

  // the ticket of this split's group
  const int grp = split / kAttnGroup, ngroups = (nsplits + kAttnGroup - 1) / kAttnGroup;
  const int gsize = min(kAttnGroup, nsplits - grp * kAttnGroup);
  __syncthreads();
  if (t == 0) {
    unsigned* tk = a.tick0 + bg * maxg + grp;
    const unsigned old = ticket_acq_rel(tk);
    last = old == (unsigned)(gsize - 1);
    if (last) atomicExch(tk, 0u);
  }
  __syncthreads();
  if (!last) return;
  float* wsm = reinterpret_cast<float*>(smem + kAttnWarps * kAttnMaxG * kAttnDim * 4);
  float* hsm = cm[0];  // M then L per head (the warp maxima are no longer read)
  float O[kAttnMaxG];
  const float* src0 = a.part0 + (bg * maxs + (size_t)grp * kAttnGroup) * G * kPartStride;
  merge_cta(src0, gsize, G, t, wsm, hsm, O);
  if (ngroups == 1) {
    write_heads(a, b, g, d, O, hsm);
    return;
  }
  float* dst1 = a.part1 + (bg * maxg + grp) * G * kPartStride;
#pragma unroll
  for (int h = 0; h < kAttnMaxG; ++h) {
    if (h < G) {
      dst1[h * kPartStride + d] = O[h];
      if (d == 0) {
        dst1[h * kPartStride + kAttnDim] = hsm[h];
        dst1[h * kPartStride + kAttnDim + 1] = hsm[kAttnMaxG + h];
      }
    }
  }

  // the ticket of the (row, head)
  __syncthreads();
  if (t == 0) {
    unsigned* tk = a.tick1 + bg;
    const unsigned old = ticket_acq_rel(tk);
    last = old == (unsigned)(ngroups - 1);
    if (last) atomicExch(tk, 0u);
  }
  __syncthreads();
  if (!last) return;
  merge_cta(a.part1 + bg * maxg * G * kPartStride, ngroups, G, t, wsm, hsm, O);
  write_heads(a, b, g, d, O, hsm);
}

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct AttnLayout {
  size_t tick1, part0, part1, total;
};

// Workspace: tickets per group of 16 splits [B][nkv][groups], tickets per
// (row, head) [B][nkv], partials per split (at most s_max / 64 splits: four
// tiles of 16 slots each), partials per group; each part 256-byte aligned.
static AttnLayout attention_workspace(int B, int nh, int nkv, int s_max) {
  const int G = nh / nkv, maxs = s_max / (kAttnTile * kAttnWarps);
  const int maxg = (maxs + kAttnGroup - 1) / kAttnGroup;
  const size_t bg = (size_t)B * nkv;
  AttnLayout l;
  l.tick1 = align256(bg * maxg * 4);
  l.part0 = l.tick1 + align256(bg * 4);
  l.part1 = l.part0 + align256(bg * maxs * G * kPartStride * 4);
  l.total = l.part1 + bg * maxg * G * kPartStride * 4;
  return l;
}

// Splits per (row, head): one wave of resident CTAs over all rows and heads,
// at most one split per four tiles.
// The kernel attribute and the occupancy are set up once per device (the
// attribute is per device), under a lock.
static int attention_splits(int B, int nkv, int s_max, cudaError_t* err) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static int per_sm[kMaxDev] = {0}, sms[kMaxDev] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return 0;
  }
  int ctas_per_sm = 0, nsm = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!per_sm[dev]) {
      e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_decode_attention, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kAttnSmem);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas_per_sm, k_decode_attention,
                                                          kAttnThreads, kAttnSmem);
      if (e != cudaSuccess || ctas_per_sm < 1) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
        return 0;
      }
      per_sm[dev] = ctas_per_sm;
      sms[dev] = nsm;
    }
    ctas_per_sm = per_sm[dev];
    nsm = sms[dev];
  }
  const int maxs = s_max / (kAttnTile * kAttnWarps);
  const int fill = ctas_per_sm * nsm / (B * nkv);
  int splits = fill < 1 ? 1 : (fill < maxs ? fill : maxs);
  // a merge takes at most kMergeMax entries: groups of the splits included
  if (splits > kAttnGroup * kMergeMax) splits = kAttnGroup * kMergeMax;
  return splits;
}

ws_status decode_attention(const float* q, const float* k_new, const float* v_new,
                           void* k_cache, void* v_cache, const int32_t* pos, float* out_f32,
                           void* out_bf16, int B, int n_heads, int n_kv_heads, int head_dim,
                           int s_max, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream, bool pdl);

}  // namespace ws

using namespace ws;

extern "C" {

size_t ws_attention_workspace_bytes(int B, int n_heads, int n_kv_heads, int head_dim, int s_max) {
  if (B < 1 || B > kMaxBatch || n_kv_heads < 1 || n_heads % n_kv_heads || head_dim != kAttnDim ||
      s_max < kAttnTile * kAttnWarps || s_max % (kAttnTile * kAttnWarps) ||
      n_heads / n_kv_heads > kAttnMaxG)
    return 0;
  return attention_workspace(B, n_heads, n_kv_heads, s_max).total;
}

ws_status ws_decode_attention(const float* q, const float* k_new, const float* v_new,
                              void* k_cache, void* v_cache, const int32_t* pos, float* out_f32,
                              void* out_bf16, int B, int n_heads, int n_kv_heads, int head_dim,
                              int s_max, void* workspace, size_t workspace_bytes,
                              ws_stream_t stream) {
  return ws::decode_attention(q, k_new, v_new, k_cache, v_cache, pos, out_f32, out_bf16, B,
                              n_heads, n_kv_heads, head_dim, s_max, workspace, workspace_bytes,
                              (cudaStream_t)stream, false);
}

}  // extern "C"

// The entry point's body; pdl: launched as a programmatic dependent of the
// previous kernel on the stream (inside a chain).
ws_status ws::decode_attention(const float* q, const float* k_new, const float* v_new,
                               void* k_cache, void* v_cache, const int32_t* pos, float* out_f32,
                               void* out_bf16, int B, int n_heads, int n_kv_heads, int head_dim,
                               int s_max, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream, bool pdl) {
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !pos || (!out_f32 && !out_bf16) ||
      !workspace) {
    set_error("null argument");
    return WS_ERR_ARG;
  }
  if (B < 1 || B > kMaxBatch || n_kv_heads < 1 || n_heads % n_kv_heads || head_dim != kAttnDim ||
      s_max < kAttnTile * kAttnWarps || s_max % (kAttnTile * kAttnWarps)) {
    set_error("decode attention: B 1..%d, head_dim %d, n_heads a multiple of n_kv_heads, "
              "s_max a multiple of %d", kMaxBatch, kAttnDim, kAttnTile * kAttnWarps);
    return WS_ERR_SHAPE;
  }
  const int G = n_heads / n_kv_heads;
  if (G < 1 || G > kAttnMaxG) {
    set_error("decode attention: %d query heads per key-value head (1 to %d)", G, kAttnMaxG);
    return WS_ERR_SHAPE;
  }
  if (((uintptr_t)k_cache & 15u) || ((uintptr_t)v_cache & 15u) || ((uintptr_t)q & 7u) ||
      ((uintptr_t)k_new & 15u) || ((uintptr_t)v_new & 15u)) {
    set_error("decode attention: caches and new rows 16-byte aligned, q 8-byte aligned");
    return WS_ERR_ALIGN;
  }
  const AttnLayout lay = attention_workspace(B, n_heads, n_kv_heads, s_max);
  if (workspace_bytes < lay.total) {
    set_error("workspace too small: need %zu bytes, got %zu", lay.total, workspace_bytes);
    return WS_ERR_ARG;
  }
  cudaError_t e = cudaSuccess;
  const int splits = attention_splits(B, n_kv_heads, s_max, &e);
  if (!splits) {
    set_error("decode attention setup failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  AttnParams a;
  memset(&a, 0, sizeof a);
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = static_cast<uint16_t*>(k_cache);
  a.v_cache = static_cast<uint16_t*>(v_cache);
  a.pos = pos;
  a.out_f32 = out_f32;
  a.out_bf16 = static_cast<uint16_t*>(out_bf16);
  a.nh = n_heads;
  a.nkv = n_kv_heads;
  a.S = s_max;
  a.G = G;
  a.scale = 1.0f / sqrtf((float)kAttnDim);
  char* w = static_cast<char*>(workspace);
  a.tick0 = reinterpret_cast<unsigned*>(w);
  a.tick1 = reinterpret_cast<unsigned*>(w + lay.tick1);
  a.part0 = reinterpret_cast<float*>(w + lay.part0);
  a.part1 = reinterpret_cast<float*>(w + lay.part1);
  a.err = device_error_ptr();
  a.timeout_ns = tuning().timeout_ns;
  // the tickets are zero on entry (a zero-filled workspace; the last arrival
  // at every ticket resets it, rows with a bad position take none)
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(splits, n_kv_heads, B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, k_decode_attention, a);
  if (e != cudaSuccess) {
    set_error("launch failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}
