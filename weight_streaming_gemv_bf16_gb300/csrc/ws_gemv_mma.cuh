// ws_gemv_mma.cuh -- the streaming GEMV on warp-level tensor cores, for the
// decode-chain forms at batch tiles 8 and 16 (device code).
//
// y[b][m] = sum_k W[m][k] * x[b][k] with bf16 W and x and fp32 accumulation
// ("One Token, Kernel by Kernel: A Decode Step on a Laptop GPU", Step 1):
// the same op as k_stream_gemv, for batches where the CUDA-core product is
// bound by instruction issue and by shared-memory reads of the activations
// (each 16-byte weight chunk meets B activation chunks) instead of by HBM.
// Every warp is still an independent pipeline over its own ring of weight
// pieces (1-D bulk copies, mbarriers, pieces issued before the dependency
// wait); a task is 16 rows, and each 16-column step of a piece is one
// m16n8k16 bf16 MMA per matrix and per 8 batch rows, its operands read with
// ldmatrix.  Piece rows and activation rows sit an odd number of 16-byte
// units apart, so the eight rows of an 8x8 ldmatrix tile fall in eight
// different bank groups.  Products of bf16 values are exact in fp32 as on the
// CUDA-core path; the MMA sums them in its own order, within the fp32
// tolerance of the oracle.
#pragma once

#include "ws_gemv_kernel.cuh"

namespace ws {

constexpr int kMmaRows = 16;  // rows per warp task: one m16 tile

// RMSNorm over the whole K (one round: NR 8-column chunks per thread), then
// the split's columns [c0, c0 + nch) of every batch row normalised, rounded
// once to bf16 and stored as [BT][xrs chunks]; rows B..BT-1 are zero.
template <int BT, int NR>
__device__ void stage_rms_mma(const GemvParams& p, float* stats, float* red, uint16_t* xs, int c0,
                              int nch, int xrs, int tid, const uint4 (&g)[NR]) {
  const int kch = p.K >> 3, n = p.B * kch;
  float* tot = red + kWarps * BT;
  float v[NR][8];
  float s[BT];
  int rb[NR], rc[NR];
  chunk_coords<NR, BT>(tid, kThreads, kch, rb, rc);
#pragma unroll
  for (int b = 0; b < BT; ++b) s[b] = 0.f;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int o = tid + i * kThreads;
    if (o < n) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x)) + 2 * o;
      const float4 lo4 = __ldcg(src), hi4 = __ldcg(src + 1);
      v[i][0] = lo4.x; v[i][1] = lo4.y; v[i][2] = lo4.z; v[i][3] = lo4.w;
      v[i][4] = hi4.x; v[i][5] = hi4.y; v[i][6] = hi4.z; v[i][7] = hi4.w;
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
    const int c = rc[i] - c0;
    if (o < n && c >= 0 && c < nch) {
      const float r = stats[2 * rb[i]];
      const float gf[8] = {bf16lo(g[i].x), bf16hi(g[i].x), bf16lo(g[i].y), bf16hi(g[i].y),
                           bf16lo(g[i].z), bf16hi(g[i].z), bf16lo(g[i].w), bf16hi(g[i].w)};
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = pack_bf16x2(v[i][2 * e] * r * gf[2 * e], v[i][2 * e + 1] * r * gf[2 * e + 1]);
      xs4[rb[i] * xrs + c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  for (int o = tid; o < (BT - p.B) * nch; o += kThreads)
    xs4[(p.B + o / nch) * xrs + o % nch] = make_uint4(0u, 0u, 0u, 0u);
}

// bf16 activations without a prologue: columns [c0, c0 + nch) of every batch
// row into [BT][xrs chunks], rows B..BT-1 zero; each thread's loads (up to
// eight chunks) in flight before its stores.
template <int BT>
__device__ void stage_copy_mma(const GemvParams& p, uint16_t* xs, int c0, int nch, int xrs,
                               int tid) {
  const int n = BT * nch;
  uint4* xs4 = reinterpret_cast<uint4*>(xs);
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x));
  const int rs = p.K >> 3;
  for (int base = tid; base < n; base += 8 * kThreads) {
    uint4 t[8];
    int b[8], c[8];
    chunk_coords<8, BT>(base, kThreads, nch, b, c);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      t[i] = (b[i] < BT && b[i] < p.B) ? __ldcg(src + (size_t)b[i] * rs + c0 + c[i])
                                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (b[i] < BT) xs4[b[i] * xrs + c[i]] = t[i];
  }
}

// One piece of a task: kMmaRows rows x len columns of every matrix, each row
// a 1-D bulk copy to its prow-strided place in the ring slot (rows past the
// segment's end are left as they are; their results are never stored).
template <int NMAT, bool Q4 = false>
__device__ __forceinline__ void issue_piece_mma(const GemvParams& p, int rg, int j, int slot, int k0,
                                                uint8_t* ring, uint64_t* full, uint64_t pol) {
  const Sched& sc = p.sc;
  if constexpr (Q4) {
    // 4-bit rows: the piece's whole super-groups of each row
    int seg, rgl;
    decode_rg(p, rg, seg, rgl);
    const Seg& S = p.seg[seg];
    const int row0 = rgl * kMmaRows;
    const int rows = min(kMmaRows, S.M - row0);
    const int c0 = k0 + j * sc.PC;
    const int len = min(sc.PC, sc.KS - j * sc.PC);
    const int rb = q4_prefix(p.K), src0 = q4_prefix(c0), nb = q4_prefix(c0 + len) - src0;
    uint8_t* dst = ring + (size_t)slot * sc.piece_bytes;
    mbar_arrive_expect_tx(&full[slot], (uint32_t)(NMAT * rows * nb));
#pragma unroll
    for (int mat = 0; mat < NMAT; ++mat) {
      const uint8_t* W = reinterpret_cast<const uint8_t*>(mat == 0 ? S.W0 : S.W1);
      for (int r = 0; r < rows; ++r)
        bulk_copy_g2s(dst + (size_t)(mat * kMmaRows + r) * sc.prow,
                      W + (size_t)(row0 + r) * rb + src0, (uint32_t)nb, &full[slot], pol);
    }
    return;
  }
  int seg, rgl;
  decode_rg(p, rg, seg, rgl);
  const Seg& S = p.seg[seg];
  const int row0 = rgl * kMmaRows;
  const int rows = min(kMmaRows, S.M - row0);
  const int c0 = k0 + j * sc.PC;
  const int len = min(sc.PC, sc.KS - j * sc.PC);
  uint8_t* dst = ring + (size_t)slot * sc.piece_bytes;
  const int K = p.K;
  mbar_arrive_expect_tx(&full[slot], (uint32_t)(NMAT * rows * len * 2));
#pragma unroll
  for (int mat = 0; mat < NMAT; ++mat) {
    const uint16_t* W = mat == 0 ? S.W0 : S.W1;
    for (int r = 0; r < rows; ++r)
      bulk_copy_g2s(dst + (size_t)(mat * kMmaRows + r) * sc.prow, W + (size_t)(row0 + r) * K + c0,
                    (uint32_t)(len * 2), &full[slot], pol);
  }
}

// d[mat][g8] += W_mat[16 rows][len] x x[8 g8 .. 8 g8 + 7][len]^T over one
// piece (st: its shared address; xa: the activations of its first column).
template <int BT, int NMAT>
__device__ __forceinline__ void mma_piece(float (&d)[NMAT][BT / 8][4], uint32_t st, uint32_t xa,
                                          int len, int prow, int xrow, int lane) {
  constexpr int NG = BT / 8;
  // A tile 16 x 16: lane l addresses row (l % 8) + 8 ((l / 8) % 2), columns
  // 8 (l / 16) .. + 7, so that the four 8x8 matrices come out as a0..a3
  const uint32_t a0 = st + (uint32_t)(((lane & 7) + ((lane >> 3) & 1) * 8) * prow) +
                      (uint32_t)((lane >> 4) * 16);
  // B tile 16 x 8 per batch group: lane l addresses batch row (l % 8) (+ 8
  // for l >= 16 with two groups), columns 8 ((l / 8) % 2) .. + 7
  const uint32_t b0 = xa + (uint32_t)(((lane & 7) + (NG == 2 ? (lane >> 4) * 8 : 0)) * xrow) +
                      (uint32_t)(((lane >> 3) & 1) * 16);
#pragma unroll 2
  for (int kk = 0; kk < len; kk += 16) {
    uint32_t b[NG][2];
    if constexpr (NG == 2)
      ldsm_x4(b0 + kk * 2, b[0][0], b[0][1], b[1][0], b[1][1]);
    else
      ldsm_x2(b0 + kk * 2, b[0][0], b[0][1]);
#pragma unroll
    for (int mat = 0; mat < NMAT; ++mat) {
      uint32_t f0, f1, f2, f3;
      ldsm_x4(a0 + (uint32_t)(mat * kMmaRows * prow) + kk * 2, f0, f1, f2, f3);
#pragma unroll
      for (int g8 = 0; g8 < NG; ++g8) mma_bf16_16816(d[mat][g8], f0, f1, f2, f3, b[g8][0], b[g8][1]);
    }
  }
}

// Two 4-bit codes of a word (bits 4j.. and 16 + 4j..) as a bf16 pair 128 + q
// (0x4300 is 128 in bf16; the nibble lands in the low mantissa bits).
__device__ __forceinline__ uint32_t q4_mma_pair(uint32_t w, int j) {
  return ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
}

// 4-bit rows (16 of each matrix, prow bytes apart in the ring) against the
// staged activations over one piece, group by group.  Lane (g, t) builds the
// A fragments of rows g and g + 8 from their code words (pair t of a word is
// weights 2t and 2t + 1 of its eight, as 128 + q in bf16), one m16n8k16 MMA
// per 16 columns, each into its own accumulator (the eight MMAs of a group
// are independent: the MMA's latency, not its rate, is what a chain would
// pay), summed per group, then
// d += s * D + (z - 136 s) * X with the group's (s, z) per row and X the
// batch column's sum of the group's 128 activations: the sum of
// (s (q - 8) + z) x.  Batch rows past the staged ones read a zero row.
template <int NMAT>
__device__ __forceinline__ void mma_piece_q4(float (&d)[NMAT][1][4], const uint8_t* st,
                                             uint32_t xa, uint32_t xzero, const float* xsg,
                                             int len, int prow, int xrow, int nxg, int nb_rows,
                                             int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int ngr = len >> 7;
  const int br = lane & 7;
  const bool bz = br >= nb_rows;
  const uint32_t bbase = bz ? xzero : xa + (uint32_t)(br * xrow + (lane >> 3) * 16);
#pragma unroll 2
  for (int gg = 0; gg < ngr; ++gg) {
    const int u = gg >> 2, gi = gg & 3;
    const int gu = min(4, ngr - 4 * u);
    const int coff = u * kQ4SuperBytes + gi * 64;
    const int soff = u * kQ4SuperBytes + gu * 64 + gi * 4;
    float dg[NMAT][8][4];
    uint32_t sz0[NMAT], sz1[NMAT];
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int i = 0; i < 4; ++i) dg[m][kk][i] = 0.f;
      sz0[m] = *reinterpret_cast<const uint32_t*>(st + (size_t)(m * kMmaRows + g) * prow + soff);
      sz1[m] = *reinterpret_cast<const uint32_t*>(st + (size_t)(m * kMmaRows + g + 8) * prow + soff);
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {  // 32 columns: two MMA steps
      uint32_t b0, b1, b2, b3;
      ldsm_x4(bz ? bbase : bbase + (uint32_t)((gg * 128 + h * 32) * 2), b0, b1, b2, b3);
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        const uint4 w0 = *reinterpret_cast<const uint4*>(
            st + (size_t)(m * kMmaRows + g) * prow + coff + h * 16);
        const uint4 w1 = *reinterpret_cast<const uint4*>(
            st + (size_t)(m * kMmaRows + g + 8) * prow + coff + h * 16);
        mma_bf16_16816(dg[m][2 * h], q4_mma_pair(w0.x, t), q4_mma_pair(w1.x, t),
                       q4_mma_pair(w0.y, t), q4_mma_pair(w1.y, t), b0, b1);
        mma_bf16_16816(dg[m][2 * h + 1], q4_mma_pair(w0.z, t), q4_mma_pair(w1.z, t),
                       q4_mma_pair(w0.w, t), q4_mma_pair(w1.w, t), b2, b3);
      }
    }
    const float x0 = xsg[(2 * t) * nxg + gg], x1 = xsg[(2 * t + 1) * nxg + gg];
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      const float s0 = bf16lo(sz0[m]), z0 = fmaf(-136.f, s0, bf16hi(sz0[m]));
      const float s1 = bf16lo(sz1[m]), z1 = fmaf(-136.f, s1, bf16hi(sz1[m]));
      float D[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        D[i] = ((dg[m][0][i] + dg[m][1][i]) + (dg[m][2][i] + dg[m][3][i])) +
               ((dg[m][4][i] + dg[m][5][i]) + (dg[m][6][i] + dg[m][7][i]));
      d[m][0][0] = fmaf(z0, x0, fmaf(s0, D[0], d[m][0][0]));
      d[m][0][1] = fmaf(z0, x1, fmaf(s0, D[1], d[m][0][1]));
      d[m][0][2] = fmaf(z1, x0, fmaf(s1, D[2], d[m][0][2]));
      d[m][0][3] = fmaf(z1, x1, fmaf(s1, D[3], d[m][0][3]));
    }
  }
}

// The tensor-core kernel for the chain forms F at batch tile BT (8 or 16):
// the same ring, waits, staging order, epilogues and split-K protocol as
// k_stream_gemv; 16-row tasks and MMA fragments in place of the lane dot
// products and the warp reduction.
template <int BT, int NMAT, int F, bool Q4 = false>
__global__ void __launch_bounds__(kThreads, 1) k_stream_gemv_mma(const __grid_constant__ GemvParams p) {
  static_assert(BT == 8 || BT == 16, "tensor-core kernel: batch tile 8 or 16");
  static_assert(!Q4 || BT == 8, "4-bit rows: one batch group (B <= 4 staged)");
  constexpr int NG = BT / 8;
  // streaming warps: all of them for 4-bit rows (small pieces), else kMmaWarps
  constexpr int NWS = Q4 ? kWarps : kMmaWarps;
  constexpr int SBT = Q4 ? 4 : BT;  // activation rows staged
  using FT = FormTraits<F>;
  constexpr int EPI = FT::epi;
  static_assert(EPI >= 0, "tensor-core kernel: chain forms only");
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
  // pieces of this warp: row groups rg0 + warp + t * kMmaWarps
  const int npw =
      (warp < NWS && rg1 - rg0 > warp) ? (rg1 - rg0 - warp + NWS - 1) / NWS * NP : 0;
  const int rgw = rg0 + warp;  // this warp's first row group

  int iq = 0, iti = 0, ij = 0, islot = 0;
  uint64_t pol = 0;
  if (lane == 0) {
    for (int s = 0; s < NSW; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    pol = p.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
    while (iq < NSW && iq < npw) {  // the whole ring before the dependency wait
      issue_piece_mma<NMAT, Q4>(p, rgw + iti * NWS, ij, islot, k0, ring, full, pol);
      ++iq;
      if (++ij == NP) { ij = 0; ++iti; }
      if (++islot == NSW) islot = 0;
    }
  }
  constexpr int NR = form_round_chunks(SBT);
  uint4 gpre[NR];
  if constexpr (FT::rms1) gamma_preload<NR, SBT>(p, tid, gpre);
  pdl_launch_dependents();
  pdl_wait();
  if (stamp && tid == 0) stamp[1] = global_ns();

  // the residual input of this CTA's rows (unsplit K), read while the
  // activations stage
  float* res_s = EPI == EPI_RESID && sc.off_res ? reinterpret_cast<float*>(smem + sc.off_res)
                                                : nullptr;
  const int res_row0 = rg0 * kMmaRows;
  if (res_s) {
    const float* src = p.res_in ? p.res_in : static_cast<const float*>(p.seg[0].out);
    const int nr = min(rg1 * kMmaRows, p.seg[0].M) - res_row0;
#pragma unroll 1
    for (int i = tid; i < p.B * nr; i += kThreads) {
      const int b = i / nr, r = i - (i / nr) * nr;
      res_s[b * sc.res_rows + r] = __ldcg(src + (size_t)b * p.seg[0].M + res_row0 + r);
    }
  }
  if constexpr (FT::rms1)
    stage_rms_mma<SBT, NR>(p, stats, red, xs, k0 >> 3, sc.KS >> 3, sc.xrs, tid, gpre);
  else
    stage_copy_mma<SBT>(p, xs, k0 >> 3, sc.KS >> 3, sc.xrs, tid);
  __syncthreads();
  // 4-bit rows: per batch row (8, rows past the staged 4 zero) the sum of
  // each 128-column group of the staged activations, and a zero row for the
  // padding rows of the activation fragments
  float* xsg = Q4 ? reinterpret_cast<float*>(smem + sc.off_xsum) : nullptr;
  const int nxg = sc.KS >> 7;
  if constexpr (Q4) {
    for (int o = tid; o < 8 * nxg; o += kThreads) {
      const int b = o / nxg, c = o - b * nxg;
      float sum = 0.f;
      if (b < SBT) {
        const uint4* src = reinterpret_cast<const uint4*>(xs) + (size_t)b * sc.xrs + 16 * c;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const uint4 v = src[i];
          sum += bf16lo(v.x) + bf16hi(v.x) + bf16lo(v.y) + bf16hi(v.y);
          sum += bf16lo(v.z) + bf16hi(v.z) + bf16lo(v.w) + bf16hi(v.w);
        }
      }
      xsg[o] = sum;
    }
    if (tid < 4) reinterpret_cast<uint32_t*>(smem + sc.off_xzero)[tid] = 0u;
    __syncthreads();
  }
  if (stamp && tid == 0) stamp[2] = global_ns();

  const int xrow = sc.xrs * 16;  // bytes between activation rows
  const uint32_t xs_a = smem_addr(xs);
  const uint32_t ring_a = smem_addr(ring);
  const int g = lane >> 2, t = lane & 3;  // fragment row group and column pair
  float best_v[NG * 2];
  int best_i[NG * 2];
#pragma unroll
  for (int s = 0; s < NG * 2; ++s) {
    best_v[s] = -INFINITY;
    best_i[s] = 0x7fffffff;
  }
  bool abort = false;

  float d[NMAT][NG][4];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int g8 = 0; g8 < NG; ++g8)
#pragma unroll
      for (int i = 0; i < 4; ++i) d[m][g8][i] = 0.f;

  int ti = 0, j = 0, slot = 0;
  uint32_t phase = 0;
  for (int q = 0; q < npw; ++q) {
    const int rg = rgw + ti * NWS;
    int seg, rgl;
    decode_rg(p, rg, seg, rgl);
    const int row0 = rgl * kMmaRows;
    const int rows = min(kMmaRows, p.seg[seg].M - row0);
    const int len = min(sc.PC, sc.KS - j * sc.PC);
    const bool ok = abort || mbar_wait_bounded(&full[slot], phase, p.timeout_ns);
    if (__any_sync(0xffffffffu, !ok) && !abort) {
      abort = true;
      if (lane == 0) raise_device_error(p.err, DERR_TIMEOUT);
    }
    if (!abort) {
      if constexpr (Q4)
        mma_piece_q4<NMAT>(d, ring + (size_t)slot * sc.piece_bytes,
                           xs_a + (uint32_t)(j * sc.PC * 2), smem_addr(smem + sc.off_xzero),
                           xsg + j * (sc.PC >> 7), len, sc.prow, xrow, nxg, SBT, lane);
      else
        mma_piece<BT, NMAT>(d, ring_a + (uint32_t)(slot * sc.piece_bytes),
                            xs_a + (uint32_t)(j * sc.PC * 2), len, sc.prow, xrow, lane);
    }
    // ldmatrix has returned every lane's values (they fed the MMAs above):
    // refill the slot
    __syncwarp();
    if (lane == 0 && !abort && iq < npw) {
      issue_piece_mma<NMAT, Q4>(p, rgw + iti * NWS, ij, islot, k0, ring, full, pol);
      ++iq;
      if (++ij == NP) { ij = 0; ++iti; }
      if (++islot == NSW) islot = 0;
    }

    if (j == NP - 1) {
      // task complete: lane holds rows g, g + 8 and batch columns
      // 8 g8 + 2 t, + 1 of each matrix's 16 x BT block
      const int rowg = p.seg[seg].row_base + row0;
      if (sc.S == 1) {
#pragma unroll
        for (int g8 = 0; g8 < NG; ++g8)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = g + 8 * (i >> 1), b = 8 * g8 + 2 * t + (i & 1);
            if (r < rows && b < p.B)
              apply_epilogue<EPI>(p, seg, row0 + r, b, d[0][g8][i], d[NMAT - 1][g8][i],
                                  best_v[g8 * 2 + (i & 1)], best_i[g8 * 2 + (i & 1)], res_s,
                                  res_row0, sc.res_rows);
          }
      } else {
        // split-K: this split's partials; the last split of the row group
        // adds all splits in split order and runs the epilogue
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
          for (int g8 = 0; g8 < NG; ++g8)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = g + 8 * (i >> 1), b = 8 * g8 + 2 * t + (i & 1);
              if (r < rows && b < p.B)
                p.part[((size_t)(ks * NMAT + m) * p.B + b) * p.M_total + rowg + r] = d[m][g8][i];
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
          constexpr int U = 8;
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
                                    nullptr, 0, 0);
              }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int g8 = 0; g8 < NG; ++g8)
#pragma unroll
          for (int i = 0; i < 4; ++i) d[m][g8][i] = 0.f;
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

  if (stamp) {
    __syncthreads();
    if (tid == 0) stamp[3] = global_ns();
  }

  if constexpr (EPI == EPI_ARGMAX) {
    // per batch column: the best over the lanes sharing t (rows g), then
    // thread b combines the warps, then the last CTA (ticket) all CTAs
#pragma unroll
    for (int s = 0; s < NG * 2; ++s) {
      float v = best_v[s];
      int i = best_i[s];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (arg_better(ov, oi, v, i)) {
          v = ov;
          i = oi;
        }
      }
      if (lane < 4) {  // g = 0: column 8 (s / 2) + 2 t + s % 2
        const int b = 8 * (s >> 1) + 2 * lane + (s & 1);
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

GemvKernel pick_kernel_mma(int BT, int nmat, int F);
GemvKernel pick_kernel_q4mma(int nmat, int F);

}  // namespace ws
