// ws_persist.cu -- the persistent chain kernel: a whole decode step (every op
// of the chain) in one cooperative launch, one CTA per SM.
//
// The ops of a chain depend on each other only through their small
// activation vectors; their weights -- all but ~0.01% of the bytes -- do not
// depend on anything.  So each warp streams its weight pieces of every op, in
// order, through its own byte ring in shared memory, and its copy cursor runs
// ahead across op boundaries.  Between ops the CTAs meet at a grid barrier
// (the previous op's outputs are complete), normalise the next activation
// vector into shared memory and compute on pieces that have usually already
// landed.  HBM keeps streaming through every barrier and prologue as long as
// the rings have room, which a chain of separate launches cannot do: there
// each op boundary drains the memory pipeline ("One Token, Kernel by Kernel:
// A Decode Step on a Laptop GPU", Step 3, where kernel gaps are counted
// against the bandwidth floor).
//
// Work: an op's units (row group of RT rows x one of S K-splits) are dealt
// round-robin over all warps of the grid, so every warp gets the same number
// of units to within one; long rows are split in K so the per-warp load
// evens out, the splits' partial sums being added by the last split to finish
// (atomic ticket), in split order.  Pieces (RT rows x up to PC columns) are
// packed back to back in the warp's byte ring; a piece's place follows from
// the sizes of the pieces before it, so the copy cursor and the consumer
// compute it the same way without sharing any state.  Eight mbarriers per
// warp track up to eight pieces in flight.
//
// Epilogues and numerics are those of the standalone kernel.  All waits are
// bounded: a grid barrier or a copy that does not arrive within timeout_ns
// sets the device error flag and the kernel runs to its end without waiting.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "wsgemv.h"
#include "ws_common.cuh"
#include "ws_gemv_kernel.cuh"

namespace ws {

constexpr int kBars = 8;  // mbarriers (pieces in flight) per warp

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Units of op sc for global warp gw: u = gw, gw + GW, ...
__device__ __forceinline__ int warp_units(const Sched& sc, int gw, int GW) {
  const int U = sc.RG * sc.S;
  return U > gw ? (U - gw + GW - 1) / GW : 0;
}

// Bytes a piece takes in the ring: RT rows reserved, `len` columns each.
__device__ __forceinline__ int piece_size(int nmat, int RT, int len) { return nmat * RT * len * 2; }

// A position in a warp's ring: the linear byte count since the start and its
// offset within the ring (kept side by side, so placing costs no division).
struct RingPos {
  long long lin;
  int off;
};

// Place a piece of `sz` bytes at `pos`: returns its offset in the ring and
// advances `pos` past it (a piece never wraps; the tail is skipped instead).
__device__ __forceinline__ int ring_place(RingPos& pos, int sz, int R) {
  if (pos.off + sz > R) {
    pos.lin += R - pos.off;
    pos.off = 0;
  }
  const int at = pos.off;
  pos.off += sz;
  pos.lin += sz;
  return at;
}

// The copy cursor of one warp (advanced by lane 0 only): the next piece to
// stream, walking this warp's pieces of every op in order, with the current
// op's shape and weight pointers cached in registers.
struct IssueCursor {
  int f;          // op
  int q;          // piece within the op for this warp
  int npw;        // pieces of this warp in op f
  int ui;         // unit index within this warp's units of op f
  int j;          // piece within the unit
  int n;          // pieces issued so far
  RingPos pos;    // ring position of the next piece
  int nseg, nmat, RT, PC, NP, K, KS, S;
  int M[kMaxSeg], rgb[kMaxSeg];
  const uint16_t* W0[kMaxSeg];
  const uint16_t* W1[kMaxSeg];
};

__device__ __forceinline__ void cursor_seek(const PersistParams& pp, IssueCursor& c, int gw,
                                            int GW) {
  while (c.f < pp.nops && c.q >= c.npw) {
    ++c.f;
    c.q = 0;
    c.ui = 0;
    c.j = 0;
    c.npw = 0;
    if (c.f < pp.nops) {
      const GemvParams& P = pp.ops[c.f];
      c.NP = P.sc.NP;
      c.npw = warp_units(P.sc, gw, GW) * c.NP;
      c.nseg = P.nseg;
      c.nmat = P.nmat;
      c.RT = P.sc.RT;
      c.PC = P.sc.PC;
      c.K = P.K;
      c.KS = P.sc.KS;
      c.S = P.sc.S;
#pragma unroll
      for (int s = 0; s < kMaxSeg; ++s) {
        c.M[s] = P.seg[s].M;
        c.rgb[s] = P.seg[s].rg_begin;
        c.W0[s] = P.seg[s].W0;
        c.W1[s] = P.seg[s].W1;
      }
    }
  }
}

// Bytes of the cursor's next piece.
__device__ __forceinline__ int cursor_piece_bytes(const IssueCursor& c) {
  const int len = min(c.PC, c.KS - c.j * c.PC);
  return piece_size(c.nmat, c.RT, len);
}

__device__ __forceinline__ void issue_next(const PersistParams& pp, IssueCursor& c, int gw, int GW,
                                           uint8_t* ring, uint64_t* bars, uint64_t pol) {
  const int u = gw + c.ui * GW;
  const int rg = u / c.S;
  const int ks = u - rg * c.S;
  const bool s1 = c.nseg > 1 && rg >= c.rgb[1];
  const bool s2 = c.nseg > 2 && rg >= c.rgb[2];
  const int rgb = s2 ? c.rgb[2] : (s1 ? c.rgb[1] : c.rgb[0]);
  const int Mseg = s2 ? c.M[2] : (s1 ? c.M[1] : c.M[0]);
  const uint16_t* W0 = s2 ? c.W0[2] : (s1 ? c.W0[1] : c.W0[0]);
  const uint16_t* W1 = s2 ? c.W1[2] : (s1 ? c.W1[1] : c.W1[0]);
  const int RT = c.RT, K = c.K;
  const int row0 = (rg - rgb) * RT;
  const int rows = min(RT, Mseg - row0);
  const int c0 = ks * c.KS + c.j * c.PC;
  const int len = min(c.PC, c.KS - c.j * c.PC);
  const int sz = piece_size(c.nmat, RT, len);
  uint8_t* dst = ring + ring_place(c.pos, sz, pp.slot_bytes);
  uint64_t* bar = &bars[c.n & (kBars - 1)];
  mbar_arrive_expect_tx(bar, (uint32_t)(c.nmat * rows * len * 2));
  for (int mat = 0; mat < c.nmat; ++mat) {
    const uint16_t* W = mat == 0 ? W0 : W1;
    if (len == K) {
      bulk_copy_g2s(dst + (size_t)mat * RT * len * 2, W + (size_t)row0 * K,
                    (uint32_t)(rows * K * 2), bar, pol);
    } else {
      for (int r = 0; r < rows; ++r)
        bulk_copy_g2s(dst + ((size_t)mat * RT + r) * len * 2, W + (size_t)(row0 + r) * K + c0,
                      (uint32_t)(len * 2), bar, pol);
    }
  }
  ++c.n;
  ++c.q;
  if (++c.j == c.NP) {
    c.j = 0;
    ++c.ui;
  }
  cursor_seek(pp, c, gw, GW);
}

// The consumer's view of the ring, the same in every lane.
struct ConsumeState {
  int n;          // pieces consumed
  RingPos pos;    // ring position of the next piece
  bool abort;
};

// Issue pieces while a barrier is free and the next piece fits behind the
// consumer (lane 0 only).
__device__ __forceinline__ void refill(const PersistParams& pp, IssueCursor& ic,
                                       const ConsumeState& cs, int gw, int GW, uint8_t* ring,
                                       uint64_t* bars, uint64_t pol) {
  const int R = pp.slot_bytes;
  while (ic.f < pp.nops && ic.n - cs.n < kBars) {
    const int sz = cursor_piece_bytes(ic);
    RingPos end = ic.pos;
    ring_place(end, sz, R);
    if (end.lin - cs.pos.lin > R) break;
    issue_next(pp, ic, gw, GW, ring, bars, pol);
  }
}

// Asynchronous 16-byte copies of an op descriptor into shared memory (the
// next op's, fetched while the current op computes).
__device__ __forceinline__ void prefetch_descriptor(const GemvParams* src, GemvParams* dst,
                                                    int tid) {
  constexpr int n16 = (int)(sizeof(GemvParams) / 16);
  if (tid < n16) {
    const char* s = reinterpret_cast<const char*>(src) + 16 * tid;
    const uint32_t d = smem_addr(reinterpret_cast<char*>(dst) + 16 * tid);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(s) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void wait_descriptor() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// One unit (RT rows x one K split) of op P: consume its NP pieces (refilling
// the ring as they free up), reduce over lanes, then run the epilogue -- or,
// for a split, publish the partial sums and let the last split finish.
template <int BT, int NMAT, int RT>
__device__ __forceinline__ void run_unit(const PersistParams& pp, const GemvParams& P, int u,
                                         uint8_t* ring, uint64_t* bars, const uint4* xs4,
                                         ConsumeState& cs, IssueCursor& ic, uint64_t pol,
                                         float& best_v, int& best_i, int gw, int GW, int lane,
                                         unsigned long long* land_stamp) {
  const int S = P.sc.S;
  const int rg = u / S;
  const int ks = u - rg * S;
  int seg, rgl;
  decode_rg(P, rg, seg, rgl);
  const int row0 = rgl * RT;
  const int rows = min(RT, P.seg[seg].M - row0);
  const int NP = P.sc.NP, PC = P.sc.PC, KS = P.sc.KS, nchx = P.K >> 3;
  const int R = pp.slot_bytes;
  float acc[NMAT][RT][BT];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[m][r][b] = 0.f;

  for (int j = 0; j < NP; ++j) {
    const int len = min(PC, KS - j * PC);
    const int ncp = len >> 3;
    const int off = ring_place(cs.pos, piece_size(NMAT, RT, len), R);
    const bool ok = cs.abort || mbar_wait_bounded(&bars[cs.n & (kBars - 1)],
                                                  (uint32_t)((cs.n / kBars) & 1), pp.timeout_ns);
    if (land_stamp && j == 0 && lane == 0) *land_stamp = global_ns();
    if (__any_sync(0xffffffffu, !ok) && !cs.abort) {
      cs.abort = true;
      if (lane == 0) raise_device_error(pp.err, DERR_TIMEOUT);
    }
    const uint4* st = reinterpret_cast<const uint4*>(ring + off);
    const int xoff = (ks * KS + j * PC) >> 3;
#pragma unroll 2
    for (int c = lane; c < ncp; c += 32) {
      float wf[NMAT][RT][8];
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint4 w = r < rows ? st[(size_t)(m * RT + r) * ncp + c] : make_uint4(0, 0, 0, 0);
          wf[m][r][0] = bf16lo(w.x); wf[m][r][1] = bf16hi(w.x);
          wf[m][r][2] = bf16lo(w.y); wf[m][r][3] = bf16hi(w.y);
          wf[m][r][4] = bf16lo(w.z); wf[m][r][5] = bf16hi(w.z);
          wf[m][r][6] = bf16lo(w.w); wf[m][r][7] = bf16hi(w.w);
        }
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        const uint4 xv = xs4[(size_t)b * nchx + xoff + c];
        const float xf[8] = {bf16lo(xv.x), bf16hi(xv.x), bf16lo(xv.y), bf16hi(xv.y),
                             bf16lo(xv.z), bf16hi(xv.z), bf16lo(xv.w), bf16hi(xv.w)};
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[m][r][b] = fmaf(wf[m][r][e], xf[e], acc[m][r][b]);
      }
    }
    // every lane's reads of this piece have returned: its bytes are free
    __syncwarp();
    ++cs.n;
    if (lane == 0 && !cs.abort) refill(pp, ic, cs, gw, GW, ring, bars, pol);
  }
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[m][r][b] = warp_sum(acc[m][r][b]);
  if (S == 1) {
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b)
        if (lane == r * BT + b && r < rows && b < P.B)
          apply_epilogue(P, seg, row0 + r, b, acc[0][r][b], acc[NMAT - 1][r][b], best_v, best_i);
    return;
  }
  const int rowg = P.seg[seg].row_base + row0;
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int b = 0; b < BT; ++b)
      if (lane == r * BT + b && r < rows && b < P.B) {
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
          P.part[((size_t)(ks * NMAT + m) * P.B + b) * P.M_total + rowg + r] = acc[m][r][b];
      }
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    const unsigned old = atomicAdd(&P.tickets[rg], 1u);
    last = old == (unsigned)(S - 1);
    if (last) atomicExch(&P.tickets[rg], 0u);
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) {
    __threadfence();
    for (int o = lane; o < rows * P.B; o += 32) {
      const int rr = o / P.B;
      const int b = o - rr * P.B;
      float v[NMAT];
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        float t = 0.f;
        for (int s = 0; s < S; ++s)
          t += __ldcg(&P.part[((size_t)(s * NMAT + m) * P.B + b) * P.M_total + rowg + rr]);
        v[m] = t;
      }
      float dv = -INFINITY;
      int di = 0x7fffffff;
      apply_epilogue(P, seg, row0 + rr, b, v[0], v[NMAT - 1], dv, di);
    }
  }
}

// Wait until every CTA has finished op f (bounded).  Thread 0 spins; all
// threads leave together.
__device__ __forceinline__ void grid_wait(const PersistParams& pp, int f, volatile int* flags,
                                          int tid) {
  if (tid == 0) {
    const unsigned* cnt = pp.bar + f;
    if (!flags[1] && ld_acquire_u32(cnt) < gridDim.x) {
      const uint64_t t0 = global_ns();
      while (ld_acquire_u32(cnt) < gridDim.x) {
        if (global_ns() - t0 > pp.timeout_ns) {
          raise_device_error(pp.err, DERR_TIMEOUT);
          flags[1] = 1;
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// CTA 0 copies an op's output ([B][M], fp32 or bf16) to its trace slot.
__device__ __forceinline__ void copy_trace(const GemvParams* op, int tid) {
  float* tr = op->trace_out;
  if (!tr || blockIdx.x != 0) return;
  const int esz = (op->epilogue == EPI_F32 || op->epilogue == EPI_RESID) ? 4 : 2;
  const int nwords = op->B * op->seg[0].M * esz / 4;
  const unsigned* src = static_cast<const unsigned*>(op->seg[0].out);
  unsigned* dst = reinterpret_cast<unsigned*>(tr);
  for (int i = tid; i < nwords; i += kThreads) dst[i] = __ldcg(src + i);
}

template <int BT>
__global__ void __launch_bounds__(kThreads, 1)
    k_chain_persistent(const __grid_constant__ PersistParams pp) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int GW = gridDim.x * kWarps;
  const int gw = blockIdx.x * kWarps + warp;
  GemvParams* Ps = reinterpret_cast<GemvParams*>(smem + pp.off_op);  // two buffers
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pp.off_bar) + warp * kBars;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + pp.off_flags);
  float* stats = reinterpret_cast<float*>(smem + pp.off_stats);
  float* red = reinterpret_cast<float*>(smem + pp.off_red);
  float* argv = reinterpret_cast<float*>(smem + pp.off_arg);
  int* argi = reinterpret_cast<int*>(argv + kWarps * 32);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + pp.off_xs);
  const uint4* xs4 = reinterpret_cast<const uint4*>(xs);
  uint8_t* ring = smem + pp.off_ring + (size_t)warp * pp.slot_bytes;

  IssueCursor ic;
  ic.f = -1;
  ic.q = 0;
  ic.npw = 0;
  ic.ui = 0;
  ic.j = 0;
  ic.n = 0;
  ic.pos.lin = 0;
  ic.pos.off = 0;
  ConsumeState cs;
  cs.n = 0;
  cs.pos.lin = 0;
  cs.pos.off = 0;
  cs.abort = false;
  uint64_t pol = 0;
  if (tid == 0) flags[1] = 0;
  if (lane == 0) {
    for (int s = 0; s < kBars; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    pol = pp.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
    cursor_seek(pp, ic, gw, GW);
    refill(pp, ic, cs, gw, GW, ring, bars, pol);
  }
  prefetch_descriptor(pp.ops, Ps, tid);

  for (int f = 0; f < pp.nops; ++f) {
    if (f > 0) {
      grid_wait(pp, f - 1, flags, tid);
      copy_trace(pp.ops + (f - 1), tid);
    }
    wait_descriptor();
    __syncthreads();
    unsigned long long* stamp =
        pp.stamps ? pp.stamps + ((size_t)blockIdx.x * pp.nops + f) * 4 : nullptr;
    if (stamp && tid == 0) stamp[0] = global_ns();
    const GemvParams& P = Ps[f & 1];
    // the next op's descriptor streams in while this op runs
    if (f + 1 < pp.nops) prefetch_descriptor(pp.ops + f + 1, &Ps[(f + 1) & 1], tid);
    // all K columns: units of every split index into them
    if (!prologue_stage_fused<BT>(P, stats, red, xs, tid)) {
      prologue_stats<BT>(P, stats, red, tid);
      stage_x<BT>(P, stats, xs, 0, P.K >> 3, tid);
    }
    __syncthreads();
    if (stamp && tid == 0) stamp[1] = global_ns();

    const int nunits = warp_units(P.sc, gw, GW);
    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    const int kind = (P.nmat - 1) * 3 + (P.sc.RT == 1 ? 0 : (P.sc.RT == 2 ? 1 : 2));
    for (int t = 0; t < nunits; ++t) {
      const int u = gw + t * GW;
      unsigned long long* land = (stamp && warp == 0 && t == 0) ? stamp + 3 : nullptr;
      switch (kind) {
        case 0: run_unit<BT, 1, 1>(pp, P, u, ring, bars, xs4, cs, ic, pol, best_v, best_i, gw, GW, lane, land); break;
        case 1: run_unit<BT, 1, 2>(pp, P, u, ring, bars, xs4, cs, ic, pol, best_v, best_i, gw, GW, lane, land); break;
        case 2: run_unit<BT, 1, 4>(pp, P, u, ring, bars, xs4, cs, ic, pol, best_v, best_i, gw, GW, lane, land); break;
        case 3: run_unit<BT, 2, 1>(pp, P, u, ring, bars, xs4, cs, ic, pol, best_v, best_i, gw, GW, lane, land); break;
        case 4: run_unit<BT, 2, 2>(pp, P, u, ring, bars, xs4, cs, ic, pol, best_v, best_i, gw, GW, lane, land); break;
        default: run_unit<BT, 2, 4>(pp, P, u, ring, bars, xs4, cs, ic, pol, best_v, best_i, gw, GW, lane, land); break;
      }
    }

    if (P.epilogue == EPI_ARGMAX) {
      const int RT = P.sc.RT;
      argv[warp * 32 + lane] = best_v;
      argi[warp * 32 + lane] = best_i;
      __syncthreads();
      if (tid < P.B) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int w = 0; w < kWarps; ++w)
          for (int r = 0; r < RT; ++r) {
            const int l = r * BT + tid;
            if (arg_better(argv[w * 32 + l], argi[w * 32 + l], bv, bi)) {
              bv = argv[w * 32 + l];
              bi = argi[w * 32 + l];
            }
          }
        P.arg_val[(size_t)blockIdx.x * P.B + tid] = bv;
        P.arg_idx[(size_t)blockIdx.x * P.B + tid] = bi;
        __threadfence();
      }
      __syncthreads();
      if (tid == 0) {
        const unsigned old = atomicAdd(P.arg_ticket, 1u);
        const int last = old == gridDim.x - 1;
        if (last) atomicExch(P.arg_ticket, 0u);
        flags[0] = last;
      }
      __syncthreads();
      if (flags[0] && tid < P.B) {
        __threadfence();
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int c = 0; c < (int)gridDim.x; ++c) {
          const float v = __ldcg(&P.arg_val[(size_t)c * P.B + tid]);
          const int ix = __ldcg(&P.arg_idx[(size_t)c * P.B + tid]);
          if (arg_better(v, ix, bv, bi)) {
            bv = v;
            bi = ix;
          }
        }
        P.argmax_idx[tid] = bi;
      }
    }
    // this CTA is done with op f: its outputs are written
    __threadfence();
    __syncthreads();
    if (stamp && tid == 0) stamp[2] = global_ns();
    if (tid == 0) atomicAdd(pp.bar + f, 1u);
  }
  if (pp.nops > 0 && pp.ops[pp.nops - 1].trace_out) {
    grid_wait(pp, pp.nops - 1, flags, tid);
    copy_trace(pp.ops + (pp.nops - 1), tid);
  }

  if (cs.abort && lane == 0) {
    // a wait ran out: let the copies still in flight land before exit
    for (int q = cs.n; q < ic.n; ++q)
      mbar_wait_bounded(&bars[q & (kBars - 1)], (uint32_t)((q / kBars) & 1), pp.timeout_ns);
  }
  // the last CTA out resets the barrier counters for the next launch
  __syncthreads();
  if (tid == 0) {
    const unsigned old = atomicAdd(pp.bar + pp.nops, 1u);
    if (old == gridDim.x - 1)
      for (int i = 0; i <= pp.nops; ++i) atomicExch(pp.bar + i, 0u);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static int batch_template_p(int B) { return B <= 1 ? 1 : (B <= 2 ? 2 : (B <= 4 ? 4 : 0)); }
static int align_up_p(int v, int a) { return (v + a - 1) / a * a; }
static constexpr int kSmemMaxP = 227 * 1024;

// Shared-memory layout of the persistent kernel for batch B and the largest
// K of the chain; the rest of shared memory becomes the warps' byte rings.
static bool layout_persistent(PersistParams& pp, int B, int kmax, char* why, size_t why_len) {
  pp.BT = batch_template_p(B);
  if (!pp.BT) {
    snprintf(why, why_len, "the persistent chain supports batch <= 4");
    return false;
  }
  int off = 0;
  pp.off_op = off;
  off += 2 * align_up_p((int)sizeof(GemvParams), 128);
  pp.off_bar = off;
  off += kWarps * kBars * 8;
  pp.off_flags = off;
  off += 128;
  pp.off_stats = off;
  off += align_up_p(pp.BT * 2 * 4, 16);
  pp.off_red = off;
  off += align_up_p((kWarps + 1) * pp.BT * 4, 16);
  pp.off_arg = off;
  off += kWarps * 32 * 8;
  pp.off_xs = align_up_p(off, 128);
  off = pp.off_xs + align_up_p(pp.BT * kmax * 2, 128);
  pp.off_ring = align_up_p(off, 128);
  const Tuning& tu = tuning();
  int budget = kSmemMaxP - pp.off_ring;
  if (tu.ring_bytes > 96 * 1024 && tu.ring_bytes < budget) budget = tu.ring_bytes;
  pp.slot_bytes = (budget / kWarps) & ~127;  // per-warp ring bytes
  if (pp.slot_bytes < 4096) {
    snprintf(why, why_len, "activations of K=%d at batch %d leave no room for the rings", kmax, B);
    return false;
  }
  pp.NSW = kBars;
  pp.smem_bytes = pp.off_ring + kWarps * pp.slot_bytes;
  return true;
}

// Per-op schedule inside the persistent kernel: rows per unit, K split and
// pieces, for a per-warp ring of ring_bytes.
bool plan_gemv_persistent(GemvParams& p, int ring_bytes, char* why, size_t why_len) {
  const int nsm = device_sm_count();
  const int GW = nsm * kWarps;
  Sched sc;
  memset(&sc, 0, sizeof sc);
  sc.BT = batch_template_p(p.B);
  if (!sc.BT) {
    snprintf(why, why_len, "the persistent chain supports batch <= 4");
    return false;
  }
  const int K = p.K, nmat = p.nmat;
  const Tuning& tu = tuning();
  auto rgs = [&](int rt) {
    int RG = 0;
    for (int s = 0; s < p.nseg; ++s) {
      p.seg[s].rg_begin = RG;
      RG += (p.seg[s].M + rt - 1) / rt;
    }
    return RG;
  };
  int RT = 4;
  if (tu.force_rt == 1 || tu.force_rt == 2 || tu.force_rt == 4) {
    RT = tu.force_rt;
  } else {
    while (RT > 1 && rgs(RT) < 2 * GW) RT /= 2;
  }
  const int RG = rgs(RT);
  // No K split unless asked for: inside one launch every split unit would pay
  // a fence and an atomic ticket round trip through an L2 loaded by the
  // weight stream, which costs more than the imbalance it removes.
  int S = 1;
  if (tu.force_ksplit > 0 && K % (8 * tu.force_ksplit) == 0 && p.epilogue != EPI_ARGMAX)
    S = tu.force_ksplit;
  sc.RT = RT;
  sc.RG = RG;
  sc.S = S;
  sc.KS = K / S;
  // pieces of at most half the ring, multiples of 8 columns, even
  const int target = tu.piece_bytes > 0 ? tu.piece_bytes : 12288;
  const int cap = ring_bytes / 2 < target ? ring_bytes / 2 : target;
  int maxpc = (cap / (nmat * RT * 2)) & ~7;
  if (maxpc < 8) {
    snprintf(why, why_len, "ring of %d bytes too small", ring_bytes);
    return false;
  }
  if (maxpc >= sc.KS) {
    sc.PC = sc.KS;
    sc.NP = 1;
  } else {
    sc.NP = (sc.KS + maxpc - 1) / maxpc;
    sc.PC = align_up_p((sc.KS + sc.NP - 1) / sc.NP, 8);
    sc.NP = (sc.KS + sc.PC - 1) / sc.PC;
  }
  sc.piece_bytes = nmat * RT * sc.PC * 2;
  sc.NSW = kBars;
  // one "CTA per split" grouping is not used here: units go round-robin over
  // all warps of the grid; Gs and grid describe the launch for the workspace
  sc.Gs = nsm;
  sc.grid = nsm;
  p.sc = sc;
  p.M_total = 0;
  for (int s = 0; s < p.nseg; ++s) p.M_total += p.seg[s].M;
  return true;
}

// The ring bytes per warp the chain's layout leaves (0 if it does not fit).
int persistent_ring_bytes(int B, int kmax) {
  PersistParams pp;
  memset(&pp, 0, sizeof pp);
  char why[128];
  if (!layout_persistent(pp, B, kmax, why, sizeof why)) return 0;
  return pp.slot_bytes;
}

bool plan_persistent(PersistParams& pp, const GemvParams* ops, int nops, int B, char* why,
                     size_t why_len) {
  memset(&pp, 0, sizeof pp);
  if (nops <= 0) {
    snprintf(why, why_len, "empty chain");
    return false;
  }
  int kmax = 8;
  for (int i = 0; i < nops; ++i)
    if (ops[i].K > kmax) kmax = ops[i].K;
  if (!layout_persistent(pp, B, kmax, why, why_len)) return false;
  for (int i = 0; i < nops; ++i) {
    if (ops[i].sc.piece_bytes > pp.slot_bytes / 2) {
      snprintf(why, why_len, "op %d: pieces of %d bytes exceed half a ring", i,
               ops[i].sc.piece_bytes);
      return false;
    }
  }
  const Tuning& tu = tuning();
  pp.grid = device_sm_count();
  pp.nops = nops;
  pp.timeout_ns = tu.timeout_ns;
  pp.evict_first = tu.evict_first;
  pp.err = device_error_ptr();
  return true;
}

typedef void (*PersistKernel)(const PersistParams);

static PersistKernel pick_persistent(int BT) {
  switch (BT) {
    case 1: return (PersistKernel)k_chain_persistent<1>;
    case 2: return (PersistKernel)k_chain_persistent<2>;
    case 4: return (PersistKernel)k_chain_persistent<4>;
    default: return nullptr;
  }
}

bool prepare_persistent(int BT) {
  static std::mutex mu;
  static bool done[64][5] = {{false}};
  PersistKernel k = pick_persistent(BT);
  int dev = 0;
  if (!k || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (!done[dev][BT]) {
    if (cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemMaxP) != cudaSuccess)
      return false;
    done[dev][BT] = true;
  }
  return true;
}

cudaError_t launch_persistent(const PersistParams& pp, cudaStream_t stream) {
  PersistKernel k = pick_persistent(pp.BT);
  if (!k || !prepare_persistent(pp.BT)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(pp.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pp.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident, or no launch
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, pp);
}

}  // namespace ws
