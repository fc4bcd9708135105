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
constexpr int kPersistThreads = (kWarps + 1) * 32;  // eight compute warps + the producer

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The units of op sc that global warp gw runs: gw, gw + GW, ... (dealt
// round-robin over every warp of the grid).
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
  const int rg = c.S == 1 ? u : u / c.S;
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

// Prefetch the cursor's next piece into L2 (no shared memory, no barrier)
// and advance the cursor: the producer's look-ahead, so that weights keep
// streaming from HBM while the rings are full, e.g. across grid barriers.
__device__ __forceinline__ void prefetch_next(const PersistParams& pp, IssueCursor& c, int gw,
                                              int GW) {
  const int u = gw + c.ui * GW;
  const int rg = c.S == 1 ? u : u / c.S;
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
  for (int mat = 0; mat < c.nmat; ++mat) {
    const uint16_t* W = mat == 0 ? W0 : W1;
    if (len == K) {
      bulk_prefetch_l2(W + (size_t)row0 * K, (uint32_t)(rows * K * 2));
    } else {
      for (int r = 0; r < rows; ++r)
        bulk_prefetch_l2(W + (size_t)(row0 + r) * K + c0, (uint32_t)(len * 2));
    }
  }
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

// The (matrices, rows per unit) shape of an op, as one of six kinds, and its
// per-kind inner loop and lane reduction.  Only these two are specialised per
// kind; the rest of a unit's code (waits, ring refills, epilogue) exists once,
// which keeps the kernel's instruction footprint small.
__host__ __device__ inline int unit_kind(int nmat, int RT) {
  return (nmat - 1) * 3 + (RT == 1 ? 0 : (RT == 2 ? 1 : 2));
}

template <int BT>
__device__ __forceinline__ void dot_kind(int kind, float (&acc)[2][4][BT], const uint4* st,
                                         const uint4* xs, int nc, int nchx, int lane) {
  switch (kind) {
    case 0: dot_piece<BT, 1, 1>(acc, st, xs, nc, nc, nchx, lane); break;
    case 1: dot_piece<BT, 1, 2>(acc, st, xs, nc, nc, nchx, lane); break;
    case 2: dot_piece<BT, 1, 4>(acc, st, xs, nc, nc, nchx, lane); break;
    case 3: dot_piece<BT, 2, 1>(acc, st, xs, nc, nc, nchx, lane); break;
    case 4: dot_piece<BT, 2, 2>(acc, st, xs, nc, nc, nchx, lane); break;
    default: dot_piece<BT, 2, 4>(acc, st, xs, nc, nc, nchx, lane); break;
  }
}

template <int BT, int NMAT, int RT>
__device__ __forceinline__ void reduce_t(float (&acc)[2][4][BT], int lane, float& v0, float& v1) {
  constexpr int V = RT * BT;
  float v[NMAT][V];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) v[m][r * BT + b] = acc[m][r][b];
  warp_reduce_scatter<NMAT, V>(v, lane);
  v0 = v[0][0];
  v1 = v[NMAT - 1][0];
}

// Warp totals of a unit: lane group o = r * BT + b (of 32 / (RT * BT) lanes)
// ends with output (row r, batch b) in v0 (first matrix) and v1 (second).
template <int BT>
__device__ __forceinline__ void reduce_kind(int kind, float (&acc)[2][4][BT], int lane, float& v0,
                                            float& v1) {
  switch (kind) {
    case 0: reduce_t<BT, 1, 1>(acc, lane, v0, v1); break;
    case 1: reduce_t<BT, 1, 2>(acc, lane, v0, v1); break;
    case 2: reduce_t<BT, 1, 4>(acc, lane, v0, v1); break;
    case 3: reduce_t<BT, 2, 1>(acc, lane, v0, v1); break;
    case 4: reduce_t<BT, 2, 2>(acc, lane, v0, v1); break;
    default: reduce_t<BT, 2, 4>(acc, lane, v0, v1); break;
  }
}

// Per-op constants of the unit loop.
struct UnitShape {
  int kind, RT, nmat, NP, PC, KS, S, nchx;
  int lg;  // log2 of the lanes per output group, 32 / (RT * BT)
};

// One unit (RT rows x one K split) of op P: consume its NP pieces (refilling
// the ring as they free up), reduce over lanes, then run the epilogue -- or,
// for a split, publish the partial sums and let the last split finish.
template <int BT>
__device__ __forceinline__ void run_unit(const PersistParams& pp, const GemvParams& P,
                                         const UnitShape& us, int u, uint8_t* ring,
                                         uint64_t* bars, uint64_t* empty, const uint4* xs4,
                                         ConsumeState& cs, volatile int* flags,
                                         float& best_v, int& best_i, int lane,
                                         unsigned long long* land_stamp,
                                         unsigned long long* tacc) {
  const int S = us.S, RT = us.RT;
  const int rg = S == 1 ? u : u / S;
  const int ks = u - rg * S;
  int seg, rgl;
  decode_rg(P, rg, seg, rgl);
  const int row0 = rgl * RT;
  const int rows = min(RT, P.seg[seg].M - row0);
  const int R = pp.slot_bytes;
  float acc[2][4][BT];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[m][r][b] = 0.f;

  for (int j = 0; j < us.NP; ++j) {
    const int len = min(us.PC, us.KS - j * us.PC);
    const int ncp = len >> 3;
    const int off = ring_place(cs.pos, piece_size(us.nmat, RT, len), R);
    unsigned long long tw = tacc ? global_ns() : 0;
    const bool ok = cs.abort || mbar_wait_bounded(&bars[cs.n & (kBars - 1)],
                                                  (uint32_t)((cs.n / kBars) & 1), pp.timeout_ns);
    if (tacc) {
      const unsigned long long t = global_ns();
      tacc[0] += t - tw;
      tw = t;
    }
    if (land_stamp && j == 0 && lane == 0) *land_stamp = global_ns();
    if (__any_sync(0xffffffffu, !ok) && !cs.abort) {
      cs.abort = true;
      if (lane == 0) {
        raise_device_error(pp.err, DERR_TIMEOUT);
        flags[2] = 1;  // the producer stops issuing
      }
    }
    // rows of a piece are packed at its own length
    dot_kind<BT>(us.kind, acc, reinterpret_cast<const uint4*>(ring + off),
                 xs4 + ((ks * us.KS + j * us.PC) >> 3), ncp, us.nchx, lane);
    // every lane's reads of this piece have returned: its bytes are free
    __syncwarp();
    if (tacc) tacc[2] += global_ns() - tw;
    if (lane == 0) mbar_arrive(&empty[cs.n & (kBars - 1)]);
    ++cs.n;
  }
  const unsigned long long te = tacc ? global_ns() : 0;
  float v0, v1;
  reduce_kind<BT>(us.kind, acc, lane, v0, v1);
  const int o = lane >> us.lg;
  const int r = o / BT, b = o - (o / BT) * BT;
  const bool mine = (lane & ((1 << us.lg) - 1)) == 0 && r < rows && b < P.B;
  if (S == 1) {
    if (mine) apply_epilogue<-1>(P, seg, row0 + r, b, v0, v1, best_v, best_i);
    if (tacc) tacc[3] += global_ns() - te;
    return;
  }
  const int nmat = us.nmat;
  const int rowg = P.seg[seg].row_base + row0;
  if (mine) {
    P.part[((size_t)(ks * nmat) * P.B + b) * P.M_total + rowg + r] = v0;
    if (nmat == 2) P.part[((size_t)(ks * nmat + 1) * P.B + b) * P.M_total + rowg + r] = v1;
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
    for (int q = lane; q < rows * P.B; q += 32) {
      const int rr = q / P.B;
      const int bb = q - rr * P.B;
      float t0 = 0.f, t1 = 0.f;
      for (int s2 = 0; s2 < S; ++s2) {
        t0 += __ldcg(&P.part[((size_t)(s2 * nmat) * P.B + bb) * P.M_total + rowg + rr]);
        if (nmat == 2)
          t1 += __ldcg(&P.part[((size_t)(s2 * nmat + 1) * P.B + bb) * P.M_total + rowg + rr]);
      }
      float dv = -INFINITY;
      int di = 0x7fffffff;
      apply_epilogue<-1>(P, seg, row0 + rr, bb, t0, nmat == 2 ? t1 : t0, dv, di);
    }
  }
}

// Wait until every CTA has finished op f (bounded).  Thread 0 spins; the
// compute threads leave together.
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
  consumer_sync(kThreads);
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

// The copy producer (the last warp of each CTA).  Lane w < kWarps streams
// compute warp w's pieces of every op, in order, into that warp's ring: a
// piece goes out once one of the warp's eight barriers is free and the piece
// fits behind the last piece the warp has released (its "empty" barrier gets
// one arrival per consumed piece).  The producer never waits for activations,
// so it runs ahead across op boundaries as far as the ring allows.  It polls
// without blocking, so its lanes never wait on each other; if it makes no
// progress for timeout_ns it raises the error flag and stops.
__device__ __noinline__ void produce(const PersistParams& pp, uint8_t* smem, int lane,
                                     volatile int* flags) {
  const int GW = gridDim.x * kWarps;
  const bool active = lane < kWarps;
  const int w = active ? lane : 0;
  const int gw = blockIdx.x * kWarps + w;
  const int R = pp.slot_bytes;
  uint8_t* ring = smem + pp.off_ring + (size_t)w * R;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pp.off_bar) + w * kBars;
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + pp.off_empty) + w * kBars;
  long long* ends = reinterpret_cast<long long*>(smem + pp.off_ends) + w * kBars;
  const uint64_t pol = pp.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
  IssueCursor ic;
  ic.f = active ? -1 : pp.nops;
  ic.q = 0;
  ic.npw = 0;
  ic.ui = 0;
  ic.j = 0;
  ic.n = 0;
  ic.pos.lin = 0;
  ic.pos.off = 0;
  if (active) cursor_seek(pp, ic, gw, GW);
  // look-ahead cursor: up to l2_ahead pieces in front of ic, prefetched to L2
  IssueCursor pf = ic;
  int pf_n = 0;  // pieces prefetched so far
  int consumed = 0;    // pieces this warp is known to have released
  long long freed = 0;  // ring bytes (linear) released so far
  uint64_t idle_since = 0;
  for (;;) {
    bool progress = false;
    const bool stop = flags[2] != 0;
    if (!stop && ic.f < pp.nops) {
      while (consumed < ic.n &&
             mbar_test(&empty[consumed & (kBars - 1)], (uint32_t)((consumed / kBars) & 1))) {
        freed = ends[consumed & (kBars - 1)];
        ++consumed;
        progress = true;
      }
      while (ic.f < pp.nops && ic.n - consumed < kBars) {
        RingPos end = ic.pos;
        ring_place(end, cursor_piece_bytes(ic), R);
        if (end.lin - freed > R) break;
        ends[ic.n & (kBars - 1)] = end.lin;
        issue_next(pp, ic, gw, GW, ring, full, pol);
        progress = true;
      }
      while (pp.l2_ahead > 0 && pf.f < pp.nops && pf_n < ic.n + pp.l2_ahead) {
        if (pf_n < ic.n) {
          // the copies caught up with the look-ahead: skip to them
          pf = ic;
          pf_n = ic.n;
          continue;
        }
        prefetch_next(pp, pf, gw, GW);
        ++pf_n;
        progress = true;
      }
    }
    if (__all_sync(0xffffffffu, stop || ic.f >= pp.nops)) break;
    if (__any_sync(0xffffffffu, progress)) {
      idle_since = 0;
    } else {
      const uint64_t t = global_ns();
      if (idle_since == 0) {
        idle_since = t;
      } else if (t - idle_since > pp.timeout_ns) {
        if (lane == 0) {
          raise_device_error(pp.err, DERR_TIMEOUT);
          flags[2] = 1;
        }
        break;
      }
      __nanosleep(64);
    }
  }
  if (flags[2] && active) {
    // stopped early: let this warp's copies still in flight land before exit
    for (int q = consumed; q < ic.n; ++q)
      mbar_wait_bounded(&full[q & (kBars - 1)], (uint32_t)((q / kBars) & 1), pp.timeout_ns);
  }
}

template <int BT>
__global__ void __launch_bounds__(kPersistThreads, 1)
    k_chain_persistent(const __grid_constant__ PersistParams pp) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + pp.off_flags);
  if (tid == 0) {
    flags[1] = 0;
    flags[2] = 0;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + pp.off_bar);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + pp.off_empty);
    for (int s = 0; s < kWarps * kBars; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    produce(pp, smem, lane, flags);
  } else {
    const int GW = gridDim.x * kWarps;
    const int gw = blockIdx.x * kWarps + warp;
    GemvParams* Ps = reinterpret_cast<GemvParams*>(smem + pp.off_op);  // two buffers
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pp.off_bar) + warp * kBars;
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + pp.off_empty) + warp * kBars;
    float* stats = reinterpret_cast<float*>(smem + pp.off_stats);
    float* red = reinterpret_cast<float*>(smem + pp.off_red);
    float* argv = reinterpret_cast<float*>(smem + pp.off_arg);
    int* argi = reinterpret_cast<int*>(argv + kWarps * 32);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + pp.off_xs);
    const uint4* xs4 = reinterpret_cast<const uint4*>(xs);
    uint8_t* ring = smem + pp.off_ring + (size_t)warp * pp.slot_bytes;
    ConsumeState cs;
    cs.n = 0;
    cs.pos.lin = 0;
    cs.pos.off = 0;
    cs.abort = false;
    prefetch_descriptor(pp.ops, Ps, tid);

    for (int f = 0; f < pp.nops; ++f) {
      if (f > 0) {
        grid_wait(pp, f - 1, flags, tid);
        copy_trace(pp.ops + (f - 1), tid);
      }
      wait_descriptor();
      consumer_sync(kThreads);
      unsigned long long* stamp =
          pp.stamps ? pp.stamps + ((size_t)blockIdx.x * pp.nops + f) * kStampsPerOp : nullptr;
      if (stamp && tid == 0) stamp[0] = global_ns();
      const GemvParams& P = Ps[f & 1];
      // the next op's descriptor streams in while this op runs
      if (f + 1 < pp.nops) prefetch_descriptor(pp.ops + f + 1, &Ps[(f + 1) & 1], tid);
      // all K columns: units of every split index into them
      if (!prologue_stage_fused<BT>(P, stats, red, xs, tid)) {
        prologue_stats<BT>(P, stats, red, tid);
        stage_x<BT>(P, stats, xs, 0, P.K >> 3, tid);
      }
      consumer_sync(kThreads);
      if (stamp && tid == 0) stamp[1] = global_ns();

      const int nunits = warp_units(P.sc, gw, GW);
      // diagnostics: this warp's time waiting for pieces, in dot products
      // and in the reduction and epilogue, in this op
      unsigned long long tacc_v[4] = {0, 0, 0, 0};
      unsigned long long* wwait = stamp ? tacc_v : nullptr;
      float best_v = -INFINITY;
      int best_i = 0x7fffffff;
      UnitShape us;
      us.kind = unit_kind(P.nmat, P.sc.RT);
      us.RT = P.sc.RT;
      us.nmat = P.nmat;
      us.NP = P.sc.NP;
      us.PC = P.sc.PC;
      us.KS = P.sc.KS;
      us.S = P.sc.S;
      us.nchx = P.K >> 3;
      us.lg = __ffs(32 / (us.RT * BT)) - 1;
      for (int t = 0; t < nunits; ++t) {
        unsigned long long* land = (stamp && warp == 0 && t == 0) ? stamp + 3 : nullptr;
        run_unit<BT>(pp, P, us, gw + t * GW, ring, bars, empty, xs4, cs, flags, best_v, best_i,
                     lane, land, wwait);
      }

      if (stamp && lane == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) stamp[4 + 5 * warp + i] = tacc_v[i];
        stamp[8 + 5 * warp] = (unsigned long long)nunits;
      }
      if (P.epilogue == EPI_ARGMAX) {
        const int RT = P.sc.RT;
        argv[warp * 32 + lane] = best_v;
        argi[warp * 32 + lane] = best_i;
        consumer_sync(kThreads);
        if (tid < P.B) {
          float bv = -INFINITY;
          int bi = 0x7fffffff;
          for (int w = 0; w < kWarps; ++w)
            for (int r = 0; r < RT; ++r) {
              const int l = (r * BT + tid) * (32 / (RT * BT));
              if (arg_better(argv[w * 32 + l], argi[w * 32 + l], bv, bi)) {
                bv = argv[w * 32 + l];
                bi = argi[w * 32 + l];
              }
            }
          P.arg_val[(size_t)blockIdx.x * P.B + tid] = bv;
          P.arg_idx[(size_t)blockIdx.x * P.B + tid] = bi;
          __threadfence();
        }
        consumer_sync(kThreads);
        if (tid == 0) {
          const unsigned old = atomicAdd(P.arg_ticket, 1u);
          const int last = old == gridDim.x - 1;
          if (last) atomicExch(P.arg_ticket, 0u);
          flags[0] = last;
        }
        consumer_sync(kThreads);
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
      // this CTA is done with op f: its outputs are written.  The CTA barrier
      // orders every thread's stores before thread 0's fence, which makes
      // them visible GPU-wide before the arrival is counted.
      consumer_sync(kThreads);
      if (stamp && tid == 0) stamp[2] = global_ns();
      if (tid == 0) {
        __threadfence();
        atomicAdd(pp.bar + f, 1u);
      }
    }
    if (pp.nops > 0 && pp.ops[pp.nops - 1].trace_out) {
      grid_wait(pp, pp.nops - 1, flags, tid);
      copy_trace(pp.ops + (pp.nops - 1), tid);
    }
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
  pp.off_bar = off;  // "full" barriers: a piece landed
  off += kWarps * kBars * 8;
  pp.off_empty = off;  // "empty" barriers: a piece was consumed
  off += kWarps * kBars * 8;
  pp.off_ends = off;  // producer's record of its pieces' ring ends
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
  // rows per unit: 4 only where every warp gets many units (the LM head);
  // else 2 (measured faster than 1 for the decode-chain ops, even where some
  // warps then get no unit: pieces are larger and per-unit work halves)
  int RT = 2;
  if (tu.force_rt == 1 || tu.force_rt == 2 || tu.force_rt == 4) {
    RT = tu.force_rt;
  } else if (rgs(4) >= 8 * GW) {
    RT = 4;
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
  pp.l2_ahead = tu.l2_ahead;
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
  cfg.blockDim = dim3(kPersistThreads);
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
