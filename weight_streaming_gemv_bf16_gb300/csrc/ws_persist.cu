// ws_persist.cu -- the persistent chain kernel: a whole decode step (every op
// of the chain) in one cooperative launch, one CTA per SM.
//
// The ops of a chain depend on each other only through their small
// activation vectors; their weights -- all but ~0.01% of the bytes -- do not
// depend on anything.  So each warp streams its weight pieces of every op, in
// order, through its own ring of shared-memory stages, and its copy cursor
// runs ahead across op boundaries.  Between ops the CTAs meet at a grid
// barrier (the previous op's outputs are complete), normalise the next
// activation vector into shared memory and compute on pieces that have
// usually already landed.  HBM keeps streaming through every barrier and
// prologue as long as the rings (about 190 KB per SM) have room, which is
// what a chain of separate launches cannot do: there each op boundary drains
// the memory pipeline ("One Token, Kernel by Kernel: A Decode Step on a
// Laptop GPU", Step 3, where kernel gaps are counted against the bandwidth
// floor).
//
// Work split, epilogues and numerics are those of k_stream_gemv (one warp
// per task of RT rows, full K, pieces of PC columns), so every op computes
// exactly what the standalone entry point computes with S = 1.  All waits are
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

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The copy cursor of one warp (advanced by lane 0 only): the next piece to
// stream, walking this warp's pieces of every op in order.  The current op's
// shape and weight pointers are kept in registers, so a copy costs no
// descriptor reads.
struct IssueCursor {
  int f;     // op
  int q;     // piece within the op
  int npw;   // pieces of this warp in op f
  int ti;    // task within the op
  int j;     // piece within the task
  int rgw;   // this warp's first row group in op f
  int slot;  // ring stage of the next piece
  int n;     // pieces issued so far
  // op f, cached
  int nseg, nmat, RT, PC, NP, K;
  int M[kMaxSeg], rgb[kMaxSeg];
  const uint16_t* W0[kMaxSeg];
  const uint16_t* W1[kMaxSeg];
};

__device__ __forceinline__ void cursor_seek(const PersistParams& pp, IssueCursor& c, int warp) {
  while (c.f < pp.nops && c.q >= c.npw) {
    ++c.f;
    c.q = 0;
    c.ti = 0;
    c.j = 0;
    c.npw = 0;
    if (c.f < pp.nops) {
      const GemvParams& P = pp.ops[c.f];
      int ks, rg0, rg1;
      cta_range(P.sc, blockIdx.x, ks, rg0, rg1);
      c.NP = P.sc.NP;
      c.npw = warp_tasks(rg0, rg1, warp) * c.NP;
      c.rgw = rg0 + warp;
      c.nseg = P.nseg;
      c.nmat = P.nmat;
      c.RT = P.sc.RT;
      c.PC = P.sc.PC;
      c.K = P.K;
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

__device__ __forceinline__ void issue_next(const PersistParams& pp, IssueCursor& c, int warp,
                                           uint8_t* ring, uint64_t* full, uint64_t pol) {
  const int rg = c.rgw + c.ti * kWarps;
  // segment by selects (the cached arrays stay in registers)
  const bool s1 = c.nseg > 1 && rg >= c.rgb[1];
  const bool s2 = c.nseg > 2 && rg >= c.rgb[2];
  const int rgb = s2 ? c.rgb[2] : (s1 ? c.rgb[1] : c.rgb[0]);
  const int Mseg = s2 ? c.M[2] : (s1 ? c.M[1] : c.M[0]);
  const uint16_t* W0 = s2 ? c.W0[2] : (s1 ? c.W0[1] : c.W0[0]);
  const uint16_t* W1 = s2 ? c.W1[2] : (s1 ? c.W1[1] : c.W1[0]);
  const int RT = c.RT, PC = c.PC, K = c.K;
  const int row0 = (rg - rgb) * RT;
  const int rows = min(RT, Mseg - row0);
  const int c0 = c.j * PC;
  const int len = min(PC, K - c0);
  uint8_t* dst = ring + (size_t)c.slot * pp.slot_bytes;
  uint64_t* bar = &full[c.slot];
  mbar_arrive_expect_tx(bar, (uint32_t)(c.nmat * rows * len * 2));
  for (int mat = 0; mat < c.nmat; ++mat) {
    const uint16_t* W = mat == 0 ? W0 : W1;
    if (len == K) {
      bulk_copy_g2s(dst + (size_t)mat * RT * PC * 2, W + (size_t)row0 * K,
                    (uint32_t)(rows * K * 2), bar, pol);
    } else {
      for (int r = 0; r < rows; ++r)
        bulk_copy_g2s(dst + ((size_t)mat * RT + r) * PC * 2, W + (size_t)(row0 + r) * K + c0,
                      (uint32_t)(len * 2), bar, pol);
    }
  }
  ++c.n;
  ++c.q;
  if (++c.j == c.NP) {
    c.j = 0;
    ++c.ti;
  }
  if (++c.slot == pp.NSW) c.slot = 0;
  cursor_seek(pp, c, warp);
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

struct ConsumeState {
  int slot;
  uint32_t phase;
  bool abort;
};

// One task (RT rows, full K) of op P: consume its NP pieces, refilling each
// stage with the cursor's next piece, then reduce and run the epilogue.
template <int BT, int NMAT, int RT>
__device__ __forceinline__ void run_task(const PersistParams& pp, const GemvParams& P, int rg,
                                         uint8_t* ring, uint64_t* full, const uint4* xs4,
                                         ConsumeState& cs, IssueCursor& ic, uint64_t pol,
                                         float& best_v, int& best_i, int warp, int lane,
                                         unsigned long long* land_stamp) {
  int seg, rgl;
  decode_rg(P, rg, seg, rgl);
  const int row0 = rgl * RT;
  const int rows = min(RT, P.seg[seg].M - row0);
  const int NP = P.sc.NP, PC = P.sc.PC, ncp = PC >> 3, nchx = P.K >> 3;
  float acc[NMAT][RT][BT];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[m][r][b] = 0.f;

  for (int j = 0; j < NP; ++j) {
    const int len = min(PC, P.K - j * PC);
    const bool ok = cs.abort || mbar_wait_bounded(&full[cs.slot], cs.phase, pp.timeout_ns);
    if (land_stamp && j == 0 && lane == 0) *land_stamp = global_ns();
    if (__any_sync(0xffffffffu, !ok) && !cs.abort) {
      cs.abort = true;
      if (lane == 0) raise_device_error(pp.err, DERR_TIMEOUT);
    }
    const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)cs.slot * pp.slot_bytes);
    const int xoff = j * ncp;
#pragma unroll 2
    for (int c = lane; c < (len >> 3); c += 32) {
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
    // every lane's reads of this stage have returned: refill it with the
    // cursor's next piece (possibly of a later op)
    __syncwarp();
    if (lane == 0 && !cs.abort && ic.f < pp.nops) issue_next(pp, ic, warp, ring, full, pol);
    if (++cs.slot == pp.NSW) {
      cs.slot = 0;
      cs.phase ^= 1u;
    }
  }
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[m][r][b] = warp_sum(acc[m][r][b]);
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int b = 0; b < BT; ++b)
      if (lane == r * BT + b && r < rows && b < P.B)
        apply_epilogue(P, seg, row0 + r, b, acc[0][r][b], acc[NMAT - 1][r][b], best_v, best_i);
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
  GemvParams* Ps = reinterpret_cast<GemvParams*>(smem + pp.off_op);  // two buffers
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pp.off_bar) + warp * kMaxStages;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + pp.off_flags);
  float* stats = reinterpret_cast<float*>(smem + pp.off_stats);
  float* red = reinterpret_cast<float*>(smem + pp.off_red);
  float* argv = reinterpret_cast<float*>(smem + pp.off_arg);
  int* argi = reinterpret_cast<int*>(argv + kWarps * 32);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + pp.off_xs);
  const uint4* xs4 = reinterpret_cast<const uint4*>(xs);
  uint8_t* ring = smem + pp.off_ring + (size_t)warp * pp.NSW * pp.slot_bytes;

  IssueCursor ic;
  ic.f = -1;
  ic.q = 0;
  ic.npw = 0;
  ic.ti = 0;
  ic.j = 0;
  ic.rgw = 0;
  ic.slot = 0;
  ic.n = 0;
  uint64_t pol = 0;
  if (tid == 0) flags[1] = 0;
  if (lane == 0) {
    for (int s = 0; s < pp.NSW; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    pol = pp.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
    cursor_seek(pp, ic, warp);
    for (int k = 0; k < pp.NSW && ic.f < pp.nops; ++k) issue_next(pp, ic, warp, ring, full, pol);
  }
  ConsumeState cs;
  cs.slot = 0;
  cs.phase = 0;
  cs.abort = false;
  prefetch_descriptor(pp.ops, Ps, tid);

  for (int f = 0; f < pp.nops; ++f) {
    if (f > 0) {
      grid_wait(pp, f - 1, flags, tid);
      copy_trace(pp.ops + (f - 1), tid);
    }
    wait_descriptor();
    __syncthreads();
    unsigned long long* stamp = pp.stamps ? pp.stamps + ((size_t)blockIdx.x * pp.nops + f) * 4 : nullptr;
    if (stamp && tid == 0) stamp[0] = global_ns();
    const GemvParams& P = Ps[f & 1];
    // the next op's descriptor streams in while this op runs
    if (f + 1 < pp.nops) prefetch_descriptor(pp.ops + f + 1, &Ps[(f + 1) & 1], tid);
    if (!prologue_stage_fused<BT>(P, stats, red, xs, tid)) {
      prologue_stats<BT>(P, stats, red, tid);
      stage_x<BT>(P, stats, xs, 0, tid);
    }
    __syncthreads();
    if (stamp && tid == 0) stamp[1] = global_ns();

    int ks, rg0, rg1;
    cta_range(P.sc, blockIdx.x, ks, rg0, rg1);
    const int ntask = warp_tasks(rg0, rg1, warp);
    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    const int kind = (P.nmat - 1) * 3 + (P.sc.RT == 1 ? 0 : (P.sc.RT == 2 ? 1 : 2));
    for (int t = 0; t < ntask; ++t) {
      const int rg = rg0 + warp + t * kWarps;
      unsigned long long* land = (stamp && warp == 0 && t == 0) ? stamp + 3 : nullptr;
      switch (kind) {
        case 0: run_task<BT, 1, 1>(pp, P, rg, ring, full, xs4, cs, ic, pol, best_v, best_i, warp, lane, land); break;
        case 1: run_task<BT, 1, 2>(pp, P, rg, ring, full, xs4, cs, ic, pol, best_v, best_i, warp, lane, land); break;
        case 2: run_task<BT, 1, 4>(pp, P, rg, ring, full, xs4, cs, ic, pol, best_v, best_i, warp, lane, land); break;
        case 3: run_task<BT, 2, 1>(pp, P, rg, ring, full, xs4, cs, ic, pol, best_v, best_i, warp, lane, land); break;
        case 4: run_task<BT, 2, 2>(pp, P, rg, ring, full, xs4, cs, ic, pol, best_v, best_i, warp, lane, land); break;
        default: run_task<BT, 2, 4>(pp, P, rg, ring, full, xs4, cs, ic, pol, best_v, best_i, warp, lane, land); break;
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
    for (int q = ic.n - pp.NSW; q < ic.n; ++q)
      if (q >= 0) mbar_wait_bounded(&full[q % pp.NSW], (q / pp.NSW) & 1, pp.timeout_ns);
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

bool plan_gemv_persistent(GemvParams& p, int slot_bytes, char* why, size_t why_len) {
  const int nsm = device_sm_count();
  const int warps_total = nsm * kWarps;
  Sched sc;
  memset(&sc, 0, sizeof sc);
  sc.BT = batch_template_p(p.B);
  if (!sc.BT) {
    snprintf(why, why_len, "the persistent chain supports batch <= 4");
    return false;
  }
  const int K = p.K, nmat = p.nmat;
  const int rt_max = 4;  // BT <= 4
  int RT = rt_max;
  const Tuning& tu = tuning();
  auto rgs = [&](int rt) {
    int RG = 0;
    for (int s = 0; s < p.nseg; ++s) {
      p.seg[s].rg_begin = RG;
      RG += (p.seg[s].M + rt - 1) / rt;
    }
    return RG;
  };
  if (tu.force_rt == 1 || tu.force_rt == 2 || tu.force_rt == 4) {
    RT = tu.force_rt;
  } else {
    while (RT > 1 && rgs(RT) < 2 * warps_total) RT /= 2;
  }
  // a piece of RT rows must fit a stage with at least 8 columns
  while (RT > 1 && nmat * RT * 8 * 2 > slot_bytes) RT /= 2;
  sc.RT = RT;
  sc.RG = rgs(RT);
  sc.S = 1;
  sc.KS = K;
  int maxpc = (slot_bytes / (nmat * RT * 2)) & ~7;
  if (maxpc < 8) {
    snprintf(why, why_len, "stage of %d bytes too small", slot_bytes);
    return false;
  }
  if (maxpc >= K) {
    sc.PC = K;
    sc.NP = 1;
  } else {
    sc.NP = (K + maxpc - 1) / maxpc;
    sc.PC = align_up_p((K + sc.NP - 1) / sc.NP, 8);
    sc.NP = (K + sc.PC - 1) / sc.PC;
  }
  sc.piece_bytes = nmat * RT * sc.PC * 2;
  sc.NSW = 0;
  sc.Gs = nsm;
  sc.grid = nsm;
  p.sc = sc;
  p.M_total = 0;
  for (int s = 0; s < p.nseg; ++s) p.M_total += p.seg[s].M;
  return true;
}

bool plan_persistent(PersistParams& pp, const GemvParams* ops, int nops, int B, char* why,
                     size_t why_len) {
  memset(&pp, 0, sizeof pp);
  pp.BT = batch_template_p(B);
  if (!pp.BT || nops <= 0) {
    snprintf(why, why_len, "the persistent chain supports batch <= 4");
    return false;
  }
  const Tuning& tu = tuning();
  int kmax = 8, slot = 0;
  for (int i = 0; i < nops; ++i) {
    if (ops[i].K > kmax) kmax = ops[i].K;
    if (ops[i].sc.piece_bytes > slot) slot = ops[i].sc.piece_bytes;
  }
  pp.slot_bytes = align_up_p(slot, 128);
  int off = 0;
  pp.off_op = off;
  off += 2 * align_up_p((int)sizeof(GemvParams), 128);
  pp.off_bar = off;
  off += kWarps * kMaxStages * 8;
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
  int budget = kSmemMaxP - pp.off_ring;
  if (tu.ring_bytes > 96 * 1024 && tu.ring_bytes < budget) budget = tu.ring_bytes;
  int NSW = budget / (kWarps * pp.slot_bytes);
  if (NSW > kMaxStages) NSW = kMaxStages;
  if (NSW < 2) {
    snprintf(why, why_len, "activations of K=%d at batch %d leave no room for the rings", kmax, B);
    return false;
  }
  pp.NSW = NSW;
  pp.smem_bytes = pp.off_ring + kWarps * NSW * pp.slot_bytes;
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
