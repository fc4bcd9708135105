// ws_gemv_host.cu -- host side of the streaming GEMV: the schedule (rows per
// warp task, K splits, pieces, ring depth, grid), workspace layout, kernel
// selection and launch, and the GEMV-family entry points of the C ABI.  The
// kernel itself is in ws_gemv_kernel.cuh.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <set>

#include "wsgemv.h"
#include "ws_common.cuh"
#include "ws_gemv_kernel.cuh"

namespace ws {

// Device error flag: set by a bounded wait that ran out (read by
// ws_device_error).
__device__ int g_device_error;

// host side
// ---------------------------------------------------------------------------

static thread_local char g_msg[512];

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
}

Tuning& tuning() {
  static Tuning t = {96 * 1024, 0, 0, 0, 1, 12288, 2000000000ull, 0, 1, 0, 0, 0, 1};
  return t;
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

int* device_error_ptr() {
  static int* cache[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(ptr);
  }
  return cache[dev];
}

static int batch_template(int B) {
  if (B <= 1) return 1;
  if (B <= 2) return 2;
  if (B <= 4) return 4;
  if (B <= 8) return 8;
  return 16;
}

static int align_up(int v, int a) { return (v + a - 1) / a * a; }

static constexpr int kXsMax = 96 * 1024;  // activations in shared memory without a K split
// The same for the CUDA-core kernel: Wd (1536 x 8960) keeps an unsplit K at
// batch 8 and two splits at batch 16 (a ring of 2 x 5 KB a warp beside
// 140 KB of activations) instead of two and four: every split costs each task
// a fence and a ticket round trip, and the last split's epilogue a tail
// (measured on the decode step: batch 8 1431 -> 1279 us, Wd 19.6 -> 15.0 us;
// batch 16 2349 -> 2286 us, Wd's CTA end spread 10.2 -> 2.8 us).
static constexpr int kXsMaxCC = 144 * 1024;
static constexpr int kSmemMax = 227 * 1024;
static constexpr int kSmemReserved = 1024;  // shared memory the runtime keeps per resident CTA

// Shared memory of one SM of the current device (228 KB on GB300).
static int smem_per_sm() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 228 * 1024;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        n <= 0)
      n = 228 * 1024;
    cache[dev] = n;
  }
  return cache[dev];
}

static int resident_ctas(const GemvParams& p);

static int row_groups(GemvParams& p, int RT) {
  int RG = 0;
  for (int s = 0; s < p.nseg; ++s) {
    p.seg[s].rg_begin = RG;
    RG += (p.seg[s].M + RT - 1) / RT;
  }
  return RG;
}

static constexpr int kMmaTaskRows = 16;  // one m16 tile per warp task

// The chain form of a launch for the tensor-core kernel (any K split), or
// F_ANY.  The one-round RMSNorm reads the whole K: B x K / 8 chunks within
// form_round_chunks(BT) per thread.
static int mma_form(const GemvParams& p, int BT) {
  if (p.prologue == PRO_RMSNORM && p.x_dtype == DT_F32 &&
      p.B * (p.K >> 3) <= form_round_chunks(BT) * kThreads) {
    if (p.epilogue == EPI_F32) return F_RMS_F32;
    if (p.epilogue == EPI_SWIGLU && p.nmat == 2 && p.nseg == 1) return F_RMS_SWIGLU;
    if (p.epilogue == EPI_ARGMAX && p.nseg == 1) return F_RMS_ARGMAX;
    return F_ANY;
  }
  if (p.prologue == PRO_NONE && p.x_dtype == DT_BF16 && p.epilogue == EPI_RESID && p.nseg == 1)
    return F_BF16_RESID;
  if (p.prologue == PRO_NONE && p.x_dtype == DT_BF16 && p.epilogue == EPI_F32 && p.nseg == 1)
    return F_BF16_F32;
  return F_ANY;
}

// Schedule for the tensor-core kernel (batch tiles 8 and 16, chain forms,
// at least 8 Mi weights): 16-row tasks; a K split until the tasks cover most
// streaming warps (none for the argmax, which needs whole rows) and the
// split's activations fit; pieces of 8-24 KB; rows an odd number of
// 16-byte units apart.  Smaller ops (QKV, Wo of a 1.5B model) keep the
// CUDA-core kernels: measured at batch 16, 16-row tasks leave too few tasks
// and too long a split-K tail for them (Wo 15.9 vs 6.9 us) while gate/up, Wd
// and the LM head run faster (24 vs 37, 21 vs 31, 105 vs 201 us).  False when
// the launch does not qualify.
static bool plan_gemv_mma(GemvParams& p, int force_S, int grid_target) {
  const int BT = batch_template(p.B);
  const int K = p.K, nmat = p.nmat;
  if (BT < 8 || K % 16 != 0) return false;
  long long weights = 0;
  for (int s = 0; s < p.nseg; ++s) weights += (long long)p.seg[s].M * K * nmat;
  if (weights < (8ll << 20)) return false;
  const int F = mma_form(p, BT);
  if (F == F_ANY) return false;
  Sched sc;
  memset(&sc, 0, sizeof sc);
  sc.BT = BT;
  sc.RT = kMmaTaskRows;
  const int RG = row_groups(p, kMmaTaskRows);
  sc.RG = RG;
  const int warps_total = grid_target * kMmaWarps;
  auto valid = [&](int S) { return S >= 1 && K % (16 * S) == 0; };
  auto xs_bytes = [&](int S) { return BT * (((K / S) >> 3) | 1) * 16; };
  int S = 1;
  if (F == F_RMS_ARGMAX || force_S < 0) {
    if (xs_bytes(1) > kXsMax) return false;
  } else if (force_S > 0) {
    S = force_S;
    if (!valid(S) || xs_bytes(S) > kXsMax) return false;
  } else {
    while (S <= 64 && !(valid(S) && xs_bytes(S) <= kXsMax)) ++S;
    if (S > 64) return false;
    for (int s = S + 1; s <= 32 && RG * S < (warps_total * 3) / 4; ++s)
      if (valid(s) && K / s >= 128) S = s;
  }
  sc.S = S;
  sc.KS = K / S;
  sc.xrs = (sc.KS >> 3) | 1;
  int off = 0;
  sc.off_bar = off;
  off += kWarps * kMaxStages * 8;
  sc.off_flags = off;
  off += 128;
  sc.off_stats = off;
  off += align_up(sc.BT * 2 * 4, 16);
  sc.off_red = off;
  off += align_up((kWarps + 1) * sc.BT * 4, 16);
  sc.off_arg = off;
  off += kWarps * 32 * 8;
  sc.off_xs = align_up(off, 128);
  off = sc.off_xs + align_up(xs_bytes(S), 128);
  sc.off_ring = align_up(off, 128);
  int Gs = grid_target / S;
  if (Gs < 1) Gs = 1;
  if (Gs > RG) Gs = RG;
  if ((unsigned long long)Gs * (unsigned long long)RG >= (1ull << 32)) return false;
  sc.Gs = Gs;
  sc.grid = S * Gs;
  // residual rows of the CTA, read ahead (unsplit K only: a split's last
  // CTA reads them at the epilogue)
  const int res_bytes = (p.epilogue == EPI_RESID && S == 1)
                            ? (RG + Gs - 1) / Gs * kMmaTaskRows * BT * 4
                            : 0;
  // pieces (16-column multiples) of about 24 KB over all matrices at batch
  // tile 8 and 16 KB at 16, else smaller, with two ring stages per streaming
  // warp (measured on the chain: batch 8 24 KB 1249 vs 16 KB 1387 vs 8 KB
  // 1845 us; batch 16 16 KB 1873 vs 24 KB 1909 us)
  int NSW = 0;
  for (const int target : {24576, 16384, 8192}) {
    if (BT == 16 && target > 16384) continue;
    const int pc = target / (nmat * kMmaTaskRows * 2);
    if (pc >= sc.KS) {
      sc.PC = sc.KS;
      sc.NP = 1;
    } else {
      sc.NP = (sc.KS + pc - 1) / pc;
      sc.PC = align_up((sc.KS + sc.NP - 1) / sc.NP, 16);
      sc.NP = (sc.KS + sc.PC - 1) / sc.PC;
    }
    int u = (sc.PC * 2 + 15) / 16;
    if (u % 2 == 0) ++u;
    sc.prow = u * 16;
    sc.piece_bytes = align_up(nmat * kMmaTaskRows * sc.prow, 128);
    NSW = (kSmemMax - sc.off_ring - res_bytes - 16) / (kMmaWarps * sc.piece_bytes);
    if (NSW >= 2) break;
  }
  if (NSW > kMaxStages) NSW = kMaxStages;
  if (NSW < 2) return false;
  sc.NSW = NSW;
  sc.smem_bytes = sc.off_ring + kMmaWarps * NSW * sc.piece_bytes;
  if (res_bytes) {
    sc.off_res = align_up(sc.smem_bytes, 16);
    sc.res_rows = (RG + Gs - 1) / Gs * kMmaTaskRows;
    sc.smem_bytes = sc.off_res + res_bytes;
  }
  sc.mma = 1;
  sc.form = F;
  p.sc = sc;
  p.M_total = 0;
  for (int s = 0; s < p.nseg; ++s) p.M_total += p.seg[s].M;
  return true;
}

// Schedule of the tensor-core kernel for 4-bit rows (chain forms, B <= 4,
// every size): 16-row tasks over all eight warps, no K split, the B
// activation rows staged once (padding rows of the fragments read a zero
// row), pieces of whole super-groups of at most 24 KB over all matrices
// (whole rows when they fit), rows an odd number of 16-byte units apart,
// and as many ring stages as shared memory holds (up to eight).
static bool plan_gemv_q4mma(GemvParams& p, int grid_target) {
  const int K = p.K, nmat = p.nmat;
  if (p.B > 4 || K % kQ4Group != 0) return false;
  const int F = mma_form(p, 4);  // four activation rows staged
  if (F == F_ANY || !pick_kernel_q4mma(nmat, F)) return false;
  Sched sc;
  memset(&sc, 0, sizeof sc);
  sc.BT = 8;
  sc.RT = kMmaTaskRows;
  const int RG = row_groups(p, kMmaTaskRows);
  // only ops with at least two 16-row tasks per warp (the LM head): with
  // fewer, most warps idle and a task's single warp streams its whole K
  // (measured: the 1536 x 8960 Wd 37.6 us on this kernel, 5.6 on the
  // CUDA-core one)
  if (RG < 2 * grid_target * kWarps) return false;
  sc.RG = RG;
  sc.S = 1;
  sc.KS = K;
  sc.xrs = (K >> 3) | 1;
  const int xs_bytes = 4 * sc.xrs * 16;
  if (xs_bytes > kXsMax) return false;
  int off = 0;
  sc.off_bar = off;
  off += kWarps * kMaxStages * 8;
  sc.off_flags = off;
  off += 128;
  sc.off_stats = off;
  off += align_up(sc.BT * 2 * 4, 16);
  sc.off_red = off;
  off += align_up((kWarps + 1) * sc.BT * 4, 16);
  sc.off_arg = off;
  off += kWarps * 32 * 8;
  sc.off_xzero = off;
  off += 16;
  sc.off_xsum = off;
  off += 8 * (K / kQ4Group) * 4;
  sc.off_xs = align_up(off, 128);
  off = sc.off_xs + align_up(xs_bytes, 128);
  sc.off_ring = align_up(off, 128);
  int Gs = grid_target;
  if (Gs > RG) Gs = RG;
  if ((unsigned long long)Gs * (unsigned long long)RG >= (1ull << 32)) return false;
  sc.Gs = Gs;
  sc.grid = Gs;
  const int res_bytes =
      p.epilogue == EPI_RESID ? (RG + Gs - 1) / Gs * kMmaTaskRows * sc.BT * 4 : 0;
  // pieces: the largest run of whole super-groups (whole rows first) of at
  // most 24 KB over all matrices that leaves every warp three ring stages,
  // else two
  const int avail = kSmemMax - sc.off_ring - res_bytes - 16;
  int NSW = 0;
  for (const int need : {3, 2}) {
    for (int pc = K; pc >= kQ4Super || pc == K; pc = (pc == K ? (K - 1) / kQ4Super * kQ4Super
                                                             : pc - kQ4Super)) {
      if (pc <= 0) break;
      int u = (q4_prefix(pc) + 15) / 16;
      if (u % 2 == 0) ++u;
      const int pb = align_up(nmat * kMmaTaskRows * u * 16, 128);
      if (pb > 24576 && pc > kQ4Super) continue;
      const int nsw = avail / (kWarps * pb);
      if (nsw >= need) {
        sc.PC = pc;
        sc.prow = u * 16;
        sc.piece_bytes = pb;
        NSW = nsw;
        break;
      }
    }
    if (NSW) break;
  }
  if (NSW < 2) return false;
  sc.NP = (K + sc.PC - 1) / sc.PC;
  if (NSW > kMaxStages) NSW = kMaxStages;
  sc.NSW = NSW;
  sc.smem_bytes = sc.off_ring + kWarps * NSW * sc.piece_bytes;
  if (res_bytes) {
    sc.off_res = align_up(sc.smem_bytes, 16);
    sc.res_rows = (RG + Gs - 1) / Gs * kMmaTaskRows;
    sc.smem_bytes = sc.off_res + res_bytes;
  }
  sc.mma = 1;
  sc.form = F;
  p.sc = sc;
  p.M_total = 0;
  for (int s = 0; s < p.nseg; ++s) p.M_total += p.seg[s].M;
  return true;
}

// Schedule of the CUDA-core kernel with `cps` CTAs resident per SM: the grid
// targets cps CTAs per SM and the shared memory of each (activations, rings,
// residual rows) stays within the SM's share for that many.
static bool plan_gemv_cc(GemvParams& p, int force_S, int cps, char* why, size_t why_len) {
  const Tuning& tu = tuning();
  const int nsm = device_sm_count();
  const int grid_target = tu.grid_cap > 0 ? tu.grid_cap : nsm * cps;
  const int warps_total = grid_target * kWarps;
  const bool q4 = p.wfmt == WF_Q4;
  const int smem_cap = cps > 1 ? smem_per_sm() / cps - kSmemReserved : kSmemMax;
  Sched sc;
  memset(&sc, 0, sizeof sc);
  sc.BT = batch_template(p.B);
  const int K = p.K, nmat = p.nmat;
  // bytes of one weight row (4-bit rows: whole super-groups)
  const long row_b = q4 ? q4_prefix(K) : (long)K * 2;
  if (q4 && (K % kQ4Group != 0 || sc.BT > 4)) {
    snprintf(why, why_len, "4-bit weights need K a multiple of 128 and B <= 4 (K=%d, B=%d)", K,
             p.B);
    return false;
  }

  // rows per task: up to 4, and RT x BT <= 32 (one output per lane group).  Cost of a choice: the heaviest warp's rows,
  // ceil(tasks / warps) x RT, times the shared-memory time per weight row when
  // it exceeds the HBM time: each 16-byte weight chunk takes BT activation
  // chunks shared by the task's RT rows, and shared memory reads about 5.5x
  // an SM's share of HBM (0.18 = 1 / 5.5).  Lowest cost wins (ties within
  // 10%); among those, the largest RT whose piece still holds whole rows (one
  // contiguous copy per matrix), else the largest.  Measured on the decode
  // chain: QKV, Wo and Wd get 2 rows (a task each, 6 KB or longer pieces),
  // the LM head 4 (12 KB pieces).
  // 4-bit rows: at most four rows a task in all (NMAT x RT code registers)
  const int rt_max = q4 ? 4 / nmat : (sc.BT <= 8 ? 4 : 2);
  const int target_bytes = tu.piece_bytes > 0 ? tu.piece_bytes : 6144;
  int RT = rt_max;
  if (tu.force_rt == 1 || tu.force_rt == 2 || tu.force_rt == 4) {
    RT = tu.force_rt < rt_max ? tu.force_rt : rt_max;
  } else {
    auto load = [&](int rt) {
      const double rows = (double)((row_groups(p, rt) + warps_total - 1) / warps_total) * rt;
      const double smem = 0.18 * (1.0 + (double)sc.BT / rt);
      return rows * (smem > 1.0 ? smem : 1.0);
    };
    double best = load(1);
    for (int rt = 2; rt <= rt_max; rt *= 2) best = load(rt) < best ? load(rt) : best;
    // candidates whose row groups cover half the warps without a K split
    // first: a split's partial sums and ticket cost an op about 2 us (the
    // 768 x 768 LayerNorm block at batch 16: 1 row per task and no split,
    // 811 vs 1009 us per 72-block chain)
    const bool allow_split = force_S == 0 && tu.force_ksplit == 0;
    bool any_unsplit = false;
    for (int rt = 1; rt <= rt_max; rt *= 2)
      if (load(rt) <= best * 1.1 && row_groups(p, rt) >= warps_total / 2) any_unsplit = true;
    int pick = 0, pick_whole = 0;
    for (int rt = 1; rt <= rt_max; rt *= 2) {
      if (load(rt) > best * 1.1) continue;
      if (allow_split && any_unsplit && row_groups(p, rt) < warps_total / 2) continue;
      pick = rt;
      if ((long)nmat * rt * row_b <= target_bytes) pick_whole = rt;
    }
    RT = pick_whole ? pick_whole : pick;
  }
  sc.RT = RT;
  const int RG = row_groups(p, RT);
  sc.RG = RG;

  auto valid_split = [&](int S) { return S >= 1 && K % (8 * S) == 0; };
  auto xs_fits = [&](int S) { return (long)sc.BT * (K / S) * 2 <= kXsMaxCC; };
  int S = 1;
  if (q4) {
    // 4-bit rows are not split along K (a split would have to start on a
    // super-group); the activations of the full K stay in shared memory
  } else if (force_S > 0) {
    S = force_S;
  } else if (force_S == 0) {
    if (tu.force_ksplit > 0) {
      S = tu.force_ksplit;
    } else if (RG < warps_total / 2) {
      // skinny: split K until the tasks cover about half of the warps,
      // keeping at least 256 columns (one chunk per lane) per split
      for (int s = 2; s <= 16; ++s) {
        if (!valid_split(s)) continue;
        if (K / s < 256) break;
        S = s;
        if (RG * s >= warps_total / 2) break;
      }
    }
  }
  if (!valid_split(S)) {
    snprintf(why, why_len, "K=%d cannot be split %d ways into multiples of 8", K, S);
    return false;
  }
  if (!xs_fits(S)) {
    if (force_S < 0 || q4) {
      snprintf(why, why_len,
               "B=%d x K=%d activations exceed shared memory; pass a workspace", p.B, K);
      return false;
    }
    int s2 = S;
    while (s2 <= 64 && !(valid_split(s2) && xs_fits(s2))) ++s2;
    if (s2 > 64) {
      snprintf(why, why_len, "no K split makes B=%d x K=%d fit", p.B, K);
      return false;
    }
    S = s2;
  }
  if (p.epilogue == EPI_ARGMAX && S != 1) {
    snprintf(why, why_len, "argmax epilogue needs an unsplit K (B=%d, K=%d)", p.B, K);
    return false;
  }
  sc.S = S;
  sc.KS = K / S;

  // pieces: about piece_bytes each, evenly sized, multiples of 8 columns
  // (4-bit rows: of 512 columns, whole super-groups)
  const int pc_unit = q4 ? kQ4Super : 8;
  auto piece_row_bytes = [&](int pc_cols) { return q4 ? q4_prefix(pc_cols) : pc_cols * 2; };
  int pc = q4 ? target_bytes / (nmat * RT * kQ4SuperBytes) * kQ4Super
              : target_bytes / (nmat * RT * 2);
  pc = pc < (q4 ? kQ4Super : 256) ? (q4 ? kQ4Super : 256) : pc;
  if (pc >= sc.KS) {
    sc.PC = sc.KS;
    sc.NP = 1;
  } else {
    sc.NP = (sc.KS + pc - 1) / pc;
    sc.PC = align_up((sc.KS + sc.NP - 1) / sc.NP, pc_unit);
    sc.NP = (sc.KS + sc.PC - 1) / sc.PC;
  }
  sc.piece_bytes = align_up(nmat * RT * piece_row_bytes(sc.PC), 128);

  int off = 0;
  sc.off_bar = off;
  off += kWarps * kMaxStages * 8;
  sc.off_flags = off;
  off += 128;
  sc.off_stats = off;
  off += align_up(sc.BT * 2 * 4, 16);
  sc.off_red = off;
  off += align_up((kWarps + 1) * sc.BT * 4, 16);
  sc.off_arg = off;
  off += kWarps * 32 * 8;
  sc.off_xs = align_up(off, 128);
  off = sc.off_xs + align_up(sc.BT * sc.KS * 2, 128);
  if (q4) {
    sc.off_xsum = off;
    off += align_up(sc.BT * (sc.KS / 16) * 4, 128);
  }
  sc.off_ring = align_up(off, 128);
  // 4-bit rows: pieces are 3.76 times smaller for the same rows, so the ring
  // takes the shared memory there is, less 4 KB for the residual rows
  // (measured on the 4-bit chain: the LM head 87 -> 55 us, gate/up 11.5 ->
  // 9.2 us)
  int ring_budget =
      tu.ring_bytes > 0 ? tu.ring_bytes : (q4 ? smem_cap - sc.off_ring - 4096 : 96 * 1024);
  if (sc.off_ring + ring_budget > smem_cap) ring_budget = smem_cap - sc.off_ring;
  int NSW = ring_budget / (kWarps * sc.piece_bytes);
  if (NSW > kMaxStages) NSW = kMaxStages;
  if (NSW < 2) {
    if (sc.off_ring + 2 * kWarps * sc.piece_bytes > smem_cap) {
      // smaller pieces, so that two stages per warp fit beside the activations
      int pc_fit =
          q4 ? (smem_cap - sc.off_ring) / (2 * kWarps) / (nmat * RT * kQ4SuperBytes) * kQ4Super
             : ((smem_cap - sc.off_ring) / (2 * kWarps) / (nmat * RT * 2)) & ~7;
      // each piece is rounded up to 128 bytes: shrink until that still fits
      while (pc_fit >= pc_unit &&
             sc.off_ring + 2 * kWarps * align_up(nmat * RT * piece_row_bytes(pc_fit), 128) >
                 smem_cap)
        pc_fit -= pc_unit;
      if (pc_fit < pc_unit) {
        snprintf(why, why_len, "no two ring stages per warp fit beside %d bytes of activations",
                 sc.BT * sc.KS * 2);
        return false;
      }
      sc.NP = (sc.KS + pc_fit - 1) / pc_fit;
      sc.PC = align_up((sc.KS + sc.NP - 1) / sc.NP, pc_unit);
      sc.NP = (sc.KS + sc.PC - 1) / sc.PC;
      sc.piece_bytes = align_up(nmat * RT * piece_row_bytes(sc.PC), 128);
    }
    NSW = 2;
  }
  sc.NSW = NSW;
  sc.smem_bytes = sc.off_ring + kWarps * NSW * sc.piece_bytes;
  if (sc.smem_bytes > smem_cap) {
    snprintf(why, why_len, "no schedule fits shared memory (K=%d, B=%d, %d matrices)", K, p.B,
             nmat);
    return false;
  }
  int Gs = grid_target / S;
  if (Gs < 1) Gs = 1;
  if (Gs > RG) Gs = RG;
  if ((unsigned long long)Gs * (unsigned long long)RG >= (1ull << 32)) {
    snprintf(why, why_len, "%d row groups over %d CTAs exceed the 32-bit row arithmetic", RG, Gs);
    return false;
  }
  sc.Gs = Gs;
  sc.grid = S * Gs;
  // residual epilogues: the CTA's rows of the residual input are read into
  // shared memory while the activations are staged, off the epilogue's path
  sc.off_res = 0;
  sc.res_rows = 0;
  if (p.epilogue == EPI_RESID && p.nseg == 1) {
    const int rows = (RG + Gs - 1) / Gs * RT;
    const int off_res = align_up(sc.smem_bytes, 16);
    if (off_res + rows * sc.BT * 4 <= smem_cap) {
      sc.off_res = off_res;
      sc.res_rows = rows;
      sc.smem_bytes = off_res + rows * sc.BT * 4;
    }
  }
  p.sc = sc;
  p.M_total = 0;
  for (int s = 0; s < p.nseg; ++s) p.M_total += p.seg[s].M;
  return true;
}

// Choose the schedule.  force_S > 0 fixes the K split; force_S == 0 lets the
// heuristic split skinny shapes; force_S < 0 forbids splitting.  The tensor-
// core kernels first where they apply (4-bit rows: at batch 2-4); else the
// CUDA-core one, with two CTAs per SM for 4-bit rows at batch 1 when its
// registers and shared memory allow, else one.  Measured on the 4-bit decode
// chain at batch 1: one CTA's eight warps leave the SM waiting on copies
// (gate/up 10.3 -> 7.1 us a launch, the LM head on CUDA cores 40.5 us against
// 52.5 on tensor cores; the step 682 -> 567 us); three CTAs lose again (619
// us), and so do two at batch 4 (1074 -> 1147 us) and for bf16 rows (637 ->
// 691 us at batch 1).
bool plan_gemv(GemvParams& p, int force_S, char* why, size_t why_len) {
  const Tuning& tu = tuning();
  const int nsm = device_sm_count();
  const int grid_target = tu.grid_cap > 0 ? tu.grid_cap : nsm;
  const bool q4 = p.wfmt == WF_Q4;
  if (!q4 && tu.mma && tu.forms && plan_gemv_mma(p, force_S, grid_target)) return true;
  const bool q4_mma = tu.q4_mma == 2 || (tu.q4_mma == 1 && p.B > 1);
  if (q4 && q4_mma && tu.forms && plan_gemv_q4mma(p, grid_target)) return true;
  const int cps = tu.ctas_per_sm > 0 ? tu.ctas_per_sm : (q4 && batch_template(p.B) == 1 ? 2 : 1);
  for (int c = cps; c > 1; --c) {
    GemvParams t = p;
    if (plan_gemv_cc(t, force_S, c, why, why_len) && resident_ctas(t) >= c) {
      p = t;
      return true;
    }
  }
  return plan_gemv_cc(p, force_S, 1, why, why_len);
}

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

size_t workspace_layout(const GemvParams& p, size_t* off_tickets, size_t* off_part,
                        size_t* off_argv, size_t* off_argi, size_t* off_argt) {
  size_t off = 0;
  size_t t = 0, pt = 0, av = 0, ai = 0, at = 0;
  if (p.sc.S > 1) {
    t = off;
    off = align256(off + (size_t)p.sc.RG * 4);
    pt = off;
    off = align256(off + (size_t)p.sc.S * p.nmat * p.B * p.M_total * 4);
  }
  if (p.epilogue == EPI_ARGMAX) {
    av = off;
    off = align256(off + (size_t)p.sc.grid * p.B * 4);
    ai = off;
    off = align256(off + (size_t)p.sc.grid * p.B * 4);
    at = off;
    off = align256(off + 4);
  }
  if (off_tickets) *off_tickets = t;
  if (off_part) *off_part = pt;
  if (off_argv) *off_argv = av;
  if (off_argi) *off_argi = ai;
  if (off_argt) *off_argt = at;
  return off;
}

bool bind_workspace(GemvParams& p, void* ws, size_t ws_bytes) {
  size_t t, pt, av, ai, at;
  const size_t need = workspace_layout(p, &t, &pt, &av, &ai, &at);
  if (need == 0) return true;
  if (!ws || ws_bytes < need) return false;
  char* base = static_cast<char*>(ws);
  if (p.sc.S > 1) {
    p.tickets = reinterpret_cast<unsigned*>(base + t);
    p.part = reinterpret_cast<float*>(base + pt);
  }
  if (p.epilogue == EPI_ARGMAX) {
    p.arg_val = reinterpret_cast<float*>(base + av);
    p.arg_idx = reinterpret_cast<int*>(base + ai);
    p.arg_ticket = reinterpret_cast<unsigned*>(base + at);
  }
  return true;
}

// The kernel of a planned launch: the tensor-core one of its chain form when
// planned for it, else the CUDA-core one of its chain form where one is built
// for its batch tile, else the general one.
static GemvKernel pick_kernel(const GemvParams& p) {
  const int BT = p.sc.BT, nmat = p.nmat, RT = p.sc.RT;
  if (p.sc.mma) return p.wfmt == WF_Q4 ? pick_kernel_q4mma(nmat, p.sc.form)
                                       : pick_kernel_mma(BT, nmat, p.sc.form);
  const int F = tuning().forms ? kernel_form(p) : F_ANY;
  if (p.wfmt == WF_Q4) {
    GemvKernel k = F != F_ANY ? pick_kernel_q4(BT, nmat, RT, F) : nullptr;
    return k ? k : pick_kernel_q4(BT, nmat, RT, F_ANY);
  }
  if (F != F_ANY) {
    GemvKernel k = BT == 1   ? pick_form_b1(BT, nmat, RT, F)
                   : BT <= 4 ? pick_form_b24(BT, nmat, RT, F)
                   : BT == 8 ? pick_form_b8(BT, nmat, RT, F)
                             : pick_form_b16(BT, nmat, RT, F);
    if (k) return k;
  }
  if (BT <= 2) return pick_kernel_b12(BT, nmat, RT);
  if (BT == 4) return pick_kernel_b4(BT, nmat, RT);
  if (BT == 8) return pick_kernel_b816(BT, nmat, RT);
  return pick_kernel_b16(BT, nmat, RT);
}

// The dynamic shared-memory limit of a kernel, raised once per device (a set
// of (device, kernel) pairs: the library holds a few hundred instantiations).
static bool ensure_smem_attr(GemvKernel k) {
  static std::mutex mu;
  static std::set<std::pair<int, uintptr_t>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(mu);
  const std::pair<int, uintptr_t> key(dev, (uintptr_t)k);
  if (done.count(key)) return true;
  if (cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemMax) != cudaSuccess)
    return false;
  done.insert(key);
  return true;
}

// CTAs of a planned launch that one SM holds at once, by the kernel's
// registers and the plan's shared memory (the occupancy calculator); with no
// device to ask, by shared memory alone.
static int resident_ctas(const GemvParams& p) {
  GemvKernel k = pick_kernel(p);
  if (!k) return 0;
  int n = 0;
  if (ensure_smem_attr(k) && cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, k, kThreads, p.sc.smem_bytes) == cudaSuccess)
    return n;
  cudaGetLastError();
  return smem_per_sm() / (p.sc.smem_bytes + kSmemReserved);
}

bool prepare_gemv(const GemvParams& p) {
  GemvKernel k = pick_kernel(p);
  return k && ensure_smem_attr(k);
}

cudaError_t launch_gemv(const GemvParams& p, cudaStream_t stream, bool pdl) {
  GemvKernel k = pick_kernel(p);
  if (!k) return cudaErrorInvalidValue;
  if (!ensure_smem_attr(k)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(p.sc.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.sc.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, p);
}

cudaError_t launch_quantize_q4(const void* W, void* out, int M, int K, cudaStream_t st);

void init_gemv_params(GemvParams& p, int K, int B) {
  memset(&p, 0, sizeof p);
  p.K = K;
  p.B = B;
  p.nmat = 1;
  p.err = device_error_ptr();
  p.timeout_ns = tuning().timeout_ns;
  p.evict_first = tuning().evict_first;
}

}  // namespace ws

// ---------------------------------------------------------------------------
// C ABI: GEMV family
// ---------------------------------------------------------------------------
using namespace ws;

static bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

static ws_status check_common(int M, int K, int B) {
  if (M <= 0 || K <= 0 || K % 8 != 0 || B < 1 || B > kMaxBatch) {
    set_error("bad shape M=%d K=%d B=%d (need M>0, K>0, K%%8==0, 1<=B<=16)", M, K, B);
    return WS_ERR_SHAPE;
  }
  return WS_OK;
}

static ws_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* q : ptrs) {
    if (!q) {
      set_error("null device pointer");
      return WS_ERR_ARG;
    }
    if (!aligned16(q)) {
      set_error("device pointer %p is not 16-byte aligned", q);
      return WS_ERR_ALIGN;
    }
  }
  return WS_OK;
}

// Plan with a workspace if one is given (split allowed), else without; bind
// the workspace and launch.
static ws_status plan_bind_launch(GemvParams& p, void* ws, size_t ws_bytes, cudaStream_t st,
                                  bool allow_split = true) {
  char why[256];
  const bool have_ws = ws != nullptr && ws_bytes > 0;
  if (ws && !aligned16(ws)) {
    set_error("workspace not 16-byte aligned");
    return WS_ERR_ALIGN;
  }
  if (!plan_gemv(p, (have_ws && allow_split) ? 0 : -1, why, sizeof why)) {
    set_error("%s", why);
    return have_ws ? WS_ERR_SHAPE : WS_ERR_ARG;
  }
  if (!bind_workspace(p, ws, ws_bytes)) {
    GemvParams q = p;
    if (p.sc.S > 1 && plan_gemv(q, -1, why, sizeof why) && bind_workspace(q, ws, ws_bytes)) {
      p = q;
    } else {
      set_error("workspace too small: need %zu bytes, got %zu",
                workspace_layout(p, nullptr, nullptr, nullptr, nullptr, nullptr), ws_bytes);
      return WS_ERR_ARG;
    }
  }
  const cudaError_t e = launch_gemv(p, st, tuning().launch_pdl != 0);
  if (e != cudaSuccess) {
    set_error("launch failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

extern "C" {

const char* ws_last_error(void) { return g_msg; }

const char* ws_version(void) { return "wsgemv 0.1 (sm_103a)"; }

ws_status ws_gemv_bf16(const void* W, const void* x, float* y, int M, int K, int B,
                       void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  ws_status s = check_common(M, K, B);
  if (s) return s;
  if ((s = check_ptrs({W, x, y}))) return s;
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.seg[0].W0 = static_cast<const uint16_t*>(W);
  p.seg[0].out = y;
  p.seg[0].M = M;
  p.x = x;
  p.x_dtype = DT_BF16;
  p.prologue = PRO_NONE;
  p.epilogue = EPI_F32;
  return plan_bind_launch(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

size_t ws_q4_row_bytes(int K) {
  if (K <= 0 || K % kQ4Group) return 0;
  return (size_t)q4_prefix(K);
}

ws_status ws_quantize_q4(const void* W, void* Wq, int M, int K, ws_stream_t stream) {
  if (M <= 0 || K <= 0 || K % kQ4Group) {
    set_error("bad shape M=%d K=%d (need M>0 and K a positive multiple of 128)", M, K);
    return WS_ERR_SHAPE;
  }
  ws_status s = check_ptrs({W, Wq});
  if (s) return s;
  const cudaError_t e = launch_quantize_q4(W, Wq, M, K, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    set_error("quantize failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

ws_status ws_gemv_q4(const void* Wq, const void* x, float* y, int M, int K, int B,
                     void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  ws_status s = check_common(M, K, B);
  if (s) return s;
  if (K % kQ4Group || B > 4) {
    set_error("4-bit weights: K a multiple of 128 and B <= 4 (K=%d, B=%d)", K, B);
    return WS_ERR_SHAPE;
  }
  if ((s = check_ptrs({Wq, x, y}))) return s;
  GemvParams p;
  init_gemv_params(p, K, B);
  p.wfmt = WF_Q4;
  p.nseg = 1;
  p.seg[0].W0 = static_cast<const uint16_t*>(Wq);
  p.seg[0].out = y;
  p.seg[0].M = M;
  p.x = x;
  p.x_dtype = DT_BF16;
  p.prologue = PRO_NONE;
  p.epilogue = EPI_F32;
  return plan_bind_launch(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

ws_status ws_gemv_residual(const void* W, const void* x, const float* h_in, float* h_out, int M,
                           int K, int B, void* workspace, size_t workspace_bytes,
                           ws_stream_t stream) {
  ws_status s = check_common(M, K, B);
  if (s) return s;
  if ((s = check_ptrs({W, x, h_out}))) return s;
  if (h_in && (s = check_ptrs({h_in}))) return s;
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.seg[0].W0 = static_cast<const uint16_t*>(W);
  p.seg[0].out = h_out;
  p.seg[0].M = M;
  p.x = x;
  p.x_dtype = DT_BF16;
  p.prologue = PRO_NONE;
  p.epilogue = EPI_RESID;
  p.res_in = h_in;
  return plan_bind_launch(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

ws_status ws_rmsnorm_gemv(const void* x, int x_dtype, const void* gamma, const void* W, float* y,
                          int M, int K, int B, float eps, void* workspace,
                          size_t workspace_bytes, ws_stream_t stream) {
  ws_status s = check_common(M, K, B);
  if (s) return s;
  if ((s = check_ptrs({x, gamma, W, y}))) return s;
  if (x_dtype != WS_DTYPE_F32 && x_dtype != WS_DTYPE_BF16) {
    set_error("x_dtype must be WS_DTYPE_F32 or WS_DTYPE_BF16");
    return WS_ERR_ARG;
  }
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.seg[0].W0 = static_cast<const uint16_t*>(W);
  p.seg[0].out = y;
  p.seg[0].M = M;
  p.x = x;
  p.x_dtype = x_dtype;
  p.prologue = PRO_RMSNORM;
  p.gamma = static_cast<const uint16_t*>(gamma);
  p.eps = eps;
  p.epilogue = EPI_F32;
  return plan_bind_launch(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

ws_status ws_qkv_gemv(const void* x, int x_dtype, const void* gamma, const void* Wq,
                      const void* Wk, const void* Wv, float* q, float* k, float* v, int Mq,
                      int Mkv, int K, int B, float eps, void* workspace, size_t workspace_bytes,
                      ws_stream_t stream) {
  ws_status s = check_common(Mq, K, B);
  if (s) return s;
  if ((s = check_common(Mkv, K, B))) return s;
  if ((s = check_ptrs({x, gamma, Wq, Wk, Wv, q, k, v}))) return s;
  if (x_dtype != WS_DTYPE_F32 && x_dtype != WS_DTYPE_BF16) {
    set_error("x_dtype must be WS_DTYPE_F32 or WS_DTYPE_BF16");
    return WS_ERR_ARG;
  }
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 3;
  const void* Ws[3] = {Wq, Wk, Wv};
  float* outs[3] = {q, k, v};
  const int Ms[3] = {Mq, Mkv, Mkv};
  int base = 0;
  for (int i = 0; i < 3; ++i) {
    p.seg[i].W0 = static_cast<const uint16_t*>(Ws[i]);
    p.seg[i].out = outs[i];
    p.seg[i].M = Ms[i];
    p.seg[i].row_base = base;
    base += Ms[i];
  }
  p.x = x;
  p.x_dtype = x_dtype;
  p.prologue = PRO_RMSNORM;
  p.gamma = static_cast<const uint16_t*>(gamma);
  p.eps = eps;
  p.epilogue = EPI_F32;
  return plan_bind_launch(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

ws_status ws_swiglu_gemv(const void* x, int x_dtype, const void* gamma, const void* Wg,
                         const void* Wu, void* sbuf, int M, int K, int B, float eps,
                         void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  ws_status s = check_common(M, K, B);
  if (s) return s;
  if ((s = check_ptrs({x, Wg, Wu, sbuf}))) return s;
  if (gamma && (s = check_ptrs({gamma}))) return s;
  if (x_dtype != WS_DTYPE_F32 && x_dtype != WS_DTYPE_BF16) {
    set_error("x_dtype must be WS_DTYPE_F32 or WS_DTYPE_BF16");
    return WS_ERR_ARG;
  }
  if (!gamma && x_dtype != WS_DTYPE_BF16) {
    set_error("without a norm the SwiGLU input must be bf16");
    return WS_ERR_ARG;
  }
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.nmat = 2;
  p.seg[0].W0 = static_cast<const uint16_t*>(Wg);
  p.seg[0].W1 = static_cast<const uint16_t*>(Wu);
  p.seg[0].out = sbuf;
  p.seg[0].M = M;
  p.x = x;
  p.x_dtype = x_dtype;
  p.prologue = gamma ? PRO_RMSNORM : PRO_NONE;
  p.gamma = static_cast<const uint16_t*>(gamma);
  p.eps = eps;
  p.epilogue = EPI_SWIGLU;
  return plan_bind_launch(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

ws_status ws_ln_gemv_gelu(const void* x, const void* gamma, const void* beta, const void* W,
                          const void* bias, void* z, int M, int K, int B, float eps,
                          void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  ws_status s = check_common(M, K, B);
  if (s) return s;
  if ((s = check_ptrs({x, gamma, beta, W, bias, z}))) return s;
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.seg[0].W0 = static_cast<const uint16_t*>(W);
  p.seg[0].out = z;
  p.seg[0].M = M;
  p.x = x;
  p.x_dtype = DT_BF16;
  p.prologue = PRO_LAYERNORM;
  p.gamma = static_cast<const uint16_t*>(gamma);
  p.beta = static_cast<const uint16_t*>(beta);
  p.eps = eps;
  p.epilogue = EPI_BIAS_GELU;
  p.bias = static_cast<const uint16_t*>(bias);
  return plan_bind_launch(p, workspace, workspace_bytes, (cudaStream_t)stream);
}

ws_status ws_lmhead_argmax(const void* h, int h_dtype, const void* gamma, const void* W,
                           int32_t* idx, float* logits, int V, int K, int B, float eps,
                           void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  ws_status s = check_common(V, K, B);
  if (s) return s;
  if ((s = check_ptrs({h, gamma, W, idx, workspace}))) return s;
  if (logits && (s = check_ptrs({logits}))) return s;
  if (h_dtype != WS_DTYPE_F32 && h_dtype != WS_DTYPE_BF16) {
    set_error("h_dtype must be WS_DTYPE_F32 or WS_DTYPE_BF16");
    return WS_ERR_ARG;
  }
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.seg[0].W0 = static_cast<const uint16_t*>(W);
  p.seg[0].out = logits;
  p.seg[0].M = V;
  p.x = h;
  p.x_dtype = h_dtype;
  p.prologue = PRO_RMSNORM;
  p.gamma = static_cast<const uint16_t*>(gamma);
  p.eps = eps;
  p.epilogue = EPI_ARGMAX;
  p.argmax_idx = idx;
  p.logits = logits;
  return plan_bind_launch(p, workspace, workspace_bytes, (cudaStream_t)stream, false);
}

// variant: 0 plain bf16 x; 1 RMSNorm of fp32 x; 2 bf16 x with a residual
// epilogue (the entry points an op id covers plan differently: the tensor-
// core schedule takes the chain forms only)
static bool plan_for_op(int op, int M, int K, int B, GemvParams& p, int variant = 0) {
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.seg[0].M = M;
  p.epilogue = EPI_F32;
  p.x_dtype = DT_BF16;
  if (variant == 1) {
    p.prologue = PRO_RMSNORM;
    p.x_dtype = DT_F32;
  } else if (variant == 2) {
    p.epilogue = EPI_RESID;
  }
  if (op == WS_OP_SWIGLU_GEMV) {
    p.nmat = 2;
    p.epilogue = EPI_SWIGLU;
  } else if (op == WS_OP_LMHEAD_ARGMAX) {
    p.epilogue = EPI_ARGMAX;
  } else if (op != WS_OP_GEMV && op != WS_OP_QKV_GEMV) {
    return false;
  }
  if (variant == 2 && op != WS_OP_GEMV) {
    return false;
  }
  char why[256];
  return plan_gemv(p, op == WS_OP_LMHEAD_ARGMAX ? -1 : 0, why, sizeof why);
}

size_t ws_workspace_bytes(int op, int M, int K, int B) {
  if (op == WS_OP_ARGMAX_ROWS) return argmax_rows_workspace(M, K);
  if (M <= 0 || K <= 0 || K % 8 != 0 || B < 1 || B > kMaxBatch) return 0;
  // the largest workspace of the schedules the op id's entry points can take
  size_t need = 0;
  bool any = false;
  for (int variant = 0; variant < 3; ++variant) {
    GemvParams p;
    if (!plan_for_op(op, M, K, B, p, variant)) continue;
    any = true;
    const size_t w = workspace_layout(p, nullptr, nullptr, nullptr, nullptr, nullptr);
    need = w > need ? w : need;
  }
  return any ? need : 0;
}

int ws_device_error(int reset) {
  int* ptr = device_error_ptr();
  if (!ptr) return -1;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  int v = 0;
  if (cudaMemcpy(&v, ptr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  if (reset && v) {
    const int z = 0;
    if (cudaMemcpy(ptr, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) return -1;
  }
  return v;
}

void ws_get_tuning(ws_tuning* t) {
  if (!t) return;
  const Tuning& tu = tuning();
  t->ring_bytes = tu.ring_bytes;
  t->grid_cap = tu.grid_cap;
  t->force_ksplit = tu.force_ksplit;
  t->force_rt = tu.force_rt;
  t->evict_first = tu.evict_first;
  t->piece_bytes = tu.piece_bytes;
  t->timeout_ns = tu.timeout_ns;
  t->l2_ahead = tu.l2_ahead;
  t->forms = tu.forms;
  t->launch_pdl = tu.launch_pdl;
  t->mma = tu.mma;
  t->ctas_per_sm = tu.ctas_per_sm;
  t->q4_mma = tu.q4_mma;
}

ws_status ws_set_tuning(const ws_tuning* t) {
  if (!t || t->ring_bytes < 0 || t->ring_bytes > kSmemMax || t->grid_cap < 0 ||
      t->force_ksplit < 0 || t->force_rt < 0 || t->force_rt == 3 || t->force_rt > 4 ||
      t->piece_bytes < 0 ||
      t->piece_bytes > 64 * 1024 || t->timeout_ns == 0 || t->l2_ahead < 0 ||
      t->l2_ahead > 64 || t->forms < 0 || t->forms > 1 || t->launch_pdl < 0 ||
      t->launch_pdl > 1 || t->mma < 0 || t->mma > 1 || t->ctas_per_sm < 0 ||
      t->ctas_per_sm > 3 || t->q4_mma < 0 || t->q4_mma > 2) {
    set_error("bad tuning values");
    return WS_ERR_ARG;
  }
  Tuning& tu = tuning();
  tu.ring_bytes = t->ring_bytes;
  tu.grid_cap = t->grid_cap;
  tu.force_ksplit = t->force_ksplit;
  tu.force_rt = t->force_rt;
  tu.evict_first = t->evict_first;
  tu.piece_bytes = t->piece_bytes;
  tu.timeout_ns = t->timeout_ns;
  tu.l2_ahead = t->l2_ahead;
  tu.forms = t->forms;
  tu.launch_pdl = t->launch_pdl;
  tu.mma = t->mma;
  tu.ctas_per_sm = t->ctas_per_sm;
  tu.q4_mma = t->q4_mma;
  return WS_OK;
}

ws_status ws_gemv_plan(int M_total, int K, int B, int nmat, int prologue_kind, int epilogue_kind,
                       int allow_split, ws_gemv_schedule* out) {
  ws_status s = check_common(M_total, K, B);
  if (s) return s;
  if (!out || (nmat != 1 && nmat != 2)) {
    set_error("bad arguments");
    return WS_ERR_ARG;
  }
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.nmat = nmat;
  p.seg[0].M = M_total;
  p.prologue = prologue_kind;
  p.epilogue = epilogue_kind;
  char why[256];
  if (!plan_gemv(p, allow_split ? 0 : -1, why, sizeof why)) {
    set_error("%s", why);
    return WS_ERR_SHAPE;
  }
  const Sched& sc = p.sc;
  out->RT = sc.RT;
  out->S = sc.S;
  out->KS = sc.KS;
  out->PC = sc.PC;
  out->NP = sc.NP;
  out->NSW = sc.NSW;
  out->piece_bytes = sc.piece_bytes;
  out->RG = sc.RG;
  out->grid = sc.grid;
  out->smem_bytes = sc.smem_bytes;
  return WS_OK;
}

long ws_debug_gemv_copies_q4(int M, int K, int B, int nmat, int cta, int mma,
                             long long* triples, long max_triples, ws_gemv_schedule* out) {
  if (check_common(M, K, B) != WS_OK || K % kQ4Group || (nmat != 1 && nmat != 2)) return -1;
  GemvParams p;
  init_gemv_params(p, K, B);
  p.wfmt = WF_Q4;
  p.nseg = 1;
  p.nmat = nmat;
  p.seg[0].M = M;
  p.epilogue = nmat == 2 ? EPI_SWIGLU : EPI_F32;
  if (mma) {  // the chain forms the tensor-core kernel takes
    p.x_dtype = nmat == 2 ? DT_F32 : DT_BF16;
    p.prologue = nmat == 2 ? PRO_RMSNORM : PRO_NONE;
  }
  char why[256];
  if (!plan_gemv(p, -1, why, sizeof why)) return -1;
  const Sched& sc = p.sc;
  if (sc.mma != (mma ? 1 : 0)) return -1;
  if (out) {
    out->RT = sc.RT;
    out->S = sc.S;
    out->KS = sc.KS;
    out->PC = sc.PC;
    out->NP = sc.NP;
    out->NSW = sc.NSW;
    out->piece_bytes = sc.piece_bytes;
    out->RG = sc.RG;
    out->grid = sc.grid;
    out->smem_bytes = sc.smem_bytes;
  }
  if (cta < 0 || cta >= sc.grid) return -1;
  int ks, rg0, rg1;
  cta_range(sc, cta, ks, rg0, rg1);
  const int k0 = ks * sc.KS;
  const long long warp_ring = (long long)sc.NSW * sc.piece_bytes;
  const long long rb = q4_prefix(K);
  long n = 0;
  // the same order and arithmetic as issue_piece's 4-bit path
  for (int w = 0; w < kWarps; ++w) {
    const int npw = warp_tasks(rg0, rg1, w) * sc.NP;
    for (int q = 0; q < npw; ++q) {
      const int ti = q / sc.NP;
      const int j = q - ti * sc.NP;
      int seg, rgl;
      decode_rg(p, rg0 + w + ti * kWarps, seg, rgl);
      const int row0 = rgl * sc.RT;
      const int rows = (sc.RT < M - row0) ? sc.RT : M - row0;
      const int c0 = k0 + j * sc.PC;
      const int len = (sc.PC < sc.KS - j * sc.PC) ? sc.PC : sc.KS - j * sc.PC;
      const int src0 = q4_prefix(c0), nb = q4_prefix(c0 + len) - src0;
      const int pst = sc.mma ? sc.prow : q4_prefix(sc.PC);
      const long long dst0 = w * warp_ring + (long long)(q % sc.NSW) * sc.piece_bytes;
      for (int mat = 0; mat < nmat; ++mat)
        for (int r = 0; r < rows; ++r) {
          if (triples && n < max_triples) {
            triples[3 * n] = (long long)mat * M * rb + (long long)(row0 + r) * rb + src0;
            triples[3 * n + 1] = dst0 + ((long long)mat * sc.RT + r) * pst;
            triples[3 * n + 2] = nb;
          }
          ++n;
        }
    }
  }
  return n;
}

long ws_debug_gemv_copies(int M, int K, int B, int nmat, int allow_split, int cta,
                          long long* triples, long max_triples) {
  if (check_common(M, K, B) != WS_OK || (nmat != 1 && nmat != 2)) return -1;
  GemvParams p;
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.nmat = nmat;
  p.seg[0].M = M;
  p.epilogue = nmat == 2 ? EPI_SWIGLU : EPI_F32;
  char why[256];
  if (!plan_gemv(p, allow_split ? 0 : -1, why, sizeof why)) return -1;
  const Sched& sc = p.sc;
  if (cta < 0 || cta >= sc.grid) return -1;
  int ks, rg0, rg1;
  cta_range(sc, cta, ks, rg0, rg1);
  const int k0 = ks * sc.KS;
  const long long warp_ring = (long long)sc.NSW * sc.piece_bytes;
  long n = 0;
  // the same order as issue_piece: warp by warp, piece by piece
  for (int w = 0; w < kWarps; ++w) {
    const int npw = warp_tasks(rg0, rg1, w) * sc.NP;
    for (int q = 0; q < npw; ++q) {
      const int ti = q / sc.NP;
      const int j = q - ti * sc.NP;
      int seg, rgl;
      decode_rg(p, rg0 + w + ti * kWarps, seg, rgl);
      const int row0 = rgl * sc.RT;
      const int rows = (sc.RT < M - row0) ? sc.RT : M - row0;
      const int c0 = k0 + j * sc.PC;
      const int len = (sc.PC < sc.KS - j * sc.PC) ? sc.PC : sc.KS - j * sc.PC;
      const long long dst0 = w * warp_ring + (long long)(q % sc.NSW) * sc.piece_bytes;
      for (int mat = 0; mat < nmat; ++mat) {
        const long long mat_off = (long long)mat * M * K * 2;
        if (len == K) {
          if (triples && n < max_triples) {
            triples[3 * n] = mat_off + (long long)row0 * K * 2;
            triples[3 * n + 1] = dst0 + (long long)mat * sc.RT * sc.PC * 2;
            triples[3 * n + 2] = (long long)rows * K * 2;
          }
          ++n;
        } else {
          for (int r = 0; r < rows; ++r) {
            if (triples && n < max_triples) {
              triples[3 * n] = mat_off + ((long long)(row0 + r) * K + c0) * 2;
              triples[3 * n + 1] = dst0 + ((long long)mat * sc.RT + r) * sc.PC * 2;
              triples[3 * n + 2] = (long long)len * 2;
            }
            ++n;
          }
        }
      }
    }
  }
  return n;
}

}  // extern "C"
