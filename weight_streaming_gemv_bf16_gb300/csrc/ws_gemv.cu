// ws_gemv.cu -- the streaming GEMV kernel, its schedule, and the GEMV-family
// entry points of the C ABI.
//
// y[b][m] = sum_k W[m][k] * x[b][k], bf16 W and x, fp32 accumulation ("One
// Token, Kernel by Kernel: A Decode Step on a Laptop GPU", Step 1, "What one
// block launches").  The design for GB300:
//  * every warp is an independent pipeline: it owns whole rows (a task of
//    RT rows, one K split), streams them from HBM through its own ring of
//    shared-memory stages with 1-D bulk async copies (cp.async.bulk, mbarrier
//    completion, L2 evict-first since each weight byte is read once), and
//    refills a stage as soon as its lanes have read it; no warp ever waits for
//    another, so one slow step does not stall the CTA;
//  * the first stages are issued before griddepcontrol.wait: weights do not
//    depend on the previous op, so inside a chain the next op's weights stream
//    in while the previous op finishes (programmatic dependent launch);
//  * lanes take 16-byte chunks of each row, unpack bf16 pairs to fp32 and
//    accumulate with FMA; at the end of a task a butterfly of warp shuffles
//    gives every lane every sum, and lane r*B+b runs the epilogue of output
//    (row r, batch b);
//  * split-K for skinny shapes: partial sums go to a workspace and the last
//    of a row group's splits (atomic ticket) adds them in split order, so the
//    result is the same whatever order the CTAs finish in; the ticket is
//    reset for the next call or graph replay ("Making small PyTorch ops
//    faster on a laptop GPU", "A full decode step is a different story": the
//    last block to finish merges and resets the ticket);
//  * the activations are normalised once per CTA (RMSNorm or LayerNorm
//    prologue, fp32, rounded once to bf16) into shared memory.
// There are no tensor cores here: at batch <= 16 this is a vector product.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "wsgemv.h"
#include "ws_common.cuh"
#include "ws_device.cuh"

namespace ws {

__device__ int g_device_error;

__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ void raise_device_error(int* err, int code) {
  if (err) atomicExch(err, code);
}

// Epilogue for one output element (segment seg, row m, batch row b).  v0 is
// the dot product with the first matrix, v1 with the second (SwiGLU up).
__device__ __forceinline__ void apply_epilogue(const GemvParams& p, int seg, int m, int b,
                                               float v0, float v1, float& best_v, int& best_i) {
  const Seg& S = p.seg[seg];
  const size_t o = (size_t)b * S.M + m;
  switch (p.epilogue) {
    case EPI_F32:
      static_cast<float*>(S.out)[o] = v0;
      break;
    case EPI_BF16:
      static_cast<__nv_bfloat16*>(S.out)[o] = __float2bfloat16_rn(v0);
      break;
    case EPI_RESID: {
      const float* src = p.res_in ? p.res_in : static_cast<const float*>(S.out);
      static_cast<float*>(S.out)[o] = src[o] + v0;
      break;
    }
    case EPI_BIAS_GELU: {
      const float t = bf16_round(v0 + __uint_as_float((uint32_t)p.bias[m] << 16));
      const float z = 0.5f * t * (1.0f + erff(t * 0.70710678118654752f));
      static_cast<__nv_bfloat16*>(S.out)[o] = __float2bfloat16_rn(z);
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

__device__ __forceinline__ float load_x(const GemvParams& p, int b, int k) {
  if (p.x_dtype == DT_F32) return static_cast<const float*>(p.x)[(size_t)b * p.K + k];
  const uint16_t h = static_cast<const uint16_t*>(p.x)[(size_t)b * p.K + k];
  return __uint_as_float((uint32_t)h << 16);
}

// Per-row statistics of the prologue over the full K: RMSNorm r = rsqrt(mean
// x^2 + eps); LayerNorm mean and rstd = rsqrt(var + eps).  One warp per row.
__device__ void prologue_stats(const GemvParams& p, float* stats, int warp, int lane) {
  if (p.prologue == PRO_NONE) return;
  for (int b = warp; b < p.B; b += kWarps) {
    if (p.prologue == PRO_RMSNORM) {
      float ss = 0.f;
      for (int k = lane; k < p.K; k += 32) {
        const float v = load_x(p, b, k);
        ss = fmaf(v, v, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) stats[2 * b] = rsqrtf(ss / (float)p.K + p.eps);
    } else {
      float s = 0.f;
      for (int k = lane; k < p.K; k += 32) s += load_x(p, b, k);
      const float mean = warp_sum(s) / (float)p.K;
      float v = 0.f;
      for (int k = lane; k < p.K; k += 32) {
        const float d = load_x(p, b, k) - mean;
        v = fmaf(d, d, v);
      }
      v = warp_sum(v) / (float)p.K;
      if (lane == 0) {
        stats[2 * b] = mean;
        stats[2 * b + 1] = rsqrtf(v + p.eps);
      }
    }
  }
}

// Stage columns [k0, k0 + KS) of the (normalised) activations as bf16 into
// shared memory, [BT][KS]; rows b >= B are zero.
template <int BT>
__device__ void stage_x(const GemvParams& p, const float* stats, uint16_t* xs, int ks, int tid) {
  const int KS = p.sc.KS;
  const int nch = KS >> 3;
  const int k0 = ks * KS;
  for (int o = tid; o < BT * nch; o += kThreads) {
    const int b = o / nch;
    const int c = o - b * nch;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (b < p.B) {
      const int k = k0 + c * 8;
      if (p.prologue == PRO_NONE && p.x_dtype == DT_BF16) {
        out = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) +
                                              (size_t)b * p.K + k);
      } else {
        float v[8];
        if (p.x_dtype == DT_F32) {
          const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x) +
                                                              (size_t)b * p.K + k);
          const float4 a = src[0], c2 = src[1];
          v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
          v[4] = c2.x; v[5] = c2.y; v[6] = c2.z; v[7] = c2.w;
        } else {
          const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) +
                                                          (size_t)b * p.K + k);
          v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
          v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
        }
        if (p.prologue == PRO_RMSNORM) {
          const float r = stats[2 * b];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            v[j] = v[j] * r * __uint_as_float((uint32_t)p.gamma[k + j] << 16);
        } else if (p.prologue == PRO_LAYERNORM) {
          const float mean = stats[2 * b], rstd = stats[2 * b + 1];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            v[j] = (v[j] - mean) * rstd * __uint_as_float((uint32_t)p.gamma[k + j] << 16) +
                   __uint_as_float((uint32_t)p.beta[k + j] << 16);
        }
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * j]));
          const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * j + 1]));
          w[j] = lo | (hi << 16);
        }
        out = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    reinterpret_cast<uint4*>(xs)[(size_t)b * nch + c] = out;
  }
}

// Issue the bulk copies of piece q of this warp's task list into its ring.
template <int NMAT, int RT>
__device__ __forceinline__ void issue_piece(const GemvParams& p, int q, int warp, int rg0, int k0,
                                            uint8_t* ring, uint64_t* full, uint64_t pol) {
  const Sched& sc = p.sc;
  const int ti = q / sc.NP;
  const int j = q - ti * sc.NP;
  int seg, rgl;
  decode_rg(p, rg0 + warp + ti * kWarps, seg, rgl);
  const Seg& S = p.seg[seg];
  const int row0 = rgl * RT;
  const int rows = min(RT, S.M - row0);
  const int c0 = k0 + j * sc.PC;
  const int len = min(sc.PC, sc.KS - j * sc.PC);
  const int slot = q % sc.NSW;
  uint8_t* dst = ring + (size_t)slot * sc.piece_bytes;
  const int K = p.K;
  mbar_arrive_expect_tx(&full[slot], (uint32_t)(NMAT * rows * len * 2));
#pragma unroll
  for (int mat = 0; mat < NMAT; ++mat) {
    const uint16_t* W = mat == 0 ? S.W0 : S.W1;
    if (len == K) {  // whole rows: one contiguous copy
      bulk_copy_g2s(dst + (size_t)mat * RT * sc.PC * 2, W + (size_t)row0 * K,
                    (uint32_t)(rows * K * 2), &full[slot], pol);
    } else {
      for (int r = 0; r < rows; ++r)
        bulk_copy_g2s(dst + ((size_t)mat * RT + r) * sc.PC * 2, W + (size_t)(row0 + r) * K + c0,
                      (uint32_t)(len * 2), &full[slot], pol);
    }
  }
}

template <int BT, int NMAT, int RT>
__global__ void __launch_bounds__(kThreads) k_stream_gemv(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Sched& sc = p.sc;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sc.off_bar) + warp * kMaxStages;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + sc.off_flags);
  float* stats = reinterpret_cast<float*>(smem + sc.off_stats);
  float* argv = reinterpret_cast<float*>(smem + sc.off_arg);
  int* argi = reinterpret_cast<int*>(argv + kWarps * 32);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + sc.off_xs);
  uint8_t* ring = smem + sc.off_ring + (size_t)warp * sc.NSW * sc.piece_bytes;

  int ks, rg0, rg1;
  cta_range(sc, blockIdx.x, ks, rg0, rg1);
  const int k0 = ks * sc.KS;
  const int npw = warp_tasks(rg0, rg1, warp) * sc.NP;  // pieces of this warp
  uint64_t pol = 0;

  if (lane == 0) {
    for (int s = 0; s < sc.NSW; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    pol = p.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
    // Weights do not depend on the previous kernel: start streaming them
    // before waiting for it.
    for (int q = 0; q < sc.NSW && q < npw; ++q)
      issue_piece<NMAT, RT>(p, q, warp, rg0, k0, ring, full, pol);
  }
  pdl_launch_dependents();
  pdl_wait();

  prologue_stats(p, stats, warp, lane);
  __syncthreads();
  stage_x<BT>(p, stats, xs, ks, tid);
  __syncthreads();

  const int nchx = sc.KS >> 3;  // chunks of x in shared memory
  const int ncp = sc.PC >> 3;   // chunk stride of one row of a piece
  const uint4* xs4 = reinterpret_cast<const uint4*>(xs);
  float best_v = -INFINITY;
  int best_i = 0x7fffffff;
  bool abort = false;
  int issued = npw < sc.NSW ? npw : sc.NSW;

  float acc[NMAT][RT][BT];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[m][r][b] = 0.f;

  for (int q = 0; q < npw; ++q) {
    const int slot = q % sc.NSW;
    const int ti = q / sc.NP;
    const int j = q - ti * sc.NP;
    const int rg = rg0 + warp + ti * kWarps;
    int seg, rgl;
    decode_rg(p, rg, seg, rgl);
    const int Mseg = p.seg[seg].M;
    const int row0 = rgl * RT;
    const int rows = min(RT, Mseg - row0);
    const int len = min(sc.PC, sc.KS - j * sc.PC);
    bool ok = abort || mbar_wait_bounded(&full[slot], (q / sc.NSW) & 1, p.timeout_ns);
    if (__any_sync(0xffffffffu, !ok) && !abort) {
      abort = true;
      if (lane == 0) raise_device_error(p.err, DERR_TIMEOUT);
    }

    const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)slot * sc.piece_bytes);
    const int xoff = (j * sc.PC) >> 3;
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
    __syncwarp();
    if (lane == 0 && !abort && issued < npw) {
      // every lane has finished reading this slot: refill it
      fence_proxy_async_smem();
      issue_piece<NMAT, RT>(p, issued, warp, rg0, k0, ring, full, pol);
      ++issued;
    }

    if (j == sc.NP - 1) {
      // task complete: sum over lanes (every lane ends with every sum)
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int b = 0; b < BT; ++b) acc[m][r][b] = warp_sum(acc[m][r][b]);
      const int rowg = p.seg[seg].row_base + row0;
      if (sc.S == 1) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int b = 0; b < BT; ++b)
            if (lane == r * BT + b && r < rows && b < p.B)
              apply_epilogue(p, seg, row0 + r, b, acc[0][r][b], acc[NMAT - 1][r][b], best_v,
                             best_i);
      } else {
        // split-K: write this split's partials; the last split of the row
        // group adds all splits in split order and runs the epilogue
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int b = 0; b < BT; ++b)
            if (lane == r * BT + b && r < rows && b < p.B) {
#pragma unroll
              for (int m = 0; m < NMAT; ++m)
                p.part[((size_t)(ks * NMAT + m) * p.B + b) * p.M_total + rowg + r] = acc[m][r][b];
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
          for (int o = lane; o < rows * p.B; o += 32) {
            const int rr = o / p.B;
            const int b = o - rr * p.B;
            float v[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
              float t = 0.f;
              for (int s = 0; s < sc.S; ++s)
                t += __ldcg(&p.part[((size_t)(s * NMAT + m) * p.B + b) * p.M_total + rowg + rr]);
              v[m] = t;
            }
            float dv = -INFINITY;
            int di = 0x7fffffff;
            apply_epilogue(p, seg, row0 + rr, b, v[0], v[NMAT - 1], dv, di);
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
  }

  if (abort && lane == 0) {
    // a wait ran out: no copy may still be landing when the CTA exits
    for (int q = issued - sc.NSW; q < issued; ++q)
      if (q >= 0) mbar_wait_bounded(&full[q % sc.NSW], (q / sc.NSW) & 1, p.timeout_ns);
  }

  if (p.epilogue == EPI_ARGMAX) {
    // per batch row: lanes r*BT + b hold a running best; combine the warps,
    // then the last CTA (ticket) combines all CTAs
    argv[warp * 32 + lane] = best_v;
    argi[warp * 32 + lane] = best_i;
    __syncthreads();
    if (tid < p.B) {
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
    if (flags[0] && tid < p.B) {
      __threadfence();
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int c = 0; c < (int)gridDim.x; ++c) {
        const float v = __ldcg(&p.arg_val[(size_t)c * p.B + tid]);
        const int ix = __ldcg(&p.arg_idx[(size_t)c * p.B + tid]);
        if (arg_better(v, ix, bv, bi)) {
          bv = v;
          bi = ix;
        }
      }
      p.argmax_idx[tid] = bi;
    }
  }
}

// ---------------------------------------------------------------------------
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
  static Tuning t = {96 * 1024, 0, 0, 0, 1, 6144, 2000000000ull};
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

static constexpr int kXsMax = 64 * 1024;
static constexpr int kSmemMax = 227 * 1024;

static int row_groups(GemvParams& p, int RT) {
  int RG = 0;
  for (int s = 0; s < p.nseg; ++s) {
    p.seg[s].rg_begin = RG;
    RG += (p.seg[s].M + RT - 1) / RT;
  }
  return RG;
}

// Choose the schedule.  force_S > 0 fixes the K split; force_S == 0 lets the
// heuristic split skinny shapes; force_S < 0 forbids splitting.
bool plan_gemv(GemvParams& p, int force_S, char* why, size_t why_len) {
  const Tuning& tu = tuning();
  const int nsm = device_sm_count();
  const int grid_target = tu.grid_cap > 0 ? tu.grid_cap : nsm;
  const int warps_total = grid_target * kWarps;
  Sched sc;
  memset(&sc, 0, sizeof sc);
  sc.BT = batch_template(p.B);
  const int K = p.K, nmat = p.nmat;

  // rows per task: 2 when the batch is small enough for the accumulators and
  // there are enough tasks to keep every warp busy, else 1
  int RT = sc.BT <= 8 ? 2 : 1;
  if (tu.force_rt == 1 || tu.force_rt == 2) RT = tu.force_rt;
  if (sc.BT > 8) RT = 1;
  if (RT == 2 && tu.force_rt == 0 && row_groups(p, 2) < 2 * warps_total) RT = 1;
  sc.RT = RT;
  const int RG = row_groups(p, RT);
  sc.RG = RG;

  auto valid_split = [&](int S) { return S >= 1 && K % (8 * S) == 0; };
  auto xs_fits = [&](int S) { return (long)sc.BT * (K / S) * 2 <= kXsMax; };
  int S = 1;
  if (force_S > 0) {
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
    if (force_S < 0) {
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
  const int target = tu.piece_bytes > 0 ? tu.piece_bytes : 6144;
  int pc = target / (nmat * RT * 2);
  pc = pc < 256 ? 256 : pc;
  if (pc >= sc.KS) {
    sc.PC = sc.KS;
    sc.NP = 1;
  } else {
    sc.NP = (sc.KS + pc - 1) / pc;
    sc.PC = align_up((sc.KS + sc.NP - 1) / sc.NP, 8);
    sc.NP = (sc.KS + sc.PC - 1) / sc.PC;
  }
  sc.piece_bytes = align_up(nmat * RT * sc.PC * 2, 128);

  int off = 0;
  sc.off_bar = off;
  off += kWarps * kMaxStages * 8;
  sc.off_flags = off;
  off += 128;
  sc.off_stats = off;
  off += align_up(sc.BT * 2 * 4, 16);
  sc.off_arg = off;
  off += kWarps * 32 * 8;
  sc.off_xs = align_up(off, 128);
  off = sc.off_xs + align_up(sc.BT * sc.KS * 2, 128);
  sc.off_ring = align_up(off, 128);
  int ring_budget = tu.ring_bytes > 0 ? tu.ring_bytes : 96 * 1024;
  if (sc.off_ring + ring_budget > kSmemMax) ring_budget = kSmemMax - sc.off_ring;
  int NSW = ring_budget / (kWarps * sc.piece_bytes);
  if (NSW > kMaxStages) NSW = kMaxStages;
  if (NSW < 2) {
    if (sc.off_ring + 2 * kWarps * sc.piece_bytes <= kSmemMax) {
      NSW = 2;
    } else {
      snprintf(why, why_len, "pieces of %d bytes do not fit twice per warp", sc.piece_bytes);
      return false;
    }
  }
  sc.NSW = NSW;
  sc.smem_bytes = sc.off_ring + kWarps * NSW * sc.piece_bytes;
  int Gs = grid_target / S;
  if (Gs < 1) Gs = 1;
  if (Gs > RG) Gs = RG;
  sc.Gs = Gs;
  sc.grid = S * Gs;
  p.sc = sc;
  p.M_total = 0;
  for (int s = 0; s < p.nseg; ++s) p.M_total += p.seg[s].M;
  return true;
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

typedef void (*GemvKernel)(const GemvParams);

static GemvKernel pick_kernel(int BT, int nmat, int RT) {
#define WS_PICK2(bt)                                                                  \
  case bt:                                                                            \
    if (RT == 2)                                                                      \
      return nmat == 2 ? (GemvKernel)k_stream_gemv<bt, 2, 2>                          \
                       : (GemvKernel)k_stream_gemv<bt, 1, 2>;                         \
    return nmat == 2 ? (GemvKernel)k_stream_gemv<bt, 2, 1> : (GemvKernel)k_stream_gemv<bt, 1, 1>;
  switch (BT) {
    WS_PICK2(1)
    WS_PICK2(2)
    WS_PICK2(4)
    WS_PICK2(8)
    case 16:
      if (RT != 1) return nullptr;
      return nmat == 2 ? (GemvKernel)k_stream_gemv<16, 2, 1> : (GemvKernel)k_stream_gemv<16, 1, 1>;
    default:
      return nullptr;
  }
#undef WS_PICK2
}

static bool ensure_smem_attr(GemvKernel k) {
  static std::mutex mu;
  static unsigned long long done[64][32] = {{0}};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < 32; ++i) {
    if (done[dev][i] == (unsigned long long)(uintptr_t)k) return true;
    if (done[dev][i] == 0) {
      if (cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemMax) != cudaSuccess)
        return false;
      done[dev][i] = (unsigned long long)(uintptr_t)k;
      return true;
    }
  }
  return false;
}

bool prepare_gemv(const GemvParams& p) {
  GemvKernel k = pick_kernel(p.sc.BT, p.nmat, p.sc.RT);
  return k && ensure_smem_attr(k);
}

cudaError_t launch_gemv(const GemvParams& p, cudaStream_t stream, bool pdl) {
  GemvKernel k = pick_kernel(p.sc.BT, p.nmat, p.sc.RT);
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
  const cudaError_t e = launch_gemv(p, st, false);
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

static bool plan_for_op(int op, int M, int K, int B, GemvParams& p) {
  init_gemv_params(p, K, B);
  p.nseg = 1;
  p.seg[0].M = M;
  p.epilogue = EPI_F32;
  if (op == WS_OP_SWIGLU_GEMV) {
    p.nmat = 2;
    p.epilogue = EPI_SWIGLU;
  } else if (op == WS_OP_LMHEAD_ARGMAX) {
    p.epilogue = EPI_ARGMAX;
  } else if (op != WS_OP_GEMV && op != WS_OP_QKV_GEMV) {
    return false;
  }
  char why[256];
  return plan_gemv(p, op == WS_OP_LMHEAD_ARGMAX ? -1 : 0, why, sizeof why);
}

size_t ws_workspace_bytes(int op, int M, int K, int B) {
  if (op == WS_OP_ARGMAX_ROWS) return argmax_rows_workspace(M, K);
  if (M <= 0 || K <= 0 || K % 8 != 0 || B < 1 || B > kMaxBatch) return 0;
  GemvParams p;
  if (!plan_for_op(op, M, K, B, p)) return 0;
  return workspace_layout(p, nullptr, nullptr, nullptr, nullptr, nullptr);
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
}

ws_status ws_set_tuning(const ws_tuning* t) {
  if (!t || t->ring_bytes < 0 || t->ring_bytes > kSmemMax || t->grid_cap < 0 ||
      t->force_ksplit < 0 || t->force_rt < 0 || t->force_rt > 2 || t->piece_bytes < 0 ||
      t->piece_bytes > 64 * 1024 || t->timeout_ns == 0) {
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
