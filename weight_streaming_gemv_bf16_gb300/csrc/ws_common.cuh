// ws_common.cuh -- definitions shared by the library's translation units.
//
// The streaming GEMV computes y[b][m] = sum_k W[m][k] * x[b][k] with bf16 W and
// x and fp32 accumulation ("One Token, Kernel by Kernel: A Decode Step on a
// Laptop GPU", Step 1, "What one block launches"), with an optional
// normalisation prologue and a per-output epilogue.
//
// Work decomposition.  The rows of up to three weight matrices ("segments",
// e.g. Q, K and V) are cut into row groups of RT rows; K may be cut into S
// splits of KS columns.  One warp computes one (row group, split) task from
// start to end: it streams the task's weight rows through its own ring of
// shared-memory stages with bulk async copies, in pieces of PC columns,
// accumulates in registers and runs the epilogue itself.  Warps never wait on
// each other, so eight independent copy/compute pipelines overlap per CTA.
// CTAs are grouped by split (grid = S * Gs); CTA g of a split takes a
// contiguous, balanced range of row groups and deals them to its warps
// round-robin.  The activations (normalised by the prologue) sit in shared
// memory as bf16, the KS columns of the CTA's split.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ws {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSeg = 3;
constexpr int kMaxStages = 8;  // ring stages per warp
// tensor-core kernel: the warps of a CTA that stream and multiply (the others
// only stage): fewer rows in flight per CTA, so that each row's copy is longer
constexpr int kMmaWarps = 4;
constexpr int kMaxBatch = 16;
constexpr int kMaxChainBatch = 128;  // chains: larger batches run in tiles of kMaxBatch rows

enum Prologue { PRO_NONE = 0, PRO_RMSNORM = 1, PRO_LAYERNORM = 2 };
enum Epilogue {
  EPI_F32 = 0,        // out fp32 = acc
  EPI_BF16 = 1,       // out bf16 = acc
  EPI_RESID = 2,      // out fp32 = res_in + acc (res_in may be out itself)
  EPI_BIAS_GELU = 3,  // out bf16 = gelu(bf16(acc + bias))
  EPI_SWIGLU = 4,     // out bf16 = silu(acc_gate) * acc_up
  EPI_ARGMAX = 5      // optional fp32 logits; per-row argmax over all outputs
};
enum DType { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
enum DeviceError { DERR_TIMEOUT = 1 };

// 4-bit group-128 weights ("One Token, Kernel by Kernel", "4-bit weights"):
// a group is 128 consecutive weights of a row with a bf16 scale s and zero z,
// code q standing for s * (q - 8) + z.  A row is a run of super-groups of
// four groups: their codes (64 bytes a group; 32-bit word i of a group holds
// k = 8i .. 8i+7, even k in the low half's nibbles, odd k in the high half's),
// then their (s, z) pairs, zero-padded to 16 bytes (272 bytes for four).
constexpr int kQ4Group = 128;
constexpr int kQ4Super = 512;       // columns of a full super-group
constexpr int kQ4SuperBytes = 272;  // its bytes
__host__ __device__ constexpr int q4_super_bytes(int groups) { return (groups * 68 + 15) & ~15; }
// Bytes of a row before column k (k a multiple of 512, or the row's end).
__host__ __device__ constexpr int q4_prefix(int k) {
  return (k / kQ4Super) * kQ4SuperBytes +
         ((k % kQ4Super) ? q4_super_bytes((k % kQ4Super) / kQ4Group) : 0);
}
enum WeightFormat { WF_BF16 = 0, WF_Q4 = 1 };

struct Seg {
  const uint16_t* W0;  // bf16 [M][K]; 4-bit rows (q4_prefix(K) bytes each) for WF_Q4
  const uint16_t* W1;  // second matrix read in lockstep (SwiGLU up), or null
  void* out;           // [B][M]
  int M;
  int rg_begin;        // first row group of this segment (all segments)
  int row_base;        // first row of this segment in the concatenated rows
};

struct Sched {
  int RT;           // rows per task
  int S;            // K splits
  int KS;           // columns per split
  int PC;           // columns per piece (one ring stage)
  int NP;           // pieces per task, ceil(KS / PC)
  int NSW;          // ring stages per warp
  int piece_bytes;  // bytes of one ring stage
  int RG;           // row groups (tasks per split), all segments
  int Gs;           // CTAs per split
  int grid;         // S * Gs
  int BT;           // batch the kernel is instantiated for (>= B)
  int smem_bytes;
  int off_bar, off_flags, off_stats, off_red, off_arg, off_xs, off_ring;
  int off_res;   // residual rows of the CTA in shared memory (0: read at the epilogue)
  int res_rows;  // rows reserved there per batch row
  // tensor-core kernel (mma = 1): tasks of 16 rows, piece rows prow bytes
  // apart in the ring and activation rows xrs 16-byte chunks apart in shared
  // memory (both odd multiples of 16 bytes: ldmatrix rows in distinct banks)
  int mma, prow, xrs;
  int form;      // its chain form (F_ANY for none)
  int off_xsum;  // 4-bit weights: sums of 16 staged activations, [BT][KS / 16] fp32
                 // (tensor-core kernel: of 128, [8][KS / 128])
  int off_xzero;  // 4-bit weights, tensor-core kernel: a 16-byte zero row
};

struct alignas(16) GemvParams {
  Seg seg[kMaxSeg];
  int nseg;
  int nmat;  // 1, or 2 for a gate/up pair
  int wfmt;  // WeightFormat
  int K, B, M_total;
  const void* x;
  int x_dtype;
  int prologue;
  const uint16_t* gamma;
  const uint16_t* beta;
  float eps;
  int epilogue;
  const uint16_t* bias;
  const float* res_in;
  int* argmax_idx;
  float* logits;
  // workspace (split-K partials and tickets, argmax partials)
  float* part;
  unsigned* tickets;
  float* arg_val;
  int* arg_idx;
  unsigned* arg_ticket;
  int* err;
  unsigned long long timeout_ns;
  int evict_first;
  float* trace_out;  // persistent chain: copy seg[0].out ([B][M] fp32) here after the op
  // training forward of the LayerNorm -> Linear -> GELU block, each kept for
  // the backward when not null: the GELU's input t = bf16(ln.W^T + bias),
  // bf16 [B][M]; the GELU's derivative at t, fp32 [B][M]; the Linear's input
  // ln = bf16(LayerNorm(x)), bf16 [B][K]; the LayerNorm's mean and rstd per
  // batch row, fp32 [B][2]
  uint16_t* pre_out;
  float* gelu_grad;
  uint16_t* ln_out;
  float* ln_stats;
  // optional diagnostics of a launch inside a chain: globaltimer ns per CTA at
  // stamps[cta * stamp_stride + i], i = 0 entry, 1 dependency released,
  // 2 activations staged, 3 end
  unsigned long long* stamps;
  int stamp_stride;
  Sched sc;
};

// The persistent chain kernel: every op of a chain as one phase of a single
// cooperative launch (one CTA per SM), phases separated by grid barriers.
struct PersistParams {
  const GemvParams* ops;  // device array of nops planned ops
  int nops;
  unsigned* bar;          // nops + 1 counters, zero between launches
  int* err;
  unsigned long long timeout_ns;
  int evict_first;
  int l2_ahead;           // pieces per warp prefetched into L2 ahead of its copies
  int BT;
  int NSW;                // ring stages per warp
  int slot_bytes;         // bytes per ring stage (the largest piece of any op)
  int grid;
  int smem_bytes;
  int off_op, off_bar, off_empty, off_ends, off_flags, off_stats, off_red, off_arg, off_xs,
      off_ring;
  // optional: per CTA and op (kStampsPerOp entries), globaltimer ns at [0]
  // the start of the op (after its grid barrier), [1] after the activations
  // are staged, [2] when its tasks are done, [3] the first weight piece of
  // the op landing (warp 0); then per compute warp w, at [4 + 5w], the ns it
  // spent waiting for weight pieces, 0 (unused), in dot products and in the
  // reduction and epilogue, and the units it ran
  unsigned long long* stamps;
};
constexpr int kStampsPerOp = 4 + 5 * kWarps;

// The split and the row-group range of CTA `cta`.
__host__ __device__ inline void cta_range(const Sched& sc, int cta, int& ks, int& rg0, int& rg1) {
  ks = cta / sc.Gs;
  // 32-bit products: the planner keeps Gs * RG below 2^32
  const unsigned g = (unsigned)(cta - ks * sc.Gs);
  rg0 = (int)(g * (unsigned)sc.RG / (unsigned)sc.Gs);
  rg1 = (int)((g + 1) * (unsigned)sc.RG / (unsigned)sc.Gs);
}

// Tasks of warp `w` in a CTA whose row groups are [rg0, rg1): rg0 + w + t * kWarps.
__host__ __device__ inline int warp_tasks(int rg0, int rg1, int w) {
  return rg1 - rg0 > w ? (rg1 - rg0 - w + kWarps - 1) / kWarps : 0;
}

// Segment and local row group of a global row group.
__host__ __device__ inline void decode_rg(const GemvParams& p, int rg, int& seg, int& rgl) {
  seg = 0;
  while (seg + 1 < p.nseg && rg >= p.seg[seg + 1].rg_begin) ++seg;
  rgl = rg - p.seg[seg].rg_begin;
}

// One-round RMSNorm staging (fp32 activations, the whole K in one CTA): each
// thread holds at most kOneRound 8-column chunks of the B x K activations.
// The chain forms hold BT chunks up to batch tile 8 (K <= 2048) and 12 at
// batch tile 16 (K <= 1536).
constexpr int kOneRound = 4;

__host__ __device__ constexpr int form_round_chunks(int BT) { return BT <= 8 ? BT : 12; }

__host__ __device__ inline bool one_round_rms(const GemvParams& p, int chunks = kOneRound) {
  return p.prologue == PRO_RMSNORM && p.x_dtype == DT_F32 && p.sc.KS == p.K &&
         p.B * (p.K >> 3) <= chunks * kThreads;
}

// Compile-time form of a launch.  The ops of a decode chain each run a kernel
// holding only the code of their own form (staging path, epilogue, no K
// split); F_ANY reads all of it from the parameters.  Every launch of a chain
// starts with cold instruction caches, so code that a launch never runs
// still costs time.
enum KernelForm {
  F_ANY = 0,
  F_RMS_F32 = 1,     // one-round RMSNorm of fp32 x; fp32 outputs (QKV)
  F_RMS_SWIGLU = 2,  // one-round RMSNorm; SwiGLU of a gate/up pair (bf16 out)
  F_RMS_ARGMAX = 3,  // one-round RMSNorm; logits and argmax (LM head)
  F_BF16_RESID = 4,  // bf16 x without prologue; fp32 residual add (Wo, Wd)
  F_BF16_F32 = 5,    // bf16 x without prologue; fp32 outputs (the plain GEMV)
  F_LN_GELU = 6,     // one-round LayerNorm of bf16 x; bias + GELU (the MLP block), K split allowed
  kNumForms = 7
};

template <int F>
struct FormTraits {
  static constexpr int epi = -1;  // epilogue, or -1: read from the parameters
  static constexpr bool rms1 = false, copy_bf16 = false, no_split = false, one_seg = false;
  static constexpr bool ln1 = false;  // one-round LayerNorm staging
};
template <>
struct FormTraits<F_RMS_F32> {
  static constexpr int epi = EPI_F32;
  static constexpr bool rms1 = true, copy_bf16 = false, no_split = true, one_seg = false;
  static constexpr bool ln1 = false;
};
template <>
struct FormTraits<F_RMS_SWIGLU> {
  static constexpr int epi = EPI_SWIGLU;
  static constexpr bool rms1 = true, copy_bf16 = false, no_split = true, one_seg = true;
  static constexpr bool ln1 = false;
};
template <>
struct FormTraits<F_RMS_ARGMAX> {
  static constexpr int epi = EPI_ARGMAX;
  static constexpr bool rms1 = true, copy_bf16 = false, no_split = true, one_seg = true;
  static constexpr bool ln1 = false;
};
template <>
struct FormTraits<F_BF16_RESID> {
  static constexpr int epi = EPI_RESID;
  static constexpr bool rms1 = false, copy_bf16 = true, no_split = true, one_seg = true;
  static constexpr bool ln1 = false;
};
template <>
struct FormTraits<F_BF16_F32> {
  static constexpr int epi = EPI_F32;
  static constexpr bool rms1 = false, copy_bf16 = true, no_split = true, one_seg = true;
  static constexpr bool ln1 = false;
};
template <>
struct FormTraits<F_LN_GELU> {
  static constexpr int epi = EPI_BIAS_GELU;
  static constexpr bool rms1 = false, copy_bf16 = false, no_split = false, one_seg = true;
  static constexpr bool ln1 = true;
};

// The form a planned launch can run as.
inline int kernel_form(const GemvParams& p) {
  if (p.prologue == PRO_LAYERNORM && p.x_dtype == DT_BF16 && p.epilogue == EPI_BIAS_GELU &&
      p.nseg == 1 && p.B * (p.K >> 3) <= form_round_chunks(p.sc.BT) * kThreads)
    return F_LN_GELU;
  if (p.sc.S != 1) return F_ANY;
  if (one_round_rms(p, form_round_chunks(p.sc.BT))) {
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

struct Tuning {
  int ring_bytes;    // shared-memory ring budget per CTA (all warps)
  int grid_cap;      // max CTAs (0: one per SM)
  int force_ksplit;  // 0: heuristic
  int force_rt;      // rows per task, 1 or 2 (0: heuristic)
  int evict_first;   // weights streamed with an L2 evict-first policy
  int piece_bytes;   // target bytes per ring stage
  unsigned long long timeout_ns;
  int l2_ahead;      // persistent chain: pieces per warp prefetched into L2 ahead of the copies
  int forms;         // 1: launches of a known form run that form's kernel (0: the general one)
  int launch_pdl;    // 1: standalone GEMV launches carry the programmatic-dependent-launch attribute
  int mma;           // 1: large chain-form ops at batch tiles 8 and 16 run on tensor cores (mma.sync)
  int ctas_per_sm;   // CUDA-core launches: CTAs resident per SM (0: the planner's choice)
  int q4_mma;        // 4-bit ops with two 16-row tasks per warp or more on tensor cores: 1 at B 2..4, 2 always
};

// Host-side helpers implemented in ws_gemv.cu / ws_misc.cu.
Tuning& tuning();
int device_sm_count();
int* device_error_ptr();
void set_error(const char* fmt, ...);
bool plan_gemv(GemvParams& p, int force_S, char* why, size_t why_len);
size_t workspace_layout(const GemvParams& p, size_t* off_tickets, size_t* off_part,
                        size_t* off_argv, size_t* off_argi, size_t* off_argt);
bool bind_workspace(GemvParams& p, void* ws, size_t ws_bytes);
bool prepare_gemv(const GemvParams& p);
cudaError_t launch_gemv(const GemvParams& p, cudaStream_t stream, bool pdl);
void init_gemv_params(GemvParams& p, int K, int B);
size_t argmax_rows_workspace(int rows, int cols);
// persistent chain (ws_persist.cu)
bool plan_gemv_persistent(GemvParams& p, int ring_bytes, char* why, size_t why_len);
int persistent_ring_bytes(int B, int kmax);
bool plan_persistent(PersistParams& pp, const GemvParams* ops, int nops, int B, char* why,
                     size_t why_len);
bool prepare_persistent(int BT);
cudaError_t launch_persistent(const PersistParams& pp, cudaStream_t stream);

}  // namespace ws
