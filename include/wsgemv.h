/*
 * wsgemv.h -- C ABI of libwsgemv.so: the BF16 weight-streaming decode chain
 * for NVIDIA GB300 (sm_103a).
 *
 * What it computes.  At decode batch 1..16 every linear layer of a Llama-style
 * model is a matrix-vector product: y[b][m] = sum_k W[m][k] * x[b][k], BF16
 * weights and activations, FP32 accumulation ("One Token, Kernel by Kernel: A
 * Decode Step on a Laptop GPU", Step 1, "What one block launches").  The
 * library streams each weight matrix from HBM exactly once per call, fuses
 * the RMSNorm in front ("GPU Kernel Optimization", Architecture) and the
 * SwiGLU, residual, bias+GELU or argmax after, and replays whole decode
 * chains in one CUDA graph while a side stream prefetches the next op's
 * weights into L2 ("Making small PyTorch ops faster on a laptop GPU",
 * "Prefetching the next layer while this one runs" and "Measuring instead of
 * predicting").
 *
 * Conventions for every call:
 *  - Pointers named W*, x, h, y, gamma, beta, bias, s, z, idx, logits and
 *    workspace are DEVICE pointers owned by the caller; the library never
 *    frees them.  Host pointers appear only where a name ends in _host.
 *  - bf16/fp16 tensors are passed as void* to their 16-bit patterns.
 *  - Layouts are row-major: W is [M][K] (a linear layer's weight[out][in],
 *    K contiguous); x is [B][K]; outputs are [B][M].
 *  - Device pointers must be 16-byte aligned, K a multiple of 8 and
 *    1 <= B <= 16; otherwise WS_ERR_ALIGN / WS_ERR_SHAPE is returned and
 *    nothing is launched.  There is no fallback path of any kind.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  A launch error is returned as WS_ERR_CUDA.
 *  - Every GEMV-family call takes an optional workspace (device memory, may be
 *    NULL).  It enables split-K, which the schedule uses for skinny shapes
 *    and needs when B * K is too large for the activations to sit in shared
 *    memory (then a NULL workspace gives WS_ERR_ARG).  Size it with
 *    ws_workspace_bytes().
 *  - A workspace must be zero-filled before its first use; the library
 *    leaves it zeroed again after every successful call, so one workspace
 *    serves any number of calls ordered on one stream.  Calls that share a
 *    workspace must not overlap in time.
 *  - Device-side waits are bounded; a wait that runs out sets a device error
 *    flag read by ws_device_error() and the kernel returns.
 *  - No exception crosses the ABI.  ws_last_error() gives a thread-local
 *    message for the last failing call.
 */
#ifndef WSGEMV_H
#define WSGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WS_OK = 0,
  WS_ERR_ARG = -1,      /* null pointer, bad enum, workspace too small       */
  WS_ERR_ALIGN = -2,    /* a device pointer not 16-byte aligned              */
  WS_ERR_SHAPE = -3,    /* K % 8 != 0, B outside 1..16, sizes <= 0           */
  WS_ERR_CUDA = -4,     /* a CUDA runtime call failed                        */
  WS_ERR_TIMEOUT = -5,  /* a bounded device wait ran out                     */
  WS_ERR_NOMEM = -6,    /* the chain could not allocate its own buffers      */
  WS_ERR_STATE = -7     /* chain call out of order (e.g. run before capture) */
} ws_status;

typedef void *ws_stream_t; /* a cudaStream_t */

enum { WS_DTYPE_F32 = 0, WS_DTYPE_BF16 = 1, WS_DTYPE_F16 = 2 };

/* ------------------------------------------------------------------------
 * GEMV family.  All accumulate in fp32; the activations the dot products read
 * are bf16 (a normalisation prologue rounds its output to bf16 once).
 * ---------------------------------------------------------------------- */

/* y[b][m] = sum_k W[m][k] x[b][k].  W bf16 [M][K], x bf16 [B][K], y fp32
 * [B][M].  A workspace enables split-K for skinny shapes such as the
 * 256 x 1536 K/V projections, which lose bandwidth as one short kernel ("One
 * Token, Kernel by Kernel", Step 2, "The GEMVs, through Nsight Compute");
 * size it with ws_workspace_bytes(WS_OP_GEMV, M, K, B).  Split partials are
 * summed in a fixed order, so results do not depend on timing. */
ws_status ws_gemv_bf16(const void *W, const void *x, float *y, int M, int K, int B,
                       void *workspace, size_t workspace_bytes, ws_stream_t stream);

/* The same product as ws_gemv_bf16 for callers that cannot allocate device
 * memory when they need it: code running while a stream is captured into a
 * CUDA graph, serving loops that must not grow their memory after start-up,
 * hosts that only pass in memory they allocated themselves.  The pages have
 * no counterpart to this call; it is a convenience of this library.
 *  - It allocates nothing.  When the schedule splits K, the partial sums and
 *    tickets live in a fixed 1 MiB array of device memory owned by the
 *    library (every GPU that loads the library holds it until exit).
 *  - Shapes whose split-K scratch would exceed 1 MiB are rejected with
 *    WS_ERR_SHAPE and a message; use ws_gemv_bf16 with a workspace for those.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *    The address is kept for the life of the process: a device reset
 *    (cudaDeviceReset) while the library is loaded is not supported, since
 *    the array may come back at another address.
 *  - Each call clears the tickets on `stream` before its kernel.  All calls
 *    share the one array, which keeps the last call's contents: calls that
 *    overlap on the GPU (different streams, no ordering) race on it.
 * W bf16 [M][K], x bf16 [B][K], y fp32 [B][M]; same alignment and shape rules
 * as ws_gemv_bf16. */
ws_status ws_gemv_bf16_noalloc(const void *W, const void *x, float *y, int M, int K, int B,
                               ws_stream_t stream);

/* 4-bit group-128 weights ("One Token, Kernel by Kernel: A Decode Step on a
 * Laptop GPU", "4-bit weights": every linear layer quantised to 4-bit
 * integers in groups of 128, 0.82 GB instead of 3.09 for Qwen2.5-1.5B).  A
 * group is 128 consecutive weights of a row with a bf16 scale s and zero z;
 * code q (0..15) stands for s * (q - 8) + z.  A packed row (ws_q4_row_bytes(K)
 * bytes, K a multiple of 128) is a run of super-groups of four groups: their
 * codes, 64 bytes a group, in which 32-bit little-endian word i holds weights
 * 8i .. 8i+7 (bits 4j..4j+3: weight 8i+2j; bits 16+4j..16+4j+3: weight
 * 8i+2j+1), then their (s, z) pairs (4 bytes each, s first), zero-padded to
 * 16 bytes: 272 bytes for four groups, 4.25 bits a weight.
 *
 * ws_q4_row_bytes: bytes of one packed row, or 0 when K is not a positive
 * multiple of 128.
 * ws_quantize_q4: W bf16 [M][K] -> Wq packed [M][ws_q4_row_bytes(K)], min-max
 * per group with every decision in fp32: s = bf16((max - min) / 15),
 * z = bf16(min + 8 s), q = clamp(rint((w - z) / s) + 8, 0, 15) (8 when s is
 * 0).  Both pointers 16-byte aligned; finite weights.
 * ws_gemv_q4: y[b][m] = sum_k w[m][k] * x[b][k] for the packed rows, x bf16
 * [B][K], y fp32 [B][M], B <= 4, fp32 accumulation; the codes are expanded
 * inside the GEMV (no dequantised copy is written).  Workspace as
 * ws_gemv_bf16 (4-bit rows are never split along K, so none is needed). */
size_t ws_q4_row_bytes(int K);
ws_status ws_quantize_q4(const void *W, void *Wq, int M, int K, ws_stream_t stream);
ws_status ws_gemv_q4(const void *Wq, const void *x, float *y, int M, int K, int B,
                     void *workspace, size_t workspace_bytes, ws_stream_t stream);

/* h_out[b][m] = h_in[b][m] + sum_k W[m][k] x[b][k]: the residual add of a
 * decoder block folded into the GEMV's epilogue ("One Token, Kernel by
 * Kernel", Step 1, "What one block launches").  x bf16 [B][K]; h_in, h_out
 * fp32 [B][M]; h_in may equal h_out (in place) or be NULL (= h_out). */
ws_status ws_gemv_residual(const void *W, const void *x, const float *h_in, float *h_out,
                           int M, int K, int B, void *workspace, size_t workspace_bytes,
                           ws_stream_t stream);

/* y = bf16(RMSNorm(x, gamma)) . W^T with RMSNorm(x) = x / sqrt(mean_k x^2 + eps)
 * * gamma per row ("GPU Kernel Optimization", Architecture: mean square,
 * rsqrt and weight multiply in one kernel).  x fp32 or bf16 [B][K]
 * (x_dtype), gamma bf16 [K], y fp32 [B][M]. */
ws_status ws_rmsnorm_gemv(const void *x, int x_dtype, const void *gamma, const void *W,
                          float *y, int M, int K, int B, float eps,
                          void *workspace, size_t workspace_bytes, ws_stream_t stream);

/* Merged Q/K/V projection in one launch: a = bf16(RMSNorm(x, gamma));
 * q = a.Wq^T [B][Mq], k = a.Wk^T [B][Mkv], v = a.Wv^T [B][Mkv], all fp32.
 * One launch instead of three removes the small-GEMV loss ("One Token, Kernel
 * by Kernel", "In the real world": merged QKV projections). */
ws_status ws_qkv_gemv(const void *x, int x_dtype, const void *gamma,
                      const void *Wq, const void *Wk, const void *Wv,
                      float *q, float *k, float *v, int Mq, int Mkv, int K, int B,
                      float eps, void *workspace, size_t workspace_bytes, ws_stream_t stream);

/* SwiGLU MLP front half in one pass over Wg and Wu:
 * m = bf16(RMSNorm(x, gamma)) (or m = x when gamma is NULL; x must then be
 * bf16); s = bf16(silu(m.Wg^T) * (m.Wu^T)) with silu(g) = g / (1 + exp(-g)).
 * Wg, Wu bf16 [M][K]; s bf16 [B][M] ("One Token, Kernel by Kernel", Step 1,
 * "The setup": SwiGLU MLP). */
ws_status ws_swiglu_gemv(const void *x, int x_dtype, const void *gamma,
                         const void *Wg, const void *Wu, void *s,
                         int M, int K, int B, float eps,
                         void *workspace, size_t workspace_bytes, ws_stream_t stream);

/* z = bf16(gelu(bf16(bf16(LayerNorm(x)) . W^T + bias))), exact-erf GELU,
 * biased variance: one LayerNorm -> Linear -> GELU block in bf16 ("Making
 * small PyTorch ops faster on a laptop GPU", "Beyond language models").
 * x bf16 [B][K]; gamma, beta bf16 [K]; W bf16 [M][K]; bias bf16 [M];
 * z bf16 [B][M]. */
ws_status ws_ln_gemv_gelu(const void *x, const void *gamma, const void *beta,
                          const void *W, const void *bias, void *z,
                          int M, int K, int B, float eps,
                          void *workspace, size_t workspace_bytes, ws_stream_t stream);

/* LM head with a fused argmax: logits = bf16(RMSNorm(h, gamma)) . W^T and
 * idx[b] = the lowest j with logits[b][j] == max_j logits[b][j] ("One Token,
 * Kernel by Kernel", "The whole step": LM head 151,936 x 1,536, then an
 * argmax over the logits).  h fp32 or bf16 [B][K] (h_dtype); idx int32 [B];
 * logits fp32 [B][V] or NULL.  Workspace required:
 * ws_workspace_bytes(WS_OP_LMHEAD_ARGMAX, V, K, B). */
ws_status ws_lmhead_argmax(const void *h, int h_dtype, const void *gamma, const void *W,
                           int32_t *idx, float *logits, int V, int K, int B, float eps,
                           void *workspace, size_t workspace_bytes, ws_stream_t stream);

/* One decode step of grouped-query attention over a key-value cache
 * ("Making small PyTorch ops faster on a laptop GPU", "A full decode step is
 * a different story"; "One Token, Kernel by Kernel", "The fix: Part 10's
 * split-KV kernel").  Per batch row b: the new key and value (k_new, v_new
 * fp32 [B][n_kv_heads * 128], rounded to bf16) are written at slot pos[b] of
 * the caches (bf16 [B][n_kv_heads][s_max][128], 16-byte aligned; the caller
 * owns them); query head h (q fp32 [B][n_heads * 128]) attends over slots
 * 0 .. pos[b] of key-value head h / (n_heads / n_kv_heads) with scores
 * q.k / sqrt(128) and an fp32 softmax.  The two products run on warp-level
 * bf16 tensor-core MMAs with fp32 accumulators; q and the probabilities
 * enter as bf16 hi + lo pairs (relative error 2^-17).  Output: out_f32 [B][n_heads * 128]
 * and/or out_bf16 (bf16, the same shape); either may be NULL, not both.
 * pos: int32 [B] in device memory, read when the kernel runs (a captured
 * graph replays with the current positions); a position outside
 * 0 .. s_max - 1 skips that row and raises the device error flag (2).
 * head_dim must be 128, n_heads / n_kv_heads at most 8, s_max a multiple
 * of 64, 1 <= B <= 16; caches, k_new and v_new 16-byte aligned, q 8-byte
 * aligned.  Slots after pos are never read (they may hold anything).  Each
 * (row, key-value head) is cut into splits of whole 64-slot runs, as many as
 * fill one wave of CTAs; the last split of each group of 16 merges the
 * group's partial softmax results and the last group merges the groups.
 * Workspace (zero-filled before its first use, left zeroed by every call):
 * ws_attention_workspace_bytes(B, n_heads, n_kv_heads, 128, s_max). */
size_t ws_attention_workspace_bytes(int B, int n_heads, int n_kv_heads, int head_dim, int s_max);
ws_status ws_decode_attention(const float *q, const float *k_new, const float *v_new,
                              void *k_cache, void *v_cache, const int32_t *pos, float *out_f32,
                              void *out_bf16, int B, int n_heads, int n_kv_heads, int head_dim,
                              int s_max, void *workspace, size_t workspace_bytes,
                              ws_stream_t stream);

/* idx[r] = the lowest j with v[r][j] == max_j v[r][j] for fp32 rows
 * [rows][cols] ("One Token, Kernel by Kernel", "The whole step").  Workspace
 * required: ws_workspace_bytes(WS_OP_ARGMAX_ROWS, rows, cols, 1). */
ws_status ws_argmax_rows(const float *logits, int32_t *idx, int rows, int cols,
                         void *workspace, size_t workspace_bytes, ws_stream_t stream);

/* Standalone RMSNorm of [R][N] rows, fp16 or bf16 in and out (dtype), gamma of
 * the same dtype: y = x / sqrt(mean x^2 + eps) * gamma computed in fp32 and
 * rounded once ("GPU Kernel Optimization", Architecture: one program per
 * row).  N must be a multiple of 8. */
ws_status ws_rmsnorm(const void *x, const void *gamma, void *y, int R, int N, int dtype,
                     float eps, ws_stream_t stream);

/* ------------------------------------------------------------------------
 * L2 prefetch ("Making small PyTorch ops faster on a laptop GPU",
 * "Prefetching the next layer while this one runs"): a small kernel asks L2
 * to fetch `bytes` starting at `ptr` and never writes memory, so every result
 * of the ops around it stays bit-identical.
 * ---------------------------------------------------------------------- */
enum {
  WS_PREFETCH_NONE = 0,
  WS_PREFETCH_L2 = 1,            /* prefetch.global.L2 every stride_bytes         */
  WS_PREFETCH_L2_EVICT_LAST = 2, /* prefetch.global.L2::evict_last every stride   */
  WS_PREFETCH_BULK = 3           /* cp.async.bulk.prefetch.L2, stride_bytes chunks */
};

typedef struct {
  int blocks;       /* CTAs of the prefetch kernel                         */
  int threads;      /* threads per CTA                                     */
  int stride_bytes; /* bytes between prefetches / bytes per bulk prefetch  */
  int mode;         /* WS_PREFETCH_*                                       */
} ws_prefetch_plan;

/* Enqueue one prefetch kernel over [ptr, ptr + bytes).  mode NONE (or
 * bytes == 0) enqueues nothing.  BULK needs ptr 16-byte aligned and
 * stride_bytes a multiple of 16. */
ws_status ws_l2_prefetch(const void *ptr, size_t bytes, ws_prefetch_plan plan,
                         ws_stream_t stream);

/* ------------------------------------------------------------------------
 * Chain executor: a block list replayed as one CUDA graph.
 * ---------------------------------------------------------------------- */
enum { WS_BLOCK_QWEN = 1, WS_BLOCK_MLP = 2, WS_BLOCK_HEAD = 3 };
enum { WS_WEIGHTS_BF16 = 0, WS_WEIGHTS_Q4 = 1 };

/* One decoder block of a Llama-style model at decode ("One Token, Kernel by
 * Kernel", Step 1): a = bf16(RMSNorm(h, gamma1)); q,k,v = a.W{q,k,v}^T;
 * h += attn.Wo^T; m = bf16(RMSNorm(h, gamma2)); s = bf16(silu(m.Wg^T) *
 * m.Wu^T); h += s.Wd^T.  The attention itself is outside this library: its
 * output is supplied in `attn` (bf16 [B][H]). */
typedef struct {
  const void *gamma1, *Wq, *Wk, *Wv, *Wo, *gamma2, *Wg, *Wu, *Wd; /* bf16 */
  const void *attn;      /* bf16 [B][H]  (unused with opts.attention)    */
  float *q, *k, *v;      /* fp32 [B][H], [B][KV], [B][KV]; NULL: internal */
  /* opts.attention: the block's key-value caches, bf16
   * [B][KV / 128][s_max][128], updated at pos by every step */
  void *k_cache, *v_cache;
} ws_qwen_block;

/* z = bf16(gelu(bf16(bf16(LayerNorm(x)) . W^T + bias))) ("Making small
 * PyTorch ops faster on a laptop GPU", "Beyond language models"). */
typedef struct {
  const void *gamma, *beta, *W, *bias; /* bf16 [w], [w], [w][w], [w] */
} ws_mlp_block;

/* Final RMSNorm, LM head and argmax ("One Token, Kernel by Kernel", "The
 * whole step"). */
typedef struct {
  const void *gamma;  /* bf16 [H]            */
  const void *W;      /* bf16 [V][H]         */
  int32_t *idx;       /* int32 [B]           */
  float *logits;      /* fp32 [B][V] or NULL */
} ws_head_block;

typedef struct {
  int kind; /* WS_BLOCK_* */
  union {
    ws_qwen_block qwen;
    ws_mlp_block mlp;
    ws_head_block head;
  } u;
} ws_block_desc;

typedef struct {
  int batch;        /* B, 1..128; above 16 every op runs once per 16-row
                       batch tile, tiles of an op back to back (bf16 weights,
                       no attention, no training saves)                     */
  int hidden;       /* H (Qwen) or width (MLP)                              */
  int kv_dim;       /* K/V projection rows (Qwen)                           */
  int inter;        /* MLP rows I (Qwen)                                    */
  int vocab;        /* LM head rows V (head block)                          */
  float eps;        /* RMSNorm / LayerNorm epsilon                          */
  /* Qwen chains: the residual stream.  The first block reads h_in (fp32
   * [B][H], read-only) and every block updates h_out (fp32 [B][H]), so each
   * replay starts again from h_in. */
  const float *h_in;
  float *h_out;
  /* MLP chains: x_in bf16 [B][w] (read-only) and the chain output y_out bf16
   * [B][w]. */
  const void *x_in;
  void *y_out;
  /* Optional per-block trace (for per-block checks): Qwen chains get h
   * after every block, fp32 [L][B][H] (a copy after each block); MLP chains
   * get every block's output, bf16 [L][B][w] (written in place by the block,
   * the last one copied from y_out). */
  float *h_trace;
  int use_pdl;          /* 1: programmatic dependent launch between ops      */
  int prefetch;         /* 0 off, 1 tuned plans, 2 fixed_plan for every op   */
  ws_prefetch_plan fixed_plan;
  int distance;         /* prefetch op i + distance while op i runs (>= 1)   */
  int decoy;            /* 1: aim each prefetch at the wrong op (control)    */
  int tune_pairs;       /* paired replays per candidate (>= 8)               */
  float tune_min_gain;  /* keep a plan only if the 95% CI lower bound of its
                           relative gain exceeds this (e.g. 0.01)            */
  int weight_format;    /* WS_WEIGHTS_BF16 (0), or WS_WEIGHTS_Q4 (1): every
                           weight matrix of the Qwen and head blocks (Wq, Wk,
                           Wv, Wo, Wg, Wu, Wd, the LM head) is packed 4-bit
                           rows as ws_quantize_q4 writes them (batch <= 4,
                           one launch per op); the RMSNorm gammas stay bf16 */
  int persistent;       /* 1: run the whole step as one persistent kernel
                           (batch <= 4): each op is a phase of a cooperative
                           launch with one CTA per SM, phases separated by
                           grid barriers, and every warp's weight stream runs
                           ahead across phase boundaries.  Prefetch plans do
                           not apply in this mode.  0: one launch per op with
                           programmatic dependent launch edges.              */
  /* 1: each Qwen block runs decode attention (ws_decode_attention: the new
   * key and value appended at pos[b], query heads of 128 over key-value
   * heads of 128) on its QKV outputs, and Wo reads its bf16 output instead
   * of `attn`.  pos: int32 [B] on the device, read when the step runs (the
   * caller advances it between steps); s_max: slots of each cache. */
  int attention;
  int s_max;
  const int32_t *pos;
  /* MLP chains, training forward (one launch per block, not persistent;
   * with h_trace set every block's output is written straight into its
   * trace slot): what each module keeps for the backward, per block, any of
   * them NULL to skip it.  mlp_ln: the Linear's input ln = bf16(LayerNorm(x)),
   * bf16 [L][B][w]; mlp_pre: the GELU's input t = bf16(ln.W^T + bias), bf16
   * [L][B][w]; mlp_gelu_grad: the GELU's derivative at t, Phi(t) + t phi(t),
   * fp32 [L][B][w]; mlp_ln_stats: the LayerNorm's mean and rstd of every
   * batch row of x, fp32 [L][B][2].  ws_mlp_backward_create reads mlp_ln,
   * mlp_gelu_grad and mlp_ln_stats (mlp_pre is for checks). */
  void *mlp_ln;
  void *mlp_pre;
  float *mlp_gelu_grad;
  float *mlp_ln_stats;
} ws_chain_opts;

typedef struct ws_chain ws_chain;

ws_status ws_chain_create(const ws_block_desc *blocks, int n, const ws_chain_opts *opts,
                          ws_chain **out);
/* Measure prefetch plans per distinct op shape on throwaway weights and keep
 * the best only if its 95% confidence interval clears the minimum gain
 * ("Making small PyTorch ops faster on a laptop GPU", "Measuring instead of
 * predicting").  Blocks the calling thread; uses `stream`. */
ws_status ws_chain_tune(ws_chain *c, ws_stream_t stream);
/* Capture the chain: all ops on the main branch, each prefetch on a side
 * branch forked before op i and joined at the end, as one graph.  Capture
 * happens on a stream the chain owns (any caller stream, including the
 * legacy default stream, can then replay it); `stream` is not used. */
ws_status ws_chain_capture(ws_chain *c, ws_stream_t stream);
/* One decode step: one cudaGraphLaunch. */
ws_status ws_chain_run(ws_chain *c, ws_stream_t stream);
/* The same ops launched one by one without a graph (no prefetch). */
ws_status ws_chain_run_eager(ws_chain *c, ws_stream_t stream);
/* One decode step from HOST buffers: copies in_host (Qwen: fp32 [B][H] to
 * h_in; MLP: bf16 [B][w] to x_in) and, if not NULL, attn_host (bf16
 * [L][B][H], block order) to the chain's device inputs, replays the graph,
 * copies the result (head: int32 idx [B]; MLP: bf16 [B][w]) to out_host and
 * waits for the stream.  The copies and the step are one graph launch,
 * captured for these host buffers on first use.  Pinned host buffers that
 * are mapped into the device's address space (cudaHostAlloc, torch's
 * pin_memory) are copied by one word-copy kernel each way; other buffers by
 * cudaMemcpyAsync. */
ws_status ws_chain_step_host(ws_chain *c, const void *in_host, const void *attn_host,
                             void *out_host, ws_stream_t stream);
int ws_chain_num_ops(const ws_chain *c);
/* 1 if the chain runs as one persistent kernel per step, else 0. */
int ws_chain_is_persistent(const ws_chain *c);
/* Diagnostics.  ws_chain_grid: the CTA dimension of the stamp buffer (the
 * persistent kernel's grid, else the largest grid of any op: an op may run
 * more than one CTA per SM).
 * ws_chain_debug_stamps: a device buffer (uint64 [grid][ops][44], or NULL to
 * stop) where every later-captured step records globaltimer ns per CTA and
 * op.  Persistent chains: at the op's start (after its grid barrier), after
 * its activations are staged, when its tasks are done, and when warp 0's
 * first weight piece of the op landed; then for each of the CTA's 8 compute
 * warps the ns it spent waiting for weight pieces, 0 (unused), the ns in dot
 * products and in the reduction and epilogue, and the units it ran.  Graphs
 * of launches: at the CTA's entry, after its dependency on the previous op
 * was released, after its activations were staged, and when its tasks were
 * done; the rest 0 (CTAs beyond an op's grid are not written).  Call
 * ws_chain_capture again after setting it. */
int ws_chain_grid(const ws_chain *c);
ws_status ws_chain_debug_stamps(ws_chain *c, unsigned long long *stamps, size_t n);
/* Plan and measured gain (95% CI lower bound, mean) of each op; n entries. */
ws_status ws_chain_plans(const ws_chain *c, ws_prefetch_plan *plans, float *gain_lo,
                         float *gain_mean, int n);
/* Weight bytes each op streams (its algorithmic bytes); n entries. */
ws_status ws_chain_op_bytes(const ws_chain *c, size_t *bytes, int n);
void ws_chain_destroy(ws_chain *c);

/* ------------------------------------------------------------------------
 * Training: the backward pass of a chain of LayerNorm -> Linear(+bias) ->
 * GELU blocks ("Making small PyTorch ops faster on a laptop GPU", "It works
 * in training too": the gradient of block i reads W_i again, so while it runs
 * the prefetch fetches W_(i-1), and the gradients are bit-identical with and
 * without it).  Module by module in bf16, like the forward block: with t the
 * GELU's input, ln the Linear's input, xh = (x - mean) rstd,
 *   dlin = bf16(dz * gelu'(t)); dln = bf16(dlin . W); dW = bf16(dlin^T . ln);
 *   db = bf16(sum_b dlin); g = dln * gamma;
 *   dx = bf16(rstd (g - mean_k g - xh mean_k(g xh)));
 *   dgamma = bf16(sum_b dln xh); dbeta = bf16(sum_b dln),
 * and dx of block i is dz of block i - 1.  Sums in fp32 in a fixed order.
 * One launch per block (plus one for block 0's LayerNorm), replayed as one
 * CUDA graph with programmatic-dependent-launch edges; each launch streams
 * its weight with 2-D TMA in 8-column slabs, one slab per CTA.  dW and db of
 * every block, which nothing in the chain reads, are formed by one more
 * launch after it.
 * ---------------------------------------------------------------------- */
typedef struct {
  void *dW, *db, *dgamma, *dbeta; /* bf16 [w][w], [w], [w], [w]: written */
} ws_mlp_grads;

typedef struct {
  int batch;                /* B, 1..16                                      */
  int width;                /* w, a multiple of 64, 64..1024                 */
  /* the training forward's tensors (ws_chain_opts.mlp_* and h_trace):       */
  const void *x_in;         /* bf16 [B][w]: block 0's input                   */
  const void *acts;         /* bf16 [L][B][w]: every block's output          */
  const void *ln;           /* bf16 [L][B][w]: every block's Linear input    */
  const float *gelu_grad;   /* fp32 [L][B][w]: gelu' at every GELU input     */
  const float *ln_stats;    /* fp32 [L][B][2]: LayerNorm mean and rstd       */
  /* the gradient of the loss with respect to the last block's output, bf16
   * [B][w]; NULL: the mean-square loss of the chain output z,
   * mean(z^2) over B x w, whose gradient bf16(2 z / (B w)) is formed in fp32
   * by the first launch */
  const void *dz;
  void *dx;                 /* bf16 [B][w]: gradient of the chain input      */
  /* optional traces (NULL: not written): dx_trace bf16 [L+1][B][w], slot i
   * the gradient of block i's input (slot 0 = dx), slot L the loss gradient;
   * dlin_trace and dln_trace bf16 [L][B][w], block by block */
  void *dx_trace, *dlin_trace, *dln_trace;
  int use_pdl;              /* 1: programmatic dependent launch between launches */
  int prefetch;             /* 0 off, 1 measured plan (ws_mlp_backward_tune), 2 fixed_plan */
  ws_prefetch_plan fixed_plan;
  int distance;             /* prefetch the weight of launch s + distance (>= 1)  */
  int decoy;                /* 1: aim every prefetch at the wrong block (control) */
  int tune_pairs;           /* paired replays per candidate plan (>= 8)           */
  float tune_min_gain;      /* keep a plan only if its 95% CI lower bound exceeds */
} ws_mlp_backward_opts;

typedef struct ws_mlp_backward ws_mlp_backward;

/* blocks[i] / grads[i]: block i's parameters and its gradients (all 16-byte
 * aligned device pointers, owned by the caller, as are every tensor of
 * opts); the handle owns two dln scratch rows (when dln_trace is NULL), its
 * streams and its graph. */
ws_status ws_mlp_backward_create(const ws_mlp_block *blocks, const ws_mlp_grads *grads, int n,
                                 const ws_mlp_backward_opts *opts, ws_mlp_backward **out);
/* prefetch == 1: time the whole backward graph with each candidate plan
 * (every launch prefetching the weight of launch s + distance) against none
 * in interleaved pairs, and keep the best plan only if the 95% confidence
 * interval of its relative gain clears tune_min_gain ("Measuring instead of
 * predicting").  Runs the backward (it only rewrites the same gradients). */
ws_status ws_mlp_backward_tune(ws_mlp_backward *c, ws_stream_t stream);
ws_status ws_mlp_backward_capture(ws_mlp_backward *c, ws_stream_t stream);
/* One backward pass: one cudaGraphLaunch on `stream`. */
ws_status ws_mlp_backward_run(ws_mlp_backward *c, ws_stream_t stream);
/* The plan in use and its measured gain (95% CI lower bound, mean). */
ws_status ws_mlp_backward_plan(const ws_mlp_backward *c, ws_prefetch_plan *plan, float *gain_lo,
                               float *gain_mean);
/* Kernel launches per backward pass: one per block, one for block 0's
 * LayerNorm, one for the dW and db of every block. */
int ws_mlp_backward_num_launches(const ws_mlp_backward *c);
void ws_mlp_backward_destroy(ws_mlp_backward *c);

/* ------------------------------------------------------------------------
 * Sizing, errors, tuning knobs and measurement kernels.
 * ---------------------------------------------------------------------- */
enum {
  WS_OP_GEMV = 1,           /* ws_gemv_bf16, ws_gemv_residual, ws_rmsnorm_gemv,
                               ws_ln_gemv_gelu: M rows                          */
  WS_OP_SWIGLU_GEMV = 2,    /* ws_swiglu_gemv: M rows of each of Wg, Wu         */
  WS_OP_QKV_GEMV = 3,       /* ws_qkv_gemv: M = Mq + 2 * Mkv                    */
  WS_OP_LMHEAD_ARGMAX = 4,  /* ws_lmhead_argmax: M = V                          */
  WS_OP_ARGMAX_ROWS = 5     /* ws_argmax_rows: M = rows, K = cols               */
};

/* Workspace bytes an op's schedule uses on the current device (0: none). */
size_t ws_workspace_bytes(int op, int M, int K, int B);

const char *ws_last_error(void);

/* Device error flag of the current device (nonzero after a bounded wait ran
 * out); reset != 0 clears it.  Synchronises the device.  Returns -1 if the
 * flag cannot be read. */
int ws_device_error(int reset);

typedef struct {
  int ring_bytes;      /* shared-memory weight rings per CTA, all warps        */
  int grid_cap;        /* CTAs per GEMV launch (0: one per SM)                 */
  int force_ksplit;    /* K splits (0: heuristic)                              */
  int force_rt;        /* rows per warp task, 1, 2 or 4 (0: heuristic)         */
  int evict_first;     /* stream weights with an L2 evict-first hint           */
  int piece_bytes;     /* target bytes of one ring stage                       */
  unsigned long long timeout_ns; /* bound of every device wait                 */
  int l2_ahead;        /* persistent chain: weight pieces per warp the copy
                          producer prefetches into L2 ahead of its copies     */
  int forms;           /* 1 (default): a launch whose shape is one of a decode
                          chain's op forms (RMSNorm + fp32 out, RMSNorm +
                          SwiGLU, RMSNorm + argmax, bf16 x + residual; no K
                          split; batch <= 4) runs a kernel built for that form
                          alone; 0: every launch runs the general kernel.
                          Both compute the same values.                      */
  int launch_pdl;      /* 1: the standalone GEMV entry points launch with the
                          programmatic-dependent-launch attribute, so that a
                          GEMV following another one on the stream streams
                          its first weights while the previous one finishes
                          (every kernel here waits for the previous grid
                          before reading its activations; its weights and γ
                          it reads before, so they must not be outputs of
                          the GEMV launched just before it).  Default 0.     */
  int mma;             /* 1: launches of a chain form (with forms = 1) with
                          at least 8 Mi weights at batch 5..16 run a warp-
                          level tensor-core kernel (bf16 m16n8k16 MMA, fp32
                          accumulation, 16-row tasks); 0 (default): every
                          launch runs on CUDA cores, the vector-product
                          design.  Sums are ordered differently; both stay
                          within the fp32 tolerance of the oracle.           */
  int ctas_per_sm;     /* CUDA-core launches: CTAs each SM holds at once, 1..3;
                          the grid is that many per SM and every CTA's shared
                          memory (rings included) is sized so that they fit.
                          0 (default): the planner's choice -- two for 4-bit
                          rows at batch 1, else one.  A plan whose kernel's
                          registers or shared memory would not let that many
                          CTAs share an SM falls back to one.                */
  int q4_mma;          /* 4-bit ops of a chain form with at least two 16-row
                          tasks per warp (the LM head) run on the tensor-core
                          kernel: 1 (default) at batch 2..4, 2 at every
                          batch 1..4, 0 never (the CUDA-core kernel).       */
} ws_tuning;

void ws_get_tuning(ws_tuning *t);
ws_status ws_set_tuning(const ws_tuning *t);

/* Schedule a GEMV launch would use (for tests and reports): rows per warp
 * task RT, K splits S of KS columns, pieces of PC columns (NP per task),
 * NSW ring stages per warp of piece_bytes, RG row groups, grid CTAs. */
typedef struct {
  int RT, S, KS, PC, NP, NSW, piece_bytes, RG, grid, smem_bytes;
} ws_gemv_schedule;
ws_status ws_gemv_plan(int M_total, int K, int B, int nmat, int prologue_kind,
                       int epilogue_kind, int allow_split, ws_gemv_schedule *out);

/* Every bulk copy the producer of CTA `cta` would issue for a one-segment
 * GEMV of the given shape, as (source byte offset from the first matrix --
 * the second matrix of a pair counts from M*K*2 --, destination byte offset
 * into the CTA's ring, bytes) triples.  Returns the count (host only). */
long ws_debug_gemv_copies(int M, int K, int B, int nmat, int allow_split, int cta,
                          long long *triples, long max_triples);
/* The same for packed 4-bit rows (source offsets into [nmat][M] rows of
 * ws_q4_row_bytes(K) bytes), for the CUDA-core kernel (mma = 0) or the
 * tensor-core one (mma = 1: bf16 x for one matrix, RMSNorm + SwiGLU for a
 * pair); also returns the schedule in *sched (if given); -1 when the launch
 * would not take that kernel. */
long ws_debug_gemv_copies_q4(int M, int K, int B, int nmat, int cta, int mma,
                             long long *triples, long max_triples, ws_gemv_schedule *sched);

/* Read-only streaming kernel over [ptr, ptr + bytes): a read-roofline probe.
 * Writes one checksum per CTA into sink (uint32 [blocks]). */
ws_status ws_read_probe(const void *ptr, size_t bytes, int blocks, uint32_t *sink,
                        ws_stream_t stream);
/* An empty kernel (touch = 0), or one that makes one global-memory round trip
 * (touch = 1), for the launch-latency floor. */
ws_status ws_empty_probe(int touch, const uint32_t *ptr, uint32_t *sink, ws_stream_t stream);

/* Test hook for the bounded waits: one CTA waits on an mbarrier that nothing
 * arrives on, for timeout_ns, then records the time-out in the device error
 * flag and returns. */
ws_status ws_test_bounded_wait(unsigned long long timeout_ns, ws_stream_t stream);

const char *ws_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WSGEMV_H */
