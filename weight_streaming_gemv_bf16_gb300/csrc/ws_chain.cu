// ws_chain.cu -- the chain executor: a block list turned into GEMV ops,
// captured as one CUDA graph and replayed once per decode step.
//
//  * Ops run on the main branch in block order.  Between consecutive ops the
//    launch carries a programmatic (PDL) edge, so op i+1's CTAs start
//    streaming their weights into shared memory while op i finishes; every
//    op reads the previous op's results only after griddepcontrol.wait.
//  * While op i runs, a side branch forked just before it prefetches the
//    weights of op j = i + distance into L2 with that op's plan; the side
//    branch joins the main branch at the end of the graph ("Making small
//    PyTorch ops faster on a laptop GPU", "Prefetching the next layer while
//    this one runs").  A prefetch only reads, so outputs are bit-identical
//    with and without it.
//  * Plans are measured, not predicted: for each distinct op shape the tuner
//    times a probe chain of (op i, op j) pairs on throwaway weights with and
//    without each candidate plan, in interleaved pairs, and keeps the best
//    plan only if the 95% confidence interval of its relative gain clears the
//    threshold; otherwise the op gets no prefetch ("Measuring instead of
//    predicting").
//  * A decoy mode aims every prefetch at the wrong op (same traffic, no
//    benefit) as the control experiment of the same page.
#include <cuda_runtime.h>

#include <algorithm>
#include <initializer_list>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <utility>
#include <vector>

#include "wsgemv.h"
#include "ws_common.cuh"

using namespace ws;

namespace ws {
// decode attention on the stream (ws_attention.cu); pdl: as a programmatic
// dependent of the previous kernel
ws_status decode_attention(const float* q, const float* k_new, const float* v_new,
                           void* k_cache, void* v_cache, const int32_t* pos, float* out_f32,
                           void* out_bf16, int B, int n_heads, int n_kv_heads, int head_dim,
                           int s_max, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream, bool pdl);
}  // namespace ws

namespace {

enum OpKind { OP_QKV = 0, OP_WO = 1, OP_GATEUP = 2, OP_WD = 3, OP_HEAD = 4, OP_MLP = 5 };

struct ChainOp {
  GemvParams p;
  int kind;
  int block;        // index in the block list
  int trace_block;  // Qwen block whose h is traced after this op, or -1
  const void* trace_src = nullptr;  // the whole batch's output that the trace copies
  std::vector<std::pair<const void*, size_t>> reads;  // weight ranges
  int attn_call = -1;  // decode attention launched right after this op (QKV), or -1
  size_t bytes;     // algorithmic weight bytes
  std::string shape;
  size_t ws_off, ws_bytes;
  ws_prefetch_plan plan;
  float gain_lo, gain_mean;
};

bool al16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

const ws_prefetch_plan kNoPlan = {0, 0, 0, WS_PREFETCH_NONE};

std::string shape_key(const GemvParams& p) {
  char buf[256];
  int n = snprintf(buf, sizeof buf, "nm%d K%d B%d pro%d epi%d", p.nmat, p.K, p.B, p.prologue,
                   p.epilogue);
  for (int s = 0; s < p.nseg && n < (int)sizeof buf; ++s)
    n += snprintf(buf + n, sizeof buf - n, " M%d", p.seg[s].M);
  return std::string(buf);
}

// Two-sided 95% Student t quantile, rounded up (conservative) for df between
// tabulated values.
double t975(int df) {
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

}  // namespace

struct ws_chain {
  ws_chain_opts o;
  std::vector<ws_block_desc> blocks;
  std::vector<ChainOp> ops;
  int device = 0;
  int n_qwen = 0, n_mlp = 0, n_head = 0;
  void* ws = nullptr;
  size_t ws_total = 0;
  void* s_buf = nullptr;
  float* qkv_scratch = nullptr;
  void* pp[2] = {nullptr, nullptr};
  cudaStream_t side = nullptr;
  cudaStream_t cap = nullptr;  // graphs are captured here, launched on the caller's stream
  std::vector<cudaEvent_t> fork_ev;
  cudaEvent_t join_ev = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  // ws_chain_step_host's graph: the input copies, the step and the result
  // copy for one set of host buffers (host_key), captured on first use
  cudaGraphExec_t host_exec = nullptr;
  const void* host_key[3] = {nullptr, nullptr, nullptr};
  std::vector<const void*> attn_dev;
  // decode attention inside the chain: per Qwen block its q, k, v (the QKV
  // op's fp32 outputs) and caches; the bf16 output feeds Wo
  struct AttnCall {
    const float *q, *k, *v;
    void *k_cache, *v_cache;
  };
  std::vector<AttnCall> attn_calls;
  void* attn_buf = nullptr;
  void* attn_ws = nullptr;
  size_t attn_ws_bytes = 0;
  int32_t* idx = nullptr;
  // persistent mode: all ops in one cooperative kernel per step
  bool persistent = false;
  PersistParams persist;
  // diagnostics: per-CTA, per-op stamps of the graph-of-launches mode
  unsigned long long* dbg_stamps = nullptr;
  GemvParams* d_ops = nullptr;
  unsigned* d_bar = nullptr;
};

static void free_chain_buffers(ws_chain* c) {
  if (c->exec) cudaGraphExecDestroy(c->exec);
  if (c->host_exec) cudaGraphExecDestroy(c->host_exec);
  if (c->graph) cudaGraphDestroy(c->graph);
  for (cudaEvent_t e : c->fork_ev)
    if (e) cudaEventDestroy(e);
  if (c->join_ev) cudaEventDestroy(c->join_ev);
  if (c->side) cudaStreamDestroy(c->side);
  if (c->cap) cudaStreamDestroy(c->cap);
  if (c->ws) cudaFree(c->ws);
  if (c->s_buf) cudaFree(c->s_buf);
  if (c->qkv_scratch) cudaFree(c->qkv_scratch);
  if (c->attn_buf) cudaFree(c->attn_buf);
  if (c->attn_ws) cudaFree(c->attn_ws);
  for (void* q : c->pp)
    if (q) cudaFree(q);
  c->exec = nullptr;
  c->host_exec = nullptr;
  c->graph = nullptr;
  c->fork_ev.clear();
  c->join_ev = nullptr;
  c->side = nullptr;
  c->cap = nullptr;
  c->ws = c->s_buf = nullptr;
  c->qkv_scratch = nullptr;
  c->pp[0] = c->pp[1] = nullptr;
  if (c->d_ops) cudaFree(c->d_ops);
  if (c->d_bar) cudaFree(c->d_bar);
  c->d_ops = nullptr;
  c->d_bar = nullptr;
}

// Bytes of one trace slot: a Qwen block's fp32 residual [B][H], or an MLP
// block's bf16 output [B][w].
static size_t trace_bytes(const ws_chain* c) {
  return (size_t)c->o.batch * c->o.hidden * (c->n_mlp ? 2 : 4);
}

// Point a launch planned for the whole batch at batch rows b0 .. b0 + p.B - 1
// of its activations and outputs (all row-major [B][...]).
static void tile_rows(GemvParams& p, int b0) {
  const size_t xb = p.x_dtype == DT_F32 ? 4 : 2;
  p.x = static_cast<const char*>(p.x) + (size_t)b0 * p.K * xb;
  const bool f32_out =
      p.epilogue == EPI_F32 || p.epilogue == EPI_RESID || p.epilogue == EPI_ARGMAX;
  for (int s = 0; s < p.nseg; ++s)
    if (p.seg[s].out)
      p.seg[s].out = static_cast<char*>(p.seg[s].out) + (size_t)b0 * p.seg[s].M * (f32_out ? 4 : 2);
  if (p.res_in) p.res_in += (size_t)b0 * p.seg[0].M;
  if (p.argmax_idx) p.argmax_idx += b0;
  if (p.logits) p.logits += (size_t)b0 * p.seg[0].M;
}

static ws_status build_ops(ws_chain* c) {
  const ws_chain_opts& o = c->o;
  const int B = o.batch;
  const int H = o.hidden;
  char why[256];
  // scratch owned by the chain
  if (c->n_qwen > 0) {
    if (cudaMalloc(&c->s_buf, (size_t)B * o.inter * 2) != cudaSuccess) return WS_ERR_NOMEM;
    bool need_qkv = false;
    for (const ws_block_desc& d : c->blocks)
      if (d.kind == WS_BLOCK_QWEN && (!d.u.qwen.q || !d.u.qwen.k || !d.u.qwen.v)) need_qkv = true;
    if (o.attention) {
      c->attn_ws_bytes =
          ws_attention_workspace_bytes(B, H / 128, o.kv_dim / 128, 128, o.s_max);
      if (cudaMalloc(&c->attn_buf, (size_t)B * H * 2) != cudaSuccess ||
          cudaMalloc(&c->attn_ws, c->attn_ws_bytes) != cudaSuccess ||
          cudaMemset(c->attn_ws, 0, c->attn_ws_bytes) != cudaSuccess)
        return WS_ERR_NOMEM;
    }
    if (need_qkv &&
        cudaMalloc((void**)&c->qkv_scratch, (size_t)B * (H + 2 * o.kv_dim) * 4) != cudaSuccess)
      return WS_ERR_NOMEM;
  }
  if (c->n_mlp > 1 && !o.h_trace) {
    for (int i = 0; i < 2; ++i)
      if (cudaMalloc(&c->pp[i], (size_t)B * H * 2) != cudaSuccess) return WS_ERR_NOMEM;
  }

  int qwen_seen = 0, mlp_seen = 0;
  for (int bi = 0; bi < (int)c->blocks.size(); ++bi) {
    const ws_block_desc& d = c->blocks[bi];
    if (d.kind == WS_BLOCK_QWEN) {
      const ws_qwen_block& q = d.u.qwen;
      const float* h_src = qwen_seen == 0 ? o.h_in : o.h_out;
      float* qo = q.q ? q.q : c->qkv_scratch;
      float* ko = q.k ? q.k : c->qkv_scratch + (size_t)B * H;
      float* vo = q.v ? q.v : c->qkv_scratch + (size_t)B * (H + o.kv_dim);
      // QKV with the first RMSNorm
      ChainOp op{};
      init_gemv_params(op.p, H, B);
      op.p.nseg = 3;
      const void* Ws[3] = {q.Wq, q.Wk, q.Wv};
      float* outs[3] = {qo, ko, vo};
      const int Ms[3] = {H, o.kv_dim, o.kv_dim};
      int base = 0;
      for (int s = 0; s < 3; ++s) {
        op.p.seg[s].W0 = static_cast<const uint16_t*>(Ws[s]);
        op.p.seg[s].out = outs[s];
        op.p.seg[s].M = Ms[s];
        op.p.seg[s].row_base = base;
        base += Ms[s];
        op.reads.push_back({Ws[s], (size_t)Ms[s] * H * 2});
      }
      if (o.attention) {
        op.attn_call = (int)c->attn_calls.size();
        c->attn_calls.push_back({qo, ko, vo, q.k_cache, q.v_cache});
      }
      op.p.x = h_src;
      op.p.x_dtype = DT_F32;
      op.p.prologue = PRO_RMSNORM;
      op.p.gamma = static_cast<const uint16_t*>(q.gamma1);
      op.p.eps = o.eps;
      op.p.epilogue = EPI_F32;
      op.kind = OP_QKV;
      c->ops.push_back(op);
      // Wo with the residual add
      ChainOp wo{};
      init_gemv_params(wo.p, H, B);
      wo.p.nseg = 1;
      wo.p.seg[0].W0 = static_cast<const uint16_t*>(q.Wo);
      wo.p.seg[0].out = o.h_out;
      wo.p.seg[0].M = H;
      wo.p.x = o.attention ? c->attn_buf : q.attn;
      wo.p.x_dtype = DT_BF16;
      wo.p.prologue = PRO_NONE;
      wo.p.epilogue = EPI_RESID;
      wo.p.res_in = h_src;
      wo.reads.push_back({q.Wo, (size_t)H * H * 2});
      wo.kind = OP_WO;
      c->ops.push_back(wo);
      // gate/up with the second RMSNorm and the SwiGLU
      ChainOp gu{};
      init_gemv_params(gu.p, H, B);
      gu.p.nseg = 1;
      gu.p.nmat = 2;
      gu.p.seg[0].W0 = static_cast<const uint16_t*>(q.Wg);
      gu.p.seg[0].W1 = static_cast<const uint16_t*>(q.Wu);
      gu.p.seg[0].out = c->s_buf;
      gu.p.seg[0].M = o.inter;
      gu.p.x = o.h_out;
      gu.p.x_dtype = DT_F32;
      gu.p.prologue = PRO_RMSNORM;
      gu.p.gamma = static_cast<const uint16_t*>(q.gamma2);
      gu.p.eps = o.eps;
      gu.p.epilogue = EPI_SWIGLU;
      gu.reads.push_back({q.Wg, (size_t)o.inter * H * 2});
      gu.reads.push_back({q.Wu, (size_t)o.inter * H * 2});
      gu.kind = OP_GATEUP;
      c->ops.push_back(gu);
      // Wd with the residual add
      ChainOp wd{};
      init_gemv_params(wd.p, o.inter, B);
      wd.p.nseg = 1;
      wd.p.seg[0].W0 = static_cast<const uint16_t*>(q.Wd);
      wd.p.seg[0].out = o.h_out;
      wd.p.seg[0].M = H;
      wd.p.x = c->s_buf;
      wd.p.x_dtype = DT_BF16;
      wd.p.prologue = PRO_NONE;
      wd.p.epilogue = EPI_RESID;
      wd.p.res_in = nullptr;
      wd.reads.push_back({q.Wd, (size_t)H * o.inter * 2});
      wd.kind = OP_WD;
      wd.trace_block = qwen_seen;
      wd.trace_src = o.h_out;
      c->ops.push_back(wd);
      for (size_t k = c->ops.size() - 4; k < c->ops.size(); ++k) {
        c->ops[k].block = bi;
        if (c->ops[k].kind != OP_WD) c->ops[k].trace_block = -1;
      }
      if (!o.attention) c->attn_dev.push_back(q.attn);
      ++qwen_seen;
    } else if (d.kind == WS_BLOCK_MLP) {
      const ws_mlp_block& m = d.u.mlp;
      const int w = H;
      // with a trace every block but the last writes its output straight
      // into its trace slot (no copy, so every op boundary keeps its
      // programmatic edge) and the next block reads it there
      const size_t tb = trace_bytes(c);
      auto slot = [&](int i) -> void* {
        return o.h_trace ? static_cast<void*>(reinterpret_cast<char*>(o.h_trace) + (size_t)i * tb)
                         : c->pp[i % 2];
      };
      const void* xin = mlp_seen == 0 ? o.x_in : slot(mlp_seen - 1);
      void* yout = mlp_seen == c->n_mlp - 1 ? o.y_out : slot(mlp_seen);
      ChainOp op{};
      init_gemv_params(op.p, w, B);
      op.p.nseg = 1;
      op.p.seg[0].W0 = static_cast<const uint16_t*>(m.W);
      op.p.seg[0].out = yout;
      op.p.seg[0].M = w;
      op.p.x = xin;
      op.p.x_dtype = DT_BF16;
      op.p.prologue = PRO_LAYERNORM;
      op.p.gamma = static_cast<const uint16_t*>(m.gamma);
      op.p.beta = static_cast<const uint16_t*>(m.beta);
      op.p.eps = o.eps;
      op.p.epilogue = EPI_BIAS_GELU;
      op.p.bias = static_cast<const uint16_t*>(m.bias);
      op.reads.push_back({m.W, (size_t)w * w * 2});
      op.kind = OP_MLP;
      op.block = bi;
      // only the last block's output is copied into the trace
      op.trace_block = (o.h_trace && mlp_seen == c->n_mlp - 1) ? mlp_seen : -1;
      op.trace_src = yout;
      const size_t bw = (size_t)mlp_seen * B * w;
      if (o.mlp_ln) op.p.ln_out = static_cast<uint16_t*>(o.mlp_ln) + bw;
      if (o.mlp_pre) op.p.pre_out = static_cast<uint16_t*>(o.mlp_pre) + bw;
      if (o.mlp_gelu_grad) op.p.gelu_grad = o.mlp_gelu_grad + bw;
      if (o.mlp_ln_stats) op.p.ln_stats = o.mlp_ln_stats + (size_t)mlp_seen * B * 2;
      c->ops.push_back(op);
      ++mlp_seen;
    } else {
      const ws_head_block& hb = d.u.head;
      ChainOp op{};
      init_gemv_params(op.p, H, B);
      op.p.nseg = 1;
      op.p.seg[0].W0 = static_cast<const uint16_t*>(hb.W);
      op.p.seg[0].out = hb.logits;
      op.p.seg[0].M = o.vocab;
      op.p.x = c->n_qwen > 0 ? (const void*)o.h_out : (const void*)o.h_in;
      op.p.x_dtype = DT_F32;
      op.p.prologue = PRO_RMSNORM;
      op.p.gamma = static_cast<const uint16_t*>(hb.gamma);
      op.p.eps = o.eps;
      op.p.epilogue = EPI_ARGMAX;
      op.p.argmax_idx = hb.idx;
      op.p.logits = hb.logits;
      op.reads.push_back({hb.W, (size_t)o.vocab * H * 2});
      op.kind = OP_HEAD;
      op.block = bi;
      op.trace_block = -1;
      c->idx = hb.idx;
      c->ops.push_back(op);
    }
  }

  // 4-bit weights: every op streams packed rows (q4_prefix(K) bytes a row)
  if (o.weight_format == WS_WEIGHTS_Q4) {
    for (auto& op : c->ops) {
      op.p.wfmt = WF_Q4;
      for (auto& r : op.reads) r.second = r.second / ((size_t)2 * op.p.K) * q4_prefix(op.p.K);
    }
  }

  // batches above the kernels' batch tile: every op runs once per tile of
  // kMaxBatch rows, tiles of one op back to back (rows are independent, so
  // each launch sees its tile's rows of every activation and output); all
  // but the last tile stream the weights with the normal L2 policy, so the
  // next tile finds what still fits in L2
  if (B > kMaxBatch) {
    const int nt = (B + kMaxBatch - 1) / kMaxBatch;
    std::vector<ChainOp> tiled;
    for (const ChainOp& op : c->ops)
      for (int t = 0; t < nt; ++t) {
        ChainOp s = op;
        const int b0 = t * kMaxBatch;
        s.p.B = std::min(kMaxBatch, B - b0);
        tile_rows(s.p, b0);
        if (t != nt - 1) {
          s.trace_block = -1;
          s.p.evict_first = 0;
        }
        tiled.push_back(s);
      }
    c->ops.swap(tiled);
  }

  // persistent mode when asked for and every op fits its stage layout
  c->persistent = false;
  if (o.persistent && B <= 4 && !o.mlp_gelu_grad && !o.mlp_ln_stats && !o.mlp_ln && !o.mlp_pre) {
    int kmax = 8;
    for (ChainOp& op : c->ops) kmax = op.p.K > kmax ? op.p.K : kmax;
    const int ring = persistent_ring_bytes(B, kmax);
    bool ok = ring > 0;
    for (ChainOp& op : c->ops)
      if (ok && !plan_gemv_persistent(op.p, ring, why, sizeof why)) ok = false;
    if (ok) {
      // the shared-memory layout must fit too; otherwise run op by op
      std::vector<GemvParams> probe_ops;
      for (ChainOp& op : c->ops) probe_ops.push_back(op.p);
      PersistParams probe;
      ok = plan_persistent(probe, probe_ops.data(), (int)probe_ops.size(), B, why, sizeof why);
    }
    c->persistent = ok;
  }
  // schedules and one zeroed workspace with a slice per op
  size_t total = 0;
  for (ChainOp& op : c->ops) {
    if (!c->persistent && !plan_gemv(op.p, op.kind == OP_HEAD ? -1 : 0, why, sizeof why)) {
      set_error("op %d: %s", (int)(&op - &c->ops[0]), why);
      return WS_ERR_SHAPE;
    }
    op.ws_off = total;
    op.ws_bytes = workspace_layout(op.p, nullptr, nullptr, nullptr, nullptr, nullptr);
    total += (op.ws_bytes + 255) / 256 * 256;
    op.bytes = 0;
    for (auto& r : op.reads) op.bytes += r.second;
    op.shape = shape_key(op.p);
    op.plan = kNoPlan;
    op.gain_lo = op.gain_mean = 0.f;
  }
  c->ws_total = total;
  if (total) {
    if (cudaMalloc(&c->ws, total) != cudaSuccess) return WS_ERR_NOMEM;
    if (cudaMemset(c->ws, 0, total) != cudaSuccess) return WS_ERR_CUDA;
  }
  for (ChainOp& op : c->ops) {
    if (op.ws_bytes && !bind_workspace(op.p, static_cast<char*>(c->ws) + op.ws_off, op.ws_bytes)) {
      set_error("internal: workspace binding failed");
      return WS_ERR_ARG;
    }
    if (!c->persistent && !prepare_gemv(op.p)) {
      set_error("could not configure the GEMV kernel");
      return WS_ERR_CUDA;
    }
  }
  if (c->persistent) {
    // every op becomes one phase of the persistent kernel; the h trace is
    // written by the kernel itself after each block's last op
    std::vector<GemvParams> host_ops;
    for (ChainOp& op : c->ops) {
      op.p.trace_out =
          (o.h_trace && op.trace_block >= 0)
              ? reinterpret_cast<float*>(reinterpret_cast<char*>(o.h_trace) +
                                         (size_t)op.trace_block * trace_bytes(c))
              : nullptr;
      host_ops.push_back(op.p);
    }
    const int n = (int)host_ops.size();
    if (!plan_persistent(c->persist, host_ops.data(), n, B, why, sizeof why)) {
      set_error("%s", why);
      return WS_ERR_SHAPE;
    }
    if (cudaMalloc((void**)&c->d_ops, sizeof(GemvParams) * n) != cudaSuccess ||
        cudaMalloc((void**)&c->d_bar, sizeof(unsigned) * (n + 1)) != cudaSuccess)
      return WS_ERR_NOMEM;
    if (cudaMemcpy(c->d_ops, host_ops.data(), sizeof(GemvParams) * n, cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemset(c->d_bar, 0, sizeof(unsigned) * (n + 1)) != cudaSuccess)
      return WS_ERR_CUDA;
    c->persist.ops = c->d_ops;
    c->persist.bar = c->d_bar;
    if (!prepare_persistent(c->persist.BT)) {
      set_error("could not configure the persistent chain kernel");
      return WS_ERR_CUDA;
    }
    return WS_OK;
  }
  if (o.prefetch == 2)
    for (ChainOp& op : c->ops) op.plan = o.fixed_plan;
  return WS_OK;
}

static int decoy_target(const ws_chain* c, int j) {
  const int n = (int)c->ops.size();
  const int want = (j + n / 2) % n;
  int best = -1, best_d = 1 << 30;
  for (int k = 0; k < n; ++k) {
    if (k == j || c->ops[k].shape != c->ops[j].shape) continue;
    const int d = std::abs(k - want);
    if (d < best_d) {
      best_d = d;
      best = k;
    }
  }
  return best >= 0 ? best : (want == j ? (j + 1) % n : want);
}

// Enqueue the ops (optionally with prefetches) on `stream`; used inside
// capture.  `plans` and `reads` may differ from the chain's own (tuner).
static ws_status enqueue_ops(ws_chain* c, const std::vector<GemvParams>& ps,
                             const std::vector<std::vector<std::pair<const void*, size_t>>>& reads,
                             const std::vector<ws_prefetch_plan>& plans, int distance,
                             bool decoy, cudaStream_t stream, const std::vector<int>& trace,
                             bool use_pdl, bool after_kernel = false,
                             bool* ends_kernel = nullptr) {
  const int n = (int)ps.size();
  // after_kernel: the node before the first op is a kernel (the copy of a
  // host step's inputs), so the first op may start as its dependent
  bool forked = false, prev_kernel = after_kernel;
  for (int i = 0; i < n; ++i) {
    const int j = i + distance;
    if (j < n && plans[j].mode != WS_PREFETCH_NONE) {
      const int tgt = decoy ? decoy_target(c, j) : j;
      if (cudaEventRecord(c->fork_ev[i], stream) != cudaSuccess) return WS_ERR_CUDA;
      if (cudaStreamWaitEvent(c->side, c->fork_ev[i], 0) != cudaSuccess) return WS_ERR_CUDA;
      for (auto& r : reads[tgt]) {
        const ws_status s = ws_l2_prefetch(r.first, r.second, plans[j], c->side);
        if (s != WS_OK) return s;
      }
      forked = true;
    }
    const cudaError_t e = launch_gemv(ps[i], stream, use_pdl && prev_kernel);
    if (e != cudaSuccess) {
      set_error("launch of op %d failed: %s", i, cudaGetErrorString(e));
      return WS_ERR_CUDA;
    }
    prev_kernel = true;
    if (ps.size() == c->ops.size() && c->ops[i].attn_call >= 0) {
      // the block's decode attention on the QKV op's outputs (split-KV, the
      // key-value append at pos, positions read on the device)
      const ws_chain::AttnCall& a = c->attn_calls[c->ops[i].attn_call];
      const ws_chain_opts& o = c->o;
      const ws_status s = ws::decode_attention(
          a.q, a.k, a.v, a.k_cache, a.v_cache, o.pos, nullptr, c->attn_buf, o.batch,
          o.hidden / 128, o.kv_dim / 128, 128, o.s_max, c->attn_ws, c->attn_ws_bytes, stream,
          use_pdl);
      if (s != WS_OK) return s;
    }
    if (!trace.empty() && trace[i] >= 0) {
      // the whole batch's output (a tiled op's own pointer starts at its tile)
      const size_t bytes = trace_bytes(c);
      if (cudaMemcpyAsync(reinterpret_cast<char*>(c->o.h_trace) + (size_t)trace[i] * bytes,
                          c->ops[i].trace_src, bytes, cudaMemcpyDeviceToDevice,
                          stream) != cudaSuccess)
        return WS_ERR_CUDA;
      prev_kernel = false;
    }
  }
  if (forked) {
    if (cudaEventRecord(c->join_ev, c->side) != cudaSuccess) return WS_ERR_CUDA;
    if (cudaStreamWaitEvent(stream, c->join_ev, 0) != cudaSuccess) return WS_ERR_CUDA;
  }
  if (ends_kernel) *ends_kernel = prev_kernel && !forked;
  return WS_OK;
}

namespace ws {
// word copies between device-accessible buffers (ws_misc.cu)
cudaError_t launch_copy_words(void* d0, const void* s0, size_t b0, void* d1, const void* s1,
                              size_t b1, cudaStream_t stream, bool pdl);
}  // namespace ws

// Host buffers of one ws_chain_step_host graph, and their device aliases
// where the buffers are pinned host memory mapped into the device's address
// space (else null: the copies then go through the copy engines).
struct HostIO {
  const void* in;
  const void* attn;
  void* out;
  const void* in_d = nullptr;
  const void* attn_d = nullptr;
  void* out_d = nullptr;
};

// The device alias of a pinned, mapped host buffer (4-byte aligned), or null.
static void* mapped_alias(const void* p) {
  if (!p || ((uintptr_t)p & 3u)) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  return ((uintptr_t)a.devicePointer & 3u) ? nullptr : a.devicePointer;
}

static ws_status enqueue_host_in(ws_chain* c, const HostIO& io, cudaStream_t st,
                                 bool* by_kernel);
static ws_status enqueue_host_out(ws_chain* c, const HostIO& io, cudaStream_t st, bool pdl);

// Capture the ops (with prefetches and trace copies) into *out; with io, the
// copies of ws_chain_step_host's inputs come first and its result copy last.
static ws_status capture_graph(ws_chain* c, const std::vector<GemvParams>& ps,
                               const std::vector<std::vector<std::pair<const void*, size_t>>>& reads,
                               const std::vector<ws_prefetch_plan>& plans, bool decoy,
                               const std::vector<int>& trace, cudaGraphExec_t* out,
                               const HostIO* io = nullptr) {
  cudaGraph_t g = nullptr;
  cudaStream_t stream = c->cap;
  if (cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    set_error("cudaStreamBeginCapture failed");
    return WS_ERR_CUDA;
  }
  // with a host step's word copies, the first op starts as a programmatic
  // dependent of the input copy, and the output copy of the last op
  bool in_kernel = false, out_pdl = false;
  ws_status s = io ? enqueue_host_in(c, *io, stream, &in_kernel) : WS_OK;
  if (s == WS_OK)
    s = c->persistent ? (launch_persistent(c->persist, stream) == cudaSuccess ? WS_OK : WS_ERR_CUDA)
                      : enqueue_ops(c, ps, reads, plans, c->o.distance, decoy, stream, trace,
                                    c->o.use_pdl != 0, in_kernel && c->o.use_pdl != 0,
                                    &out_pdl);
  if (s == WS_OK && io)
    s = enqueue_host_out(c, *io, stream, out_pdl && !c->persistent && c->o.use_pdl != 0);
  const cudaError_t e = cudaStreamEndCapture(stream, &g);
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

static std::vector<GemvParams> chain_params(const ws_chain* c) {
  std::vector<GemvParams> ps;
  for (const ChainOp& op : c->ops) ps.push_back(op.p);
  if (c->dbg_stamps) {
    const int nops = (int)ps.size();
    for (int i = 0; i < nops; ++i) {
      ps[i].stamps = c->dbg_stamps + (size_t)i * kStampsPerOp;
      ps[i].stamp_stride = nops * kStampsPerOp;
    }
  }
  return ps;
}

static std::vector<std::vector<std::pair<const void*, size_t>>> chain_reads(const ws_chain* c) {
  std::vector<std::vector<std::pair<const void*, size_t>>> r;
  for (const ChainOp& op : c->ops) r.push_back(op.reads);
  return r;
}

// The copies of one step's inputs from host buffers to the chain's device
// inputs (Qwen: fp32 h and, if given, the bf16 attention stand-ins of every
// block; MLP: bf16 x), and of its result back.
static ws_status enqueue_host_in(ws_chain* c, const HostIO& io, cudaStream_t st,
                                 bool* by_kernel) {
  const int B = c->o.batch, H = c->o.hidden;
  *by_kernel = false;
  if (c->n_mlp) {
    if (io.in_d) {  // one word-copy launch reading the mapped host buffer
      *by_kernel = true;
      return launch_copy_words(const_cast<void*>(c->o.x_in), io.in_d, (size_t)B * H * 2, nullptr,
                               nullptr, 0, st, false) == cudaSuccess
                 ? WS_OK
                 : WS_ERR_CUDA;
    }
    return cudaMemcpyAsync(const_cast<void*>(c->o.x_in), io.in, (size_t)B * H * 2,
                           cudaMemcpyHostToDevice, st) == cudaSuccess
               ? WS_OK
               : WS_ERR_CUDA;
  }
  const size_t blk = (size_t)B * H * 2;
  bool contiguous = !c->attn_dev.empty();
  for (size_t l = 0; l < c->attn_dev.size(); ++l)
    if (static_cast<const char*>(c->attn_dev[l]) !=
        static_cast<const char*>(c->attn_dev[0]) + l * blk)
      contiguous = false;
  const bool with_attn = io.attn && !c->attn_dev.empty();
  if (io.in_d && (!with_attn || (io.attn_d && contiguous))) {
    // h and every block's attention input in one word-copy launch
    *by_kernel = true;
    return launch_copy_words(const_cast<float*>(c->o.h_in), io.in_d, (size_t)B * H * 4,
                             with_attn ? const_cast<void*>(c->attn_dev[0]) : nullptr,
                             with_attn ? io.attn_d : nullptr,
                             with_attn ? blk * c->attn_dev.size() : 0, st,
                             false) == cudaSuccess
               ? WS_OK
               : WS_ERR_CUDA;
  }
  if (cudaMemcpyAsync(const_cast<float*>(c->o.h_in), io.in, (size_t)B * H * 4,
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return WS_ERR_CUDA;
  if (with_attn) {
    if (contiguous)
      return cudaMemcpyAsync(const_cast<void*>(c->attn_dev[0]), io.attn,
                             blk * c->attn_dev.size(), cudaMemcpyHostToDevice, st) == cudaSuccess
                 ? WS_OK
                 : WS_ERR_CUDA;
    for (size_t l = 0; l < c->attn_dev.size(); ++l)
      if (cudaMemcpyAsync(const_cast<void*>(c->attn_dev[l]),
                          static_cast<const char*>(io.attn) + l * blk, blk,
                          cudaMemcpyHostToDevice, st) != cudaSuccess)
        return WS_ERR_CUDA;
  }
  return WS_OK;
}

static ws_status enqueue_host_out(ws_chain* c, const HostIO& io, cudaStream_t st, bool pdl) {
  const int B = c->o.batch, H = c->o.hidden;
  const void* src;
  size_t bytes;
  if (c->n_mlp) {
    src = c->o.y_out;
    bytes = (size_t)B * H * 2;
  } else if (c->idx) {
    src = c->idx;
    bytes = (size_t)B * 4;
  } else {
    src = c->o.h_out;
    bytes = (size_t)B * H * 4;
  }
  if (io.out_d)  // written through the mapped host buffer by one word-copy launch
    return launch_copy_words(io.out_d, src, bytes, nullptr, nullptr, 0, st, pdl) == cudaSuccess
               ? WS_OK
               : WS_ERR_CUDA;
  return cudaMemcpyAsync(io.out, src, bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess
             ? WS_OK
             : WS_ERR_CUDA;
}

extern "C" {

ws_status ws_chain_create(const ws_block_desc* blocks, int n, const ws_chain_opts* opts,
                          ws_chain** out) {
  if (!blocks || n <= 0 || !opts || !out) {
    set_error("bad arguments");
    return WS_ERR_ARG;
  }
  *out = nullptr;
  const ws_chain_opts& o = *opts;
  if (o.batch < 1 || o.batch > kMaxChainBatch || o.hidden <= 0 || o.hidden % 8 != 0) {
    set_error("bad batch %d or hidden %d", o.batch, o.hidden);
    return WS_ERR_SHAPE;
  }
  if (o.batch > kMaxBatch &&
      (o.attention || o.weight_format != WS_WEIGHTS_BF16 || o.mlp_ln || o.mlp_pre ||
       o.mlp_gelu_grad || o.mlp_ln_stats)) {
    set_error("batch %d > %d runs in batch tiles: bf16 weights, no attention, no training "
              "saves", o.batch, kMaxBatch);
    return WS_ERR_SHAPE;
  }
  if (o.distance < 1 && o.prefetch) {
    set_error("prefetch distance must be >= 1");
    return WS_ERR_ARG;
  }
  int nq = 0, nm = 0, nh = 0;
  for (int i = 0; i < n; ++i) {
    const int k = blocks[i].kind;
    if (k == WS_BLOCK_QWEN) {
      if (nm || nh) {
        set_error("Qwen blocks must come first and cannot mix with MLP blocks");
        return WS_ERR_ARG;
      }
      ++nq;
      const ws_qwen_block& q = blocks[i].u.qwen;
      const void* req[] = {q.gamma1, q.Wq,     q.Wk, q.Wv, q.Wo,
                           q.gamma2, q.Wg,     q.Wu, q.Wd,
                           o.attention ? q.k_cache : q.attn,
                           o.attention ? q.v_cache : q.attn};
      for (const void* r : req)
        if (!r || !al16(r)) {
          set_error("block %d: null or unaligned pointer", i);
          return r ? WS_ERR_ALIGN : WS_ERR_ARG;
        }
      const void* opt[] = {q.q, q.k, q.v};
      for (const void* r : opt)
        if (r && !al16(r)) {
          set_error("block %d: unaligned q/k/v", i);
          return WS_ERR_ALIGN;
        }
    } else if (k == WS_BLOCK_MLP) {
      if (nq || nh) {
        set_error("MLP blocks cannot mix with Qwen or head blocks");
        return WS_ERR_ARG;
      }
      ++nm;
      const ws_mlp_block& m = blocks[i].u.mlp;
      const void* req[] = {m.gamma, m.beta, m.W, m.bias};
      for (const void* r : req)
        if (!r || !al16(r)) {
          set_error("block %d: null or unaligned pointer", i);
          return r ? WS_ERR_ALIGN : WS_ERR_ARG;
        }
    } else if (k == WS_BLOCK_HEAD) {
      if (nh || i != n - 1) {
        set_error("one head block, last");
        return WS_ERR_ARG;
      }
      ++nh;
      const ws_head_block& h = blocks[i].u.head;
      if (!h.gamma || !h.W || !h.idx || !al16(h.gamma) || !al16(h.W) || !al16(h.idx) ||
          (h.logits && !al16(h.logits))) {
        set_error("head: null or unaligned pointer");
        return WS_ERR_ARG;
      }
    } else {
      set_error("block %d: unknown kind %d", i, k);
      return WS_ERR_ARG;
    }
  }
  if (nq && (o.kv_dim <= 0 || o.kv_dim % 8 || o.inter <= 0 || o.inter % 8 || !o.h_in ||
             !o.h_out || !al16(o.h_in) || !al16(o.h_out) || (o.h_trace && !al16(o.h_trace)))) {
    set_error("Qwen chain needs kv_dim, inter (multiples of 8) and aligned h_in, h_out");
    return WS_ERR_ARG;
  }
  if (nm && (!o.x_in || !o.y_out || !al16(o.x_in) || !al16(o.y_out) ||
             (o.h_trace && !al16(o.h_trace)))) {
    set_error("MLP chain needs aligned x_in and y_out");
    return WS_ERR_ARG;
  }
  if (nh && (o.vocab <= 0 || (!nq && (!o.h_in || !al16(o.h_in))))) {
    set_error("head needs vocab > 0 and an input h");
    return WS_ERR_ARG;
  }
  if (o.attention &&
      (!nq || o.hidden % 128 || o.kv_dim % 128 || (o.hidden / 128) % (o.kv_dim / 128) ||
       o.hidden / o.kv_dim > 8 || o.s_max < 64 || o.s_max % 64 || !o.pos || o.persistent)) {
    set_error("attention in the chain: Qwen blocks, heads of 128 (hidden and kv_dim multiples "
              "of 128, at most 8 query heads per key-value head), s_max a multiple of 64, pos, "
              "one launch per op");
    return WS_ERR_ARG;
  }
  if (o.weight_format != WS_WEIGHTS_BF16 && o.weight_format != WS_WEIGHTS_Q4) {
    set_error("unknown weight format %d", o.weight_format);
    return WS_ERR_ARG;
  }
  if (o.weight_format == WS_WEIGHTS_Q4 &&
      (nm || o.batch > 4 || o.persistent || o.hidden % kQ4Group ||
       (nq && o.inter % kQ4Group))) {
    set_error("4-bit weights: Qwen and head blocks, batch <= 4, one launch per op, hidden "
              "and inter multiples of 128");
    return WS_ERR_ARG;
  }

  ws_chain* c = new ws_chain();
  c->o = o;
  if (c->o.tune_pairs < 8) c->o.tune_pairs = 30;
  if (!(c->o.tune_min_gain > 0.f)) c->o.tune_min_gain = 0.01f;
  if (c->o.distance < 1) c->o.distance = 1;
  c->blocks.assign(blocks, blocks + n);
  c->n_qwen = nq;
  c->n_mlp = nm;
  c->n_head = nh;
  cudaGetDevice(&c->device);
  ws_status s = build_ops(c);
  if (s == WS_OK) {
    if (cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) != cudaSuccess) s = WS_ERR_CUDA;
    if (s == WS_OK && cudaStreamCreateWithFlags(&c->cap, cudaStreamNonBlocking) != cudaSuccess)
      s = WS_ERR_CUDA;
    c->fork_ev.assign(c->ops.size(), nullptr);
    for (auto& e : c->fork_ev)
      if (s == WS_OK && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
        s = WS_ERR_CUDA;
    if (s == WS_OK && cudaEventCreateWithFlags(&c->join_ev, cudaEventDisableTiming) != cudaSuccess)
      s = WS_ERR_CUDA;
  }
  if (s != WS_OK) {
    if (s == WS_ERR_NOMEM) set_error("chain buffers could not be allocated");
    free_chain_buffers(c);
    delete c;
    return s;
  }
  *out = c;
  return WS_OK;
}

ws_status ws_chain_tune(ws_chain* c, ws_stream_t stream) {
  if (!c) {
    set_error("null chain");
    return WS_ERR_ARG;
  }
  if (c->o.prefetch != 1 || c->persistent) return WS_OK;
  cudaStream_t st = (cudaStream_t)stream;
  int l2 = 0;
  cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, c->device);
  if (l2 <= 0) l2 = 128 << 20;
  const int dist = c->o.distance;
  const int n = (int)c->ops.size();
  std::map<std::string, int> done;  // shape -> first op j tuned
  std::vector<ws_prefetch_plan> cands;
  const int modes[] = {WS_PREFETCH_L2, WS_PREFETCH_L2_EVICT_LAST, WS_PREFETCH_BULK};
  const int nblk[] = {4, 16, 64};
  for (int m : modes)
    for (int b : nblk) cands.push_back({b, 256, m == WS_PREFETCH_BULK ? 16384 : 128, m});

  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  ws_status status = WS_OK;
  for (int j = dist; j < n && status == WS_OK; ++j) {
    ChainOp& tj = c->ops[j];
    if (done.count(tj.shape)) continue;
    done[tj.shape] = j;
    const ChainOp& ti = c->ops[j - dist];
    const size_t pair_bytes = ti.bytes + tj.bytes;
    int R = (int)((2.0 * l2) / (double)pair_bytes) + 1;
    R = std::max(2, std::min(16, R));

    // throwaway weights, scratch outputs and workspaces for R (i, j) pairs
    std::vector<void*> allocs;
    auto alloc = [&](size_t bytes, int fill) -> void* {
      void* q = nullptr;
      if (cudaMalloc(&q, bytes ? bytes : 16) != cudaSuccess) return nullptr;
      allocs.push_back(q);
      if (cudaMemsetAsync(q, fill, bytes ? bytes : 16, st) != cudaSuccess) return nullptr;
      return q;
    };
    std::vector<GemvParams> ps;
    std::vector<std::vector<std::pair<const void*, size_t>>> reads;
    bool ok = true;
    for (int r = 0; r < R && ok; ++r) {
      const ChainOp* pair_ops[2] = {&ti, &tj};
      for (const ChainOp* t : pair_ops) {
        GemvParams p = t->p;
        std::vector<std::pair<const void*, size_t>> rd;
        // weights: one copy per matrix, same shapes
        for (int s = 0; s < p.nseg && ok; ++s) {
          const size_t wb = (size_t)p.seg[s].M * p.K * 2;
          void* w0 = alloc(wb, 0x3c);
          ok = ok && w0;
          p.seg[s].W0 = static_cast<const uint16_t*>(w0);
          rd.push_back({w0, wb});
          if (p.nmat == 2) {
            void* w1 = alloc(wb, 0x3c);
            ok = ok && w1;
            p.seg[s].W1 = static_cast<const uint16_t*>(w1);
            rd.push_back({w1, wb});
          }
          void* outb = alloc((size_t)p.B * p.seg[s].M * 4, 0);
          ok = ok && outb;
          p.seg[s].out = outb;
          if (p.epilogue == EPI_RESID && p.res_in == nullptr) p.res_in = nullptr;
        }
        if (p.epilogue == EPI_ARGMAX) {
          void* ib = alloc(64, 0);
          ok = ok && ib;
          p.argmax_idx = static_cast<int*>(ib);
          p.logits = p.logits ? static_cast<float*>(p.seg[0].out) : nullptr;
          if (!p.logits) p.seg[0].out = nullptr;
        }
        const size_t wsb = workspace_layout(p, nullptr, nullptr, nullptr, nullptr, nullptr);
        if (wsb) {
          void* wsp = alloc(wsb, 0);
          ok = ok && wsp && bind_workspace(p, wsp, wsb);
        }
        ps.push_back(p);
        reads.push_back(rd);
      }
    }
    if (!ok) {
      for (void* q : allocs) cudaFree(q);
      set_error("tuner: could not allocate throwaway buffers");
      status = WS_ERR_NOMEM;
      break;
    }
    const int np = (int)ps.size();
    // the probe's decoy map is never used (decoy = false)
    std::vector<cudaEvent_t> saved_fork = c->fork_ev;
    std::vector<cudaEvent_t> probe_fork(np, nullptr);
    for (auto& e : probe_fork) cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    c->fork_ev = probe_fork;

    std::vector<ws_prefetch_plan> none(np, kNoPlan);
    cudaGraphExec_t gA = nullptr;
    status = capture_graph(c, ps, reads, none, false, {}, &gA);
    double best_lo = -1e30, best_mean = 0;
    int best_c = -1;
    for (size_t ci = 0; ci < cands.size() && status == WS_OK; ++ci) {
      std::vector<ws_prefetch_plan> pl(np, kNoPlan);
      for (int k = 1; k < np; k += 2) pl[k] = cands[ci];  // prefetch every op j (odd slots)
      cudaGraphExec_t gB = nullptr;
      status = capture_graph(c, ps, reads, pl, false, {}, &gB);
      if (status != WS_OK) break;
      // warm up both
      for (int w = 0; w < 3; ++w) {
        cudaGraphLaunch(gA, st);
        cudaGraphLaunch(gB, st);
      }
      const int pairs = c->o.tune_pairs;
      std::vector<double> gains;
      for (int t = 0; t < pairs; ++t) {
        float ms[2] = {0, 0};
        for (int h = 0; h < 2; ++h) {
          const int which = (t & 1) ? 1 - h : h;  // alternate the order
          cudaEventRecord(e0, st);
          cudaGraphLaunch(which ? gB : gA, st);
          cudaEventRecord(e1, st);
          cudaEventSynchronize(e1);
          cudaEventElapsedTime(&ms[which], e0, e1);
        }
        if (ms[0] > 0) gains.push_back((ms[0] - ms[1]) / ms[0]);
      }
      cudaGraphExecDestroy(gB);
      if (cudaGetLastError() != cudaSuccess) {
        set_error("tuner: a probe replay failed");
        status = WS_ERR_CUDA;
        break;
      }
      const int m = (int)gains.size();
      if (m < 2) continue;
      double mean = 0, var = 0;
      for (double g : gains) mean += g;
      mean /= m;
      for (double g : gains) var += (g - mean) * (g - mean);
      var /= (m - 1);
      const double lo = mean - t975(m - 1) * std::sqrt(var / m);
      if (lo > best_lo) {
        best_lo = lo;
        best_mean = mean;
        best_c = (int)ci;
      }
    }
    if (gA) cudaGraphExecDestroy(gA);
    cudaStreamSynchronize(st);
    for (auto& e : probe_fork) cudaEventDestroy(e);
    c->fork_ev = saved_fork;
    for (void* q : allocs) cudaFree(q);
    if (status != WS_OK) break;
    const bool keep = best_c >= 0 && best_lo > (double)c->o.tune_min_gain;
    for (ChainOp& op : c->ops) {
      if (op.shape != tj.shape) continue;
      op.plan = keep ? cands[best_c] : kNoPlan;
      op.gain_lo = best_c >= 0 ? (float)best_lo : 0.f;
      op.gain_mean = best_c >= 0 ? (float)best_mean : 0.f;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return status;
}

ws_status ws_chain_capture(ws_chain* c, ws_stream_t stream) {
  if (!c) {
    set_error("null chain");
    return WS_ERR_ARG;
  }
  if (c->exec) {
    cudaGraphExecDestroy(c->exec);
    c->exec = nullptr;
  }
  if (c->host_exec) {  // recaptured on its next use, with the new ops and plans
    cudaGraphExecDestroy(c->host_exec);
    c->host_exec = nullptr;
  }
  std::vector<ws_prefetch_plan> plans;
  for (const ChainOp& op : c->ops) plans.push_back(c->o.prefetch ? op.plan : kNoPlan);
  std::vector<int> trace;
  if (c->o.h_trace) {
    for (const ChainOp& op : c->ops) trace.push_back(op.trace_block);
  }
  (void)stream;
  if (c->persistent) {
    cudaGraph_t g = nullptr;
    if (cudaStreamBeginCapture(c->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      set_error("cudaStreamBeginCapture failed");
      return WS_ERR_CUDA;
    }
    const cudaError_t le = launch_persistent(c->persist, c->cap);
    const cudaError_t ce = cudaStreamEndCapture(c->cap, &g);
    if (le != cudaSuccess || ce != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      set_error("capture of the persistent chain failed: %s",
                cudaGetErrorString(le != cudaSuccess ? le : ce));
      cudaGetLastError();
      return WS_ERR_CUDA;
    }
    const cudaError_t ie = cudaGraphInstantiate(&c->exec, g, 0);
    cudaGraphDestroy(g);
    if (ie != cudaSuccess) {
      set_error("graph instantiation failed: %s", cudaGetErrorString(ie));
      return WS_ERR_CUDA;
    }
    return WS_OK;
  }
  return capture_graph(c, chain_params(c), chain_reads(c), plans, c->o.decoy != 0, trace,
                       &c->exec);
}

ws_status ws_chain_run(ws_chain* c, ws_stream_t stream) {
  if (!c) {
    set_error("null chain");
    return WS_ERR_ARG;
  }
  if (!c->exec) {
    set_error("chain not captured");
    return WS_ERR_STATE;
  }
  const cudaError_t e = cudaGraphLaunch(c->exec, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    set_error("graph launch failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

ws_status ws_chain_run_eager(ws_chain* c, ws_stream_t stream) {
  if (!c) {
    set_error("null chain");
    return WS_ERR_ARG;
  }
  if (c->persistent) {
    const cudaError_t e = launch_persistent(c->persist, (cudaStream_t)stream);
    if (e != cudaSuccess) {
      set_error("launch of the persistent chain failed: %s", cudaGetErrorString(e));
      return WS_ERR_CUDA;
    }
    return WS_OK;
  }
  for (size_t i = 0; i < c->ops.size(); ++i) {
    const cudaError_t e = launch_gemv(c->ops[i].p, (cudaStream_t)stream, false);
    if (e != cudaSuccess) {
      set_error("launch of op %zu failed: %s", i, cudaGetErrorString(e));
      return WS_ERR_CUDA;
    }
    if (c->o.h_trace && c->ops[i].trace_block >= 0) {
      const size_t bytes = trace_bytes(c);
      if (cudaMemcpyAsync(reinterpret_cast<char*>(c->o.h_trace) +
                              (size_t)c->ops[i].trace_block * bytes,
                          c->ops[i].trace_src, bytes, cudaMemcpyDeviceToDevice,
                          (cudaStream_t)stream) != cudaSuccess)
        return WS_ERR_CUDA;
    }
  }
  return WS_OK;
}

ws_status ws_chain_step_host(ws_chain* c, const void* in_host, const void* attn_host,
                             void* out_host, ws_stream_t stream) {
  if (!c || !in_host || !out_host) {
    set_error("bad arguments");
    return WS_ERR_ARG;
  }
  if (!c->exec) {
    set_error("chain not captured");
    return WS_ERR_STATE;
  }
  cudaStream_t st = (cudaStream_t)stream;
  HostIO io = {in_host, attn_host, out_host};
  io.in_d = mapped_alias(in_host);
  io.attn_d = mapped_alias(attn_host);
  io.out_d = mapped_alias(out_host);
  // one graph launch per step: the copies in, the step, the copy out.  It is
  // captured for these host buffers on first use (pinned memory; a capture
  // that fails, e.g. on pageable buffers, leaves the copies outside)
  if (c->host_exec && (c->host_key[0] != in_host || c->host_key[1] != attn_host ||
                       c->host_key[2] != out_host)) {
    cudaGraphExecDestroy(c->host_exec);
    c->host_exec = nullptr;
  }
  if (!c->host_exec) {
    std::vector<ws_prefetch_plan> plans;
    for (const ChainOp& op : c->ops) plans.push_back(c->o.prefetch ? op.plan : kNoPlan);
    std::vector<int> trace;
    if (c->o.h_trace && !c->persistent)
      for (const ChainOp& op : c->ops) trace.push_back(op.trace_block);
    if (capture_graph(c, chain_params(c), chain_reads(c), plans, c->o.decoy != 0, trace,
                      &c->host_exec, &io) == WS_OK) {
      c->host_key[0] = in_host;
      c->host_key[1] = attn_host;
      c->host_key[2] = out_host;
    } else {
      c->host_exec = nullptr;
      cudaGetLastError();
    }
  }
  if (c->host_exec) {
    if (cudaGraphLaunch(c->host_exec, st) != cudaSuccess) {
      set_error("graph launch failed");
      return WS_ERR_CUDA;
    }
  } else {
    bool by_kernel = false;
    ws_status s = enqueue_host_in(c, io, st, &by_kernel);
    if (s == WS_OK) s = ws_chain_run(c, stream);
    if (s == WS_OK) s = enqueue_host_out(c, io, st, false);
    if (s != WS_OK) return s;
  }
  const cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    set_error("step failed: %s", cudaGetErrorString(e));
    return WS_ERR_CUDA;
  }
  return WS_OK;
}

int ws_chain_num_ops(const ws_chain* c) { return c ? (int)c->ops.size() : 0; }

int ws_chain_is_persistent(const ws_chain* c) { return c && c->persistent ? 1 : 0; }

ws_status ws_chain_debug_stamps(ws_chain* c, unsigned long long* stamps, size_t n) {
  if (!c) {
    set_error("null chain");
    return WS_ERR_ARG;
  }
  const size_t need = (size_t)ws_chain_grid(c) * c->ops.size() * kStampsPerOp;
  if (stamps && n < need) {
    set_error("stamp buffer too small: need %zu entries", need);
    return WS_ERR_ARG;
  }
  if (c->persistent)
    c->persist.stamps = stamps;
  else
    c->dbg_stamps = stamps;
  return WS_OK;
}

int ws_chain_grid(const ws_chain* c) {
  if (!c) return 0;
  if (c->persistent) return c->persist.grid;
  // every CTA of every op writes its own row: the largest grid of any op
  int g = 0;
  for (const ChainOp& op : c->ops) g = op.p.sc.grid > g ? op.p.sc.grid : g;
  return g;
}

ws_status ws_chain_plans(const ws_chain* c, ws_prefetch_plan* plans, float* gain_lo,
                         float* gain_mean, int n) {
  if (!c || n < 0) {
    set_error("bad arguments");
    return WS_ERR_ARG;
  }
  for (int i = 0; i < n && i < (int)c->ops.size(); ++i) {
    if (plans) plans[i] = c->o.prefetch ? c->ops[i].plan : kNoPlan;
    if (gain_lo) gain_lo[i] = c->ops[i].gain_lo;
    if (gain_mean) gain_mean[i] = c->ops[i].gain_mean;
  }
  return WS_OK;
}

ws_status ws_chain_op_bytes(const ws_chain* c, size_t* bytes, int n) {
  if (!c || !bytes || n < 0) {
    set_error("bad arguments");
    return WS_ERR_ARG;
  }
  for (int i = 0; i < n && i < (int)c->ops.size(); ++i) bytes[i] = c->ops[i].bytes;
  return WS_OK;
}

void ws_chain_destroy(ws_chain* c) {
  if (!c) return;
  free_chain_buffers(c);
  delete c;
}

}  // extern "C"
