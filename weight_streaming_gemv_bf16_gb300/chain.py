"""Assemble decode chains from device tensors and hand them to the C ABI.

Two chain kinds, both replayed as one CUDA graph by the library:
* a Llama-style decode weight chain ("One Token, Kernel by Kernel: A Decode
  Step on a Laptop GPU", Step 1 and "The whole step"): L decoder blocks
  (merged QKV with the first RMSNorm, Wo + residual, gate/up with the second
  RMSNorm and SwiGLU, Wd + residual), then the final RMSNorm, the LM head and
  the argmax;
* an MLP chain of LayerNorm -> Linear -> GELU blocks ("Making small PyTorch
  ops faster on a laptop GPU", "Beyond language models").

Only pointers, sizes and options are marshalled here; the tensors stay owned
by the returned objects.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import binding as wb


@dataclass
class QwenChain:
    chain: wb.Chain
    h_in: torch.Tensor
    h_out: torch.Tensor
    attn: torch.Tensor
    idx: torch.Tensor | None
    logits: torch.Tensor | None
    h_trace: torch.Tensor | None
    qkv: list = field(default_factory=list)

    def run(self, stream=None):
        self.chain.run(stream)


@dataclass
class MlpChain:
    chain: wb.Chain
    x_in: torch.Tensor
    y_out: torch.Tensor
    trace: torch.Tensor | None = None
    gelu_grad: torch.Tensor | None = None
    ln_stats: torch.Tensor | None = None
    ln: torch.Tensor | None = None
    pre: torch.Tensor | None = None

    def run(self, stream=None):
        self.chain.run(stream)


def _opts(B, H, KV, I, V, eps, use_pdl, prefetch, fixed_plan, distance, decoy, tune_pairs,
          min_gain, persistent=False):
    o = wb.ChainOpts()
    o.persistent = 1 if persistent else 0
    o.batch, o.hidden, o.kv_dim, o.inter, o.vocab, o.eps = B, H, KV, I, V, eps
    o.use_pdl = 1 if use_pdl else 0
    o.prefetch = prefetch
    if fixed_plan is not None:
        o.fixed_plan = fixed_plan
    o.distance = distance
    o.decoy = 1 if decoy else 0
    o.tune_pairs = tune_pairs
    o.tune_min_gain = min_gain
    return o


def qwen_chain(blocks, head, attn, h_in, *, eps=1e-6, use_pdl=True, prefetch=0,
               fixed_plan=None, distance=1, decoy=False, trace=False, keep_qkv=False,
               logits=False, tune_pairs=30, min_gain=0.01, persistent=False,
               q4=False, caches=None, pos=None) -> QwenChain:
    """blocks: list of dicts of bf16 device tensors gamma1, Wq, Wk, Wv, Wo, gamma2,
    Wg, Wu, Wd; head: dict gamma_f, Wlm (or None); attn: bf16 [L, B, H];
    h_in: fp32 [B, H].  q4=True: the weight matrices are packed 4-bit rows
    (uint8 [M, q4_row_bytes(K)], as binding.quantize_q4 writes them).
    caches: per block (k_cache, v_cache) bf16 [B, KV/128, s_max, 128] and pos
    int32 [B] on the device: each block runs decode attention on its q, k, v
    (attn may then be None)."""
    B, H = h_in.shape
    L = len(blocks)
    KV = blocks[0]["Wk"].shape[0] if L else 0
    I = blocks[0]["Wg"].shape[0] if L else 0
    V = head["Wlm"].shape[0] if head else 0
    dev = h_in.device
    h_out = torch.empty_like(h_in)
    h_trace = torch.empty((L, B, H), dtype=torch.float32, device=dev) if trace else None
    descs, keep, qkv = [], [blocks, head, attn, h_in], []
    for l, w in enumerate(blocks):
        d = wb.BlockDesc(kind=wb.BLOCK_QWEN)
        q = k = v = None
        if keep_qkv:
            q = torch.empty((B, H), device=dev)
            k = torch.empty((B, KV), device=dev)
            v = torch.empty((B, KV), device=dev)
            qkv.append((q, k, v))
        kc, vc = caches[l] if caches is not None else (None, None)
        d.u.qwen = wb.QwenBlock(*(w[n].data_ptr() for n in ("gamma1", "Wq", "Wk", "Wv", "Wo",
                                                             "gamma2", "Wg", "Wu", "Wd")),
                                attn[l].data_ptr() if attn is not None else None,
                                q.data_ptr() if q is not None else None,
                                k.data_ptr() if k is not None else None,
                                v.data_ptr() if v is not None else None,
                                kc.data_ptr() if kc is not None else None,
                                vc.data_ptr() if vc is not None else None)
        descs.append(d)
    idx = lg = None
    if head is not None:
        idx = torch.full((B,), -1, dtype=torch.int32, device=dev)
        lg = torch.empty((B, V), device=dev) if logits else None
        d = wb.BlockDesc(kind=wb.BLOCK_HEAD)
        d.u.head = wb.HeadBlock(head["gamma_f"].data_ptr(), head["Wlm"].data_ptr(),
                                idx.data_ptr(), lg.data_ptr() if lg is not None else None)
        descs.append(d)
    o = _opts(B, H, KV, I, V, eps, use_pdl, prefetch, fixed_plan, distance, decoy, tune_pairs,
              min_gain, persistent)
    o.h_in = h_in.data_ptr()
    o.h_out = h_out.data_ptr()
    o.h_trace = h_trace.data_ptr() if h_trace is not None else None
    o.weight_format = 1 if q4 else 0
    if caches is not None:
        o.attention = 1
        o.s_max = caches[0][0].shape[2]
        o.pos = pos.data_ptr()
        keep += [caches, pos]
    keep += [h_out, h_trace, idx, lg, qkv]
    ch = wb.Chain(descs, o, keepalive=keep)
    return QwenChain(ch, h_in, h_out, attn, idx, lg, h_trace, qkv)


def mlp_chain(blocks, x_in, *, eps=1e-5, use_pdl=True, prefetch=0, fixed_plan=None,
              distance=1, decoy=False, tune_pairs=30, min_gain=0.01,
              persistent=False, trace=False, training=False) -> MlpChain:
    """blocks: list of dicts of bf16 device tensors gamma, beta, W, b; x_in bf16 [B, w].
    trace=True keeps every block's output in `trace` (bf16 [L, B, w]).
    training=True (implies trace) also keeps what each module keeps for the
    backward: the Linear's input (`ln`, bf16 [L, B, w]), the GELU's input
    (`pre`, bf16 [L, B, w]) and derivative there (`gelu_grad`, fp32
    [L, B, w]), and the LayerNorm mean and rstd of every block's input
    (`ln_stats`, fp32 [L, B, 2])."""
    B, w = x_in.shape
    L = len(blocks)
    trace = trace or training
    y_out = torch.empty_like(x_in)
    tr = torch.empty((L, B, w), dtype=torch.bfloat16, device=x_in.device) if trace else None
    gg = torch.empty((L, B, w), dtype=torch.float32, device=x_in.device) if training else None
    st = torch.empty((L, B, 2), dtype=torch.float32, device=x_in.device) if training else None
    ln = torch.empty((L, B, w), dtype=torch.bfloat16, device=x_in.device) if training else None
    pre = torch.empty((L, B, w), dtype=torch.bfloat16, device=x_in.device) if training else None
    descs = []
    for blk in blocks:
        d = wb.BlockDesc(kind=wb.BLOCK_MLP)
        d.u.mlp = wb.MlpBlock(blk["gamma"].data_ptr(), blk["beta"].data_ptr(),
                              blk["W"].data_ptr(), blk["b"].data_ptr())
        descs.append(d)
    o = _opts(B, w, 0, 0, 0, eps, use_pdl, prefetch, fixed_plan, distance, decoy, tune_pairs,
              min_gain, persistent)
    o.x_in = x_in.data_ptr()
    o.y_out = y_out.data_ptr()
    o.h_trace = tr.data_ptr() if tr is not None else None
    o.mlp_gelu_grad = gg.data_ptr() if gg is not None else None
    o.mlp_ln_stats = st.data_ptr() if st is not None else None
    o.mlp_ln = ln.data_ptr() if ln is not None else None
    o.mlp_pre = pre.data_ptr() if pre is not None else None
    ch = wb.Chain(descs, o, keepalive=[blocks, x_in, y_out, tr, gg, st, ln, pre])
    return MlpChain(ch, x_in, y_out, tr, gg, st, ln, pre)


@dataclass
class MlpBackwardRun:
    bwd: wb.MlpBackward
    grads: list
    dx: torch.Tensor
    dx_trace: torch.Tensor | None = None
    dlin_trace: torch.Tensor | None = None
    dln_trace: torch.Tensor | None = None

    def run(self, stream=None):
        self.bwd.run(stream)


def mlp_backward(blocks, fwd: MlpChain, *, dz=None, use_pdl=True, prefetch=0, fixed_plan=None,
                 distance=1, decoy=False, tune_pairs=30, min_gain=0.01,
                 traces=False) -> MlpBackwardRun:
    """The backward pass of the chain `fwd` (built with training=True) over
    the same blocks ("Making small PyTorch ops faster on a laptop GPU", "It
    works in training too").  dz: bf16 [B, w] gradient of the loss with
    respect to the chain output, or None for the mean-square loss of the
    output.  Returns the gradient tensors (per block dW, db, dgamma, dbeta
    in `grads`; dx of the chain input); traces=True also keeps every block's
    input gradient (dx_trace [L+1, B, w], slot L the loss gradient), dlin
    and dln (bf16 [L, B, w])."""
    if fwd.gelu_grad is None:
        raise ValueError("the forward chain was not built with training=True")
    B, w = fwd.x_in.shape
    L = len(blocks)
    dev = fwd.x_in.device
    grads = [{"dW": torch.empty((w, w), dtype=torch.bfloat16, device=dev),
              "db": torch.empty((w,), dtype=torch.bfloat16, device=dev),
              "dgamma": torch.empty((w,), dtype=torch.bfloat16, device=dev),
              "dbeta": torch.empty((w,), dtype=torch.bfloat16, device=dev)} for _ in range(L)]
    dx = torch.empty((B, w), dtype=torch.bfloat16, device=dev)
    dxt = torch.empty((L + 1, B, w), dtype=torch.bfloat16, device=dev) if traces else None
    dlt = torch.empty((L, B, w), dtype=torch.bfloat16, device=dev) if traces else None
    dnt = torch.empty((L, B, w), dtype=torch.bfloat16, device=dev) if traces else None
    o = wb.MlpBackwardOpts()
    o.batch, o.width = B, w
    o.x_in = fwd.x_in.data_ptr()
    o.acts = fwd.trace.data_ptr()
    o.ln = fwd.ln.data_ptr()
    o.gelu_grad = fwd.gelu_grad.data_ptr()
    o.ln_stats = fwd.ln_stats.data_ptr()
    o.dz = dz.data_ptr() if dz is not None else None
    o.dx = dx.data_ptr()
    o.dx_trace = dxt.data_ptr() if dxt is not None else None
    o.dlin_trace = dlt.data_ptr() if dlt is not None else None
    o.dln_trace = dnt.data_ptr() if dnt is not None else None
    o.use_pdl = 1 if use_pdl else 0
    o.prefetch = prefetch
    if fixed_plan is not None:
        o.fixed_plan = fixed_plan
    o.distance = distance
    o.decoy = 1 if decoy else 0
    o.tune_pairs = tune_pairs
    o.tune_min_gain = min_gain
    bl = [wb.MlpBlock(b["gamma"].data_ptr(), b["beta"].data_ptr(), b["W"].data_ptr(),
                      b["b"].data_ptr()) for b in blocks]
    gr = [wb.MlpGrads(g["dW"].data_ptr(), g["db"].data_ptr(), g["dgamma"].data_ptr(),
                      g["dbeta"].data_ptr()) for g in grads]
    bwd = wb.MlpBackward(bl, gr, o, keepalive=[blocks, fwd, grads, dx, dxt, dlt, dnt, dz])
    return MlpBackwardRun(bwd, grads, dx, dxt, dlt, dnt)
