"""Thin ctypes binding of libwsgemv.so (argument marshalling only).

Every function here has the name of a C entry point without its ``ws_``
prefix and forwards to it; all arithmetic runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (torch supplies device memory and streams);
their data pointers, shapes and the current stream's handle are what cross the
ABI.  A nonzero status raises ``WsError`` carrying the library's message.

If the shared library is missing the import fails loudly: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

C = ctypes
P = C.c_void_p
I32 = C.c_int
SZ = C.c_size_t
F32 = C.c_float

DTYPE_F32, DTYPE_BF16, DTYPE_F16 = 0, 1, 2
PREFETCH_NONE, PREFETCH_L2, PREFETCH_L2_EVICT_LAST, PREFETCH_BULK = 0, 1, 2, 3
BLOCK_QWEN, BLOCK_MLP, BLOCK_HEAD = 1, 2, 3
OP_GEMV, OP_SWIGLU_GEMV, OP_QKV_GEMV, OP_LMHEAD_ARGMAX, OP_ARGMAX_ROWS = 1, 2, 3, 4, 5
PRO_NONE, PRO_RMSNORM, PRO_LAYERNORM = 0, 1, 2
EPI_F32, EPI_BF16, EPI_RESID, EPI_BIAS_GELU, EPI_SWIGLU, EPI_ARGMAX = 0, 1, 2, 3, 4, 5

STATUS = {0: "WS_OK", -1: "WS_ERR_ARG", -2: "WS_ERR_ALIGN", -3: "WS_ERR_SHAPE",
          -4: "WS_ERR_CUDA", -5: "WS_ERR_TIMEOUT", -6: "WS_ERR_NOMEM", -7: "WS_ERR_STATE"}


class WsError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class PrefetchPlan(C.Structure):
    _fields_ = [("blocks", I32), ("threads", I32), ("stride_bytes", I32), ("mode", I32)]


class QwenBlock(C.Structure):
    _fields_ = [(n, P) for n in ("gamma1", "Wq", "Wk", "Wv", "Wo", "gamma2", "Wg", "Wu", "Wd",
                                 "attn", "q", "k", "v", "k_cache", "v_cache")]


class MlpBlock(C.Structure):
    _fields_ = [(n, P) for n in ("gamma", "beta", "W", "bias")]


class HeadBlock(C.Structure):
    _fields_ = [(n, P) for n in ("gamma", "W", "idx", "logits")]


class _BlockUnion(C.Union):
    _fields_ = [("qwen", QwenBlock), ("mlp", MlpBlock), ("head", HeadBlock)]


class BlockDesc(C.Structure):
    _fields_ = [("kind", I32), ("u", _BlockUnion)]


class ChainOpts(C.Structure):
    _fields_ = [("batch", I32), ("hidden", I32), ("kv_dim", I32), ("inter", I32),
                ("vocab", I32), ("eps", F32), ("h_in", P), ("h_out", P), ("x_in", P),
                ("y_out", P), ("h_trace", P), ("use_pdl", I32), ("prefetch", I32),
                ("fixed_plan", PrefetchPlan), ("distance", I32), ("decoy", I32),
                ("tune_pairs", I32), ("tune_min_gain", F32), ("weight_format", I32),
                ("persistent", I32), ("attention", I32), ("s_max", I32), ("pos", P),
                ("mlp_ln", P), ("mlp_pre", P), ("mlp_gelu_grad", P), ("mlp_ln_stats", P)]


class MlpGrads(C.Structure):
    _fields_ = [("dW", P), ("db", P), ("dgamma", P), ("dbeta", P)]


class MlpBackwardOpts(C.Structure):
    _fields_ = [("batch", I32), ("width", I32), ("x_in", P), ("acts", P), ("ln", P),
                ("gelu_grad", P), ("ln_stats", P), ("dz", P), ("dx", P), ("dx_trace", P),
                ("dlin_trace", P), ("dln_trace", P), ("use_pdl", I32), ("prefetch", I32),
                ("fixed_plan", PrefetchPlan), ("distance", I32), ("decoy", I32),
                ("tune_pairs", I32), ("tune_min_gain", F32)]


class Tuning(C.Structure):
    _fields_ = [("ring_bytes", I32), ("grid_cap", I32), ("force_ksplit", I32),
                ("force_rt", I32), ("evict_first", I32), ("piece_bytes", I32),
                ("timeout_ns", C.c_ulonglong), ("l2_ahead", I32),
                ("forms", I32), ("launch_pdl", I32), ("mma", I32), ("ctas_per_sm", I32),
                ("q4_mma", I32)]


class GemvSchedule(C.Structure):
    _fields_ = [(n, I32) for n in ("RT", "S", "KS", "PC", "NP", "NSW", "piece_bytes", "RG",
                                   "grid", "smem_bytes")]


_SIGS = {
    "ws_gemv_bf16": [P, P, P, I32, I32, I32, P, SZ, P],
    "ws_gemv_bf16_noalloc": [P, P, P, I32, I32, I32, P],
    "ws_gemv_residual": [P, P, P, P, I32, I32, I32, P, SZ, P],
    "ws_rmsnorm_gemv": [P, I32, P, P, P, I32, I32, I32, F32, P, SZ, P],
    "ws_qkv_gemv": [P, I32, P, P, P, P, P, P, P, I32, I32, I32, I32, F32, P, SZ, P],
    "ws_swiglu_gemv": [P, I32, P, P, P, P, I32, I32, I32, F32, P, SZ, P],
    "ws_ln_gemv_gelu": [P, P, P, P, P, P, I32, I32, I32, F32, P, SZ, P],
    "ws_lmhead_argmax": [P, I32, P, P, P, P, I32, I32, I32, F32, P, SZ, P],
    "ws_argmax_rows": [P, P, I32, I32, P, SZ, P],
    "ws_decode_attention": [P, P, P, P, P, P, P, P, I32, I32, I32, I32, I32, P, SZ, P],
    "ws_quantize_q4": [P, P, I32, I32, P],
    "ws_gemv_q4": [P, P, P, I32, I32, I32, P, SZ, P],
    "ws_rmsnorm": [P, P, P, I32, I32, I32, F32, P],
    "ws_l2_prefetch": [P, SZ, PrefetchPlan, P],
    "ws_chain_create": [P, I32, P, P],
    "ws_chain_tune": [P, P],
    "ws_chain_capture": [P, P],
    "ws_chain_run": [P, P],
    "ws_chain_run_eager": [P, P],
    "ws_chain_step_host": [P, P, P, P, P],
    "ws_chain_plans": [P, P, P, P, I32],
    "ws_chain_op_bytes": [P, P, I32],
    "ws_mlp_backward_create": [P, P, I32, P, P],
    "ws_mlp_backward_tune": [P, P],
    "ws_mlp_backward_capture": [P, P],
    "ws_mlp_backward_run": [P, P],
    "ws_mlp_backward_plan": [P, P, P, P],
    "ws_set_tuning": [P],
    "ws_gemv_plan": [I32, I32, I32, I32, I32, I32, I32, P],
    "ws_read_probe": [P, SZ, I32, P, P],
    "ws_empty_probe": [I32, P, P, P],
    "ws_test_bounded_wait": [C.c_ulonglong, P],
}
_OTHER = {
    "ws_workspace_bytes": ([I32, I32, I32, I32], SZ),
    "ws_attention_workspace_bytes": ([I32, I32, I32, I32, I32], SZ),
    "ws_q4_row_bytes": ([I32], SZ),
    "ws_last_error": ([], C.c_char_p),
    "ws_device_error": ([I32], I32),
    "ws_chain_num_ops": ([P], I32),
    "ws_chain_is_persistent": ([P], I32),
    "ws_chain_grid": ([P], I32),
    "ws_chain_debug_stamps": ([P, P, SZ], I32),
    "ws_chain_destroy": ([P], None),
    "ws_mlp_backward_num_launches": ([P], I32),
    "ws_mlp_backward_destroy": ([P], None),
    "ws_get_tuning": ([P], None),
    "ws_debug_gemv_copies": ([I32, I32, I32, I32, I32, I32, P, C.c_long], C.c_long),
    "ws_debug_gemv_copies_q4": ([I32, I32, I32, I32, I32, I32, P, C.c_long, P], C.c_long),
    "ws_version": ([], C.c_char_p),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libwsgemv.so (built by ``build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: run __graft_entry__.build() (nvcc, sm_103a) first")
    lib = C.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I32
    for name, (args, res) in _OTHER.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise WsError(status, load().ws_last_error().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ws(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def _dtype_code(t):
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float16:
        return DTYPE_F16
    raise TypeError(f"unsupported dtype {t.dtype}")


# --------------------------------------------------------------------------- ops

def workspace_bytes(op: int, M: int, K: int, B: int) -> int:
    return int(load().ws_workspace_bytes(op, M, K, B))


def new_workspace(op: int, M: int, K: int, B: int, device="cuda"):
    """A zero-filled workspace sized for the op (None when it needs none)."""
    n = workspace_bytes(op, M, K, B)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


def gemv_bf16(W, x, y, workspace=None, stream=None):
    M, K = W.shape
    B = x.shape[0]
    wp, wb = _ws(workspace)
    _check(load().ws_gemv_bf16(_ptr(W), _ptr(x), _ptr(y), M, K, B, wp, wb, _stream(stream)))


def gemv_bf16_noalloc(W, x, y, stream=None):
    """ws_gemv_bf16 without a workspace argument and without any allocation:
    split-K scratch comes from the library's fixed device array."""
    M, K = W.shape
    B = x.shape[0]
    _check(load().ws_gemv_bf16_noalloc(_ptr(W), _ptr(x), _ptr(y), M, K, B, _stream(stream)))


def gemv_residual(W, x, h_out, h_in=None, workspace=None, stream=None):
    M, K = W.shape
    B = x.shape[0]
    wp, wb = _ws(workspace)
    _check(load().ws_gemv_residual(_ptr(W), _ptr(x), _ptr(h_in), _ptr(h_out), M, K, B, wp, wb,
                                   _stream(stream)))


def rmsnorm_gemv(x, gamma, W, y, eps, workspace=None, stream=None):
    M, K = W.shape
    B = x.shape[0]
    wp, wb = _ws(workspace)
    _check(load().ws_rmsnorm_gemv(_ptr(x), _dtype_code(x), _ptr(gamma), _ptr(W), _ptr(y), M, K,
                                  B, float(eps), wp, wb, _stream(stream)))


def qkv_gemv(x, gamma, Wq, Wk, Wv, q, k, v, eps, workspace=None, stream=None):
    Mq, K = Wq.shape
    Mkv = Wk.shape[0]
    B = x.shape[0]
    wp, wb = _ws(workspace)
    _check(load().ws_qkv_gemv(_ptr(x), _dtype_code(x), _ptr(gamma), _ptr(Wq), _ptr(Wk),
                              _ptr(Wv), _ptr(q), _ptr(k), _ptr(v), Mq, Mkv, K, B, float(eps),
                              wp, wb, _stream(stream)))


def swiglu_gemv(x, gamma, Wg, Wu, s, eps, workspace=None, stream=None):
    M, K = Wg.shape
    B = x.shape[0]
    wp, wb = _ws(workspace)
    _check(load().ws_swiglu_gemv(_ptr(x), _dtype_code(x), _ptr(gamma), _ptr(Wg), _ptr(Wu),
                                 _ptr(s), M, K, B, float(eps), wp, wb, _stream(stream)))


def ln_gemv_gelu(x, gamma, beta, W, bias, z, eps, workspace=None, stream=None):
    M, K = W.shape
    B = x.shape[0]
    wp, wb = _ws(workspace)
    _check(load().ws_ln_gemv_gelu(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(W), _ptr(bias),
                                  _ptr(z), M, K, B, float(eps), wp, wb, _stream(stream)))


def lmhead_argmax(h, gamma, W, idx, eps, workspace, logits=None, stream=None):
    V, K = W.shape
    B = h.shape[0]
    wp, wb = _ws(workspace)
    _check(load().ws_lmhead_argmax(_ptr(h), _dtype_code(h), _ptr(gamma), _ptr(W), _ptr(idx),
                                   _ptr(logits), V, K, B, float(eps), wp, wb, _stream(stream)))


def argmax_rows(logits, idx, workspace, stream=None):
    rows, cols = logits.shape
    wp, wb = _ws(workspace)
    _check(load().ws_argmax_rows(_ptr(logits), _ptr(idx), rows, cols, wp, wb, _stream(stream)))


def q4_row_bytes(K: int) -> int:
    return int(load().ws_q4_row_bytes(K))


def quantize_q4(W, Wq, stream=None):
    """W bf16 [M, K] -> Wq uint8 [M, q4_row_bytes(K)] (4-bit groups of 128)."""
    M, K = W.shape
    _check(load().ws_quantize_q4(_ptr(W), _ptr(Wq), M, K, _stream(stream)))


def gemv_q4(Wq, x, y, K, workspace=None, stream=None):
    """y [B, M] fp32 = x [B, K] bf16 . W^T for packed 4-bit rows Wq [M, q4_row_bytes(K)]."""
    M = Wq.shape[0]
    B = x.shape[0]
    wp, wb = _ws(workspace)
    _check(load().ws_gemv_q4(_ptr(Wq), _ptr(x), _ptr(y), M, K, B, wp, wb, _stream(stream)))


def attention_workspace_bytes(B, n_heads, n_kv_heads, s_max, head_dim=128) -> int:
    return int(load().ws_attention_workspace_bytes(B, n_heads, n_kv_heads, head_dim, s_max))


def decode_attention(q, k_new, v_new, k_cache, v_cache, pos, workspace, out_f32=None,
                     out_bf16=None, stream=None):
    """q [B, n_heads*128] fp32, k_new/v_new [B, n_kv*128] fp32, caches bf16
    [B, n_kv, s_max, 128] (updated in place at pos), pos int32 [B] on the device."""
    B, n_kv, s_max, d = k_cache.shape
    n_heads = q.shape[1] // d
    wp, wb = _ws(workspace)
    _check(load().ws_decode_attention(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(pos), _ptr(out_f32), _ptr(out_bf16),
                                      B, n_heads, n_kv, d, s_max, wp, wb, _stream(stream)))


def rmsnorm(x, gamma, y, eps, stream=None):
    R, N = x.shape
    _check(load().ws_rmsnorm(_ptr(x), _ptr(gamma), _ptr(y), R, N, _dtype_code(x), float(eps),
                             _stream(stream)))


def l2_prefetch(ptr, nbytes, plan: PrefetchPlan, stream=None):
    _check(load().ws_l2_prefetch(_ptr(ptr), int(nbytes), plan, _stream(stream)))


def read_probe(buf, nbytes, blocks, sink, stream=None):
    _check(load().ws_read_probe(_ptr(buf), int(nbytes), int(blocks), _ptr(sink), _stream(stream)))


def empty_probe(touch, ptr=None, sink=None, stream=None):
    _check(load().ws_empty_probe(int(touch), _ptr(ptr), _ptr(sink), _stream(stream)))


def test_bounded_wait(timeout_ns, stream=None):
    _check(load().ws_test_bounded_wait(int(timeout_ns), _stream(stream)))


def device_error(reset=False) -> int:
    return int(load().ws_device_error(1 if reset else 0))


def get_tuning() -> Tuning:
    t = Tuning()
    load().ws_get_tuning(C.byref(t))
    return t


def set_tuning(t: Tuning):
    _check(load().ws_set_tuning(C.byref(t)))


def gemv_plan(M, K, B, nmat=1, prologue=PRO_NONE, epilogue=EPI_F32, allow_split=True):
    s = GemvSchedule()
    _check(load().ws_gemv_plan(M, K, B, nmat, prologue, epilogue, 1 if allow_split else 0,
                               C.byref(s)))
    return {n: getattr(s, n) for n, _ in GemvSchedule._fields_}


def debug_gemv_copies_q4(M, K, B, nmat, cta, mma=False):
    """(triples, schedule dict) of CTA `cta` for packed 4-bit rows."""
    lib = load()
    sc = GemvSchedule()
    n = lib.ws_debug_gemv_copies_q4(M, K, B, nmat, cta, int(mma), None, 0, C.byref(sc))
    if n < 0:
        raise WsError(-1, "bad arguments")
    buf = (C.c_longlong * (3 * max(n, 1)))()
    lib.ws_debug_gemv_copies_q4(M, K, B, nmat, cta, int(mma), buf, n, None)
    sched = {f: getattr(sc, f) for f, _ in GemvSchedule._fields_}
    return [(buf[3 * i], buf[3 * i + 1], buf[3 * i + 2]) for i in range(n)], sched


def debug_gemv_copies(M, K, B, nmat, allow_split, cta):
    lib = load()
    n = lib.ws_debug_gemv_copies(M, K, B, nmat, int(allow_split), cta, None, 0)
    if n < 0:
        raise WsError(-1, "bad arguments")
    buf = (C.c_longlong * (3 * max(n, 1)))()
    lib.ws_debug_gemv_copies(M, K, B, nmat, int(allow_split), cta, buf, n)
    return [(buf[3 * i], buf[3 * i + 1], buf[3 * i + 2]) for i in range(n)]


def version() -> str:
    return load().ws_version().decode()


# --------------------------------------------------------------------------- chain

class Chain:
    """A decode chain: ws_chain_create / tune / capture / run / destroy.

    Keeps the Python objects whose device memory the chain points at alive."""

    def __init__(self, blocks, opts: ChainOpts, keepalive=()):
        arr = (BlockDesc * len(blocks))(*blocks)
        h = P()
        _check(load().ws_chain_create(arr, len(blocks), C.byref(opts), C.byref(h)))
        self.handle = h
        self.opts = opts
        self._keep = list(keepalive)
        self.n_ops = int(load().ws_chain_num_ops(h))
        self.persistent = bool(load().ws_chain_is_persistent(h))

    def tune(self, stream=None):
        _check(load().ws_chain_tune(self.handle, _stream(stream)))

    def capture(self, stream=None):
        _check(load().ws_chain_capture(self.handle, _stream(stream)))

    def run(self, stream=None):
        _check(load().ws_chain_run(self.handle, _stream(stream)))

    def run_eager(self, stream=None):
        _check(load().ws_chain_run_eager(self.handle, _stream(stream)))

    def step_host(self, in_host, attn_host, out_host, stream=None):
        _check(load().ws_chain_step_host(self.handle, _ptr(in_host), _ptr(attn_host),
                                         _ptr(out_host), _stream(stream)))

    def plans(self):
        n = self.n_ops
        pl = (PrefetchPlan * n)()
        lo = (F32 * n)()
        mean = (F32 * n)()
        _check(load().ws_chain_plans(self.handle, pl, lo, mean, n))
        return [((p.mode, p.blocks, p.threads, p.stride_bytes), lo[i], mean[i])
                for i, p in enumerate(pl)]

    def debug_stamps(self, buf):
        """Record per-CTA, per-op timestamps and per-warp wait times into `buf`
        (int64 [grid, ops, 44]) on every later-captured step; None stops.
        Re-capture afterwards."""
        n = 0 if buf is None else buf.numel()
        _check(load().ws_chain_debug_stamps(self.handle, _ptr(buf), n))

    def grid(self) -> int:
        return int(load().ws_chain_grid(self.handle))

    def op_bytes(self):
        n = self.n_ops
        b = (SZ * n)()
        _check(load().ws_chain_op_bytes(self.handle, b, n))
        return list(b)

    def close(self):
        if self.handle:
            load().ws_chain_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MlpBackward:
    """The backward pass of a LayerNorm -> Linear -> GELU chain:
    ws_mlp_backward_create / tune / capture / run / destroy.  Keeps the
    Python objects whose device memory it points at alive."""

    def __init__(self, blocks, grads, opts: MlpBackwardOpts, keepalive=()):
        n = len(blocks)
        barr = (MlpBlock * n)(*blocks)
        garr = (MlpGrads * n)(*grads)
        h = P()
        _check(load().ws_mlp_backward_create(barr, garr, n, C.byref(opts), C.byref(h)))
        self.handle = h
        self.opts = opts
        self._keep = list(keepalive)
        self.n_launches = int(load().ws_mlp_backward_num_launches(h))

    def tune(self, stream=None):
        _check(load().ws_mlp_backward_tune(self.handle, _stream(stream)))

    def capture(self, stream=None):
        _check(load().ws_mlp_backward_capture(self.handle, _stream(stream)))

    def run(self, stream=None):
        _check(load().ws_mlp_backward_run(self.handle, _stream(stream)))

    def plan(self):
        pl = PrefetchPlan()
        lo, mean = F32(), F32()
        _check(load().ws_mlp_backward_plan(self.handle, C.byref(pl), C.byref(lo), C.byref(mean)))
        return (pl.mode, pl.blocks, pl.threads, pl.stride_bytes), lo.value, mean.value

    def close(self):
        if self.handle:
            load().ws_mlp_backward_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def chain_run(chain: Chain, stream=None):
    chain.run(stream)
