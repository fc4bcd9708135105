"""Plain CPU oracle for the BF16 weight-streaming decode chain.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product package
never does.  It shares no code with the CUDA library.

The arithmetic lives in ``oracle.c`` (double accumulation, plain loops); this
module compiles it with gcc, wraps it with ctypes and composes the primitives
into the decode block, the decode chain and the MLP chain exactly in the order
the pages describe:

* "One Token, Kernel by Kernel: A Decode Step on a Laptop GPU", Step 1
  ("The setup": RMSNorm, grouped-query attention, SwiGLU MLP; "What one block
  launches": BF16 weight GEMVs with FP32 accumulation) and "The whole step"
  (final RMSNorm, LM head 151,936 x 1,536, argmax over the logits).
* "GPU Kernel Optimization", Architecture: RMSNorm = mean square, rsqrt,
  weight multiply.
* "Making small PyTorch ops faster on a laptop GPU", "Beyond language models":
  72 x [LayerNorm(768) -> Linear(768, 768) -> GELU] in bf16.

Readings where the pages are silent (each also listed in the design notes):
eps sits inside the square root; a normalisation is computed exactly and
rounded once to bf16 (x * r * gamma, then one rounding); the residual stream h
is stored in fp32 and every GEMV input (normalised activations, the attention
stand-in, the SwiGLU product) in bf16; SwiGLU is silu(g) * u on the unrounded
products, rounded once to bf16; argmax ties go to the lowest index.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP when present)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-D_DEFAULT_SOURCE", "-shared", "-fPIC",
            "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            L = ctypes.c_long
            D = ctypes.c_double
            sig = {
                "ws_oracle_bf16_to_f64": [P, P, L],
                "ws_oracle_f64_to_bf16": [P, P, L],
                "ws_oracle_fp16_to_f64": [P, P, L],
                "ws_oracle_f64_to_fp16": [P, P, L],
                "ws_oracle_round_f32": [P, L],
                "ws_oracle_gemv": [P, L, L, P, L, P, ctypes.c_int],
                "ws_oracle_rmsnorm": [P, L, L, P, D, P],
                "ws_oracle_layernorm": [P, L, L, P, P, D, P],
                "ws_oracle_gelu": [P, P, L],
                "ws_oracle_swiglu": [P, P, P, L],
                "ws_oracle_argmax_rows": [P, L, L, P],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = None
            lib.ws_oracle_openmp_threads.argtypes = []
            lib.ws_oracle_openmp_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == np.uint16, "bf16/fp16 values travel as uint16 bit patterns"
    return np.ascontiguousarray(a)


# --------------------------------------------------------------------------
# storage formats
# --------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    bits = _u16(bits)
    out = np.empty(bits.shape, np.float64)
    _load().ws_oracle_bf16_to_f64(_ptr(bits), _ptr(out), bits.size)
    return out


def f64_to_bf16(v) -> np.ndarray:
    v = _f64(v)
    out = np.empty(v.shape, np.uint16)
    _load().ws_oracle_f64_to_bf16(_ptr(v), _ptr(out), v.size)
    return out


def fp16_to_f64(bits) -> np.ndarray:
    bits = _u16(bits)
    out = np.empty(bits.shape, np.float64)
    _load().ws_oracle_fp16_to_f64(_ptr(bits), _ptr(out), bits.size)
    return out


def f64_to_fp16(v) -> np.ndarray:
    v = _f64(v)
    out = np.empty(v.shape, np.uint16)
    _load().ws_oracle_f64_to_fp16(_ptr(v), _ptr(out), v.size)
    return out


def round_bf16(v) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even) and return it as double."""
    return bf16_to_f64(f64_to_bf16(v))


def round_f32(v) -> np.ndarray:
    v = _f64(v).copy()
    _load().ws_oracle_round_f32(_ptr(v), v.size)
    return v


# --------------------------------------------------------------------------
# primitives
# --------------------------------------------------------------------------

def gemv(W_bits, x, threads: int = 1) -> np.ndarray:
    """y = x . W^T accumulated in double; W is bf16 bits [M, K], x is [B, K]."""
    W_bits = _u16(W_bits)
    M, K = W_bits.shape
    x = _f64(x).reshape(-1, K)
    B = x.shape[0]
    y = np.empty((B, M), np.float64)
    _load().ws_oracle_gemv(_ptr(W_bits), M, K, _ptr(x), B, _ptr(y), int(threads))
    return y


def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """x * r * gamma with r = 1/sqrt(mean(x^2) + eps), per row, exact (double)."""
    x = _f64(x)
    K = x.shape[-1]
    x2 = x.reshape(-1, K)
    g = _f64(gamma).reshape(K)
    out = np.empty_like(x2)
    _load().ws_oracle_rmsnorm(_ptr(x2), x2.shape[0], K, _ptr(g), float(eps), _ptr(out))
    return out.reshape(x.shape)


def layernorm(x, gamma, beta, eps: float) -> np.ndarray:
    x = _f64(x)
    N = x.shape[-1]
    x2 = x.reshape(-1, N)
    g = _f64(gamma).reshape(N)
    bt = _f64(beta).reshape(N)
    out = np.empty_like(x2)
    _load().ws_oracle_layernorm(_ptr(x2), x2.shape[0], N, _ptr(g), _ptr(bt),
                                float(eps), _ptr(out))
    return out.reshape(x.shape)


def gelu(z) -> np.ndarray:
    z = _f64(z)
    out = np.empty_like(z)
    _load().ws_oracle_gelu(_ptr(z), _ptr(out), z.size)
    return out


def swiglu(g, u) -> np.ndarray:
    g = _f64(g)
    u = _f64(u)
    assert g.shape == u.shape
    out = np.empty_like(g)
    _load().ws_oracle_swiglu(_ptr(g), _ptr(u), _ptr(out), g.size)
    return out


def argmax_rows(v) -> np.ndarray:
    v = _f64(v)
    v2 = v.reshape(-1, v.shape[-1])
    idx = np.empty(v2.shape[0], np.int32)
    _load().ws_oracle_argmax_rows(_ptr(v2), v2.shape[0], v2.shape[1], _ptr(idx))
    return idx


# --------------------------------------------------------------------------
# fused ops, as the C-ABI exposes them (same arithmetic, composed here)
# --------------------------------------------------------------------------

def rmsnorm_gemv(x, gamma, W_bits, eps: float, threads: int = 1) -> np.ndarray:
    """y = bf16(RMSNorm(x, gamma)) . W^T  (y in double; the fp32 output's target)."""
    a = round_bf16(rmsnorm(x, gamma, eps))
    return gemv(W_bits, a, threads)


def swiglu_gemv(x, gamma, Wg_bits, Wu_bits, eps: float, threads: int = 1,
                exact: bool = False) -> np.ndarray:
    """s = bf16(silu(m.Wg^T) * (m.Wu^T)), m = bf16(RMSNorm(x)) or x when gamma is None.

    Returns the bf16 bit patterns of s, or with exact=True the value of s
    before its final rounding (double)."""
    m = x if gamma is None else round_bf16(rmsnorm(x, gamma, eps))
    g = gemv(Wg_bits, m, threads)
    u = gemv(Wu_bits, m, threads)
    s = swiglu(g, u)
    return s if exact else f64_to_bf16(s)


def lmhead_logits(h, gamma, Wlm_bits, eps: float, threads: int = 1) -> np.ndarray:
    """Logits = bf16(RMSNorm(h, gamma_final)) . Wlm^T, in double."""
    return rmsnorm_gemv(h, gamma, Wlm_bits, eps, threads)


# --------------------------------------------------------------------------
# the decode block and chain
# --------------------------------------------------------------------------

def qwen_block(h, blk: dict, attn, eps: float, threads: int = 1) -> dict:
    """One decoder block of the weight chain, attention replaced by `attn`.

    h: fp32 residual [B, H] as double (not modified); blk: bf16 bit arrays
    gamma1, Wq, Wk, Wv, Wo, gamma2, Wg, Wu, Wd; attn: the bf16 stand-in for the
    attention output [B, H] (as double).  Steps:

      a = bf16(RMSNorm(h, gamma1));   q, k, v = a.Wq^T, a.Wk^T, a.Wv^T
      h = fp32(h + attn.Wo^T)
      m = bf16(RMSNorm(h, gamma2));   s = bf16(silu(m.Wg^T) * (m.Wu^T))
      h = fp32(h + s.Wd^T)
    """
    g1 = bf16_to_f64(blk["gamma1"])
    g2 = bf16_to_f64(blk["gamma2"])
    a = round_bf16(rmsnorm(h, g1, eps))
    q = gemv(blk["Wq"], a, threads)
    k = gemv(blk["Wk"], a, threads)
    v = gemv(blk["Wv"], a, threads)
    h1 = round_f32(np.asarray(h, np.float64) + gemv(blk["Wo"], attn, threads))
    m = round_bf16(rmsnorm(h1, g2, eps))
    s_bits = f64_to_bf16(swiglu(gemv(blk["Wg"], m, threads), gemv(blk["Wu"], m, threads)))
    s = bf16_to_f64(s_bits)
    h2 = round_f32(h1 + gemv(blk["Wd"], s, threads))
    return {"q": q, "k": k, "v": v, "h_mid": h1, "s": s_bits, "h": h2}


def qwen_block_attention(h, blk: dict, k_cache_bits, v_cache_bits, pos, n_kv_heads: int,
                         eps: float, qkv=None, threads: int = 1) -> dict:
    """One decoder block with decode attention over its key-value cache in
    place of the stand-in ("One Token, Kernel by Kernel", Step 1: RMSNorm,
    grouped-query attention, SwiGLU MLP; "The fix: Part 10's split-KV
    kernel"): q, k, v from the first RMSNorm, the new key and value appended
    at pos, attention with heads of 128, its output rounded once to bf16 as
    Wo's input, then the residual and the MLP as in qwen_block.  qkv, when
    given, is the (q, k, v) the attention uses instead of this block's own
    (teacher forcing on another implementation's projections)."""
    g1 = bf16_to_f64(blk["gamma1"])
    g2 = bf16_to_f64(blk["gamma2"])
    a = round_bf16(rmsnorm(h, g1, eps))
    q = gemv(blk["Wq"], a, threads)
    k = gemv(blk["Wk"], a, threads)
    v = gemv(blk["Wv"], a, threads)
    qa, ka, va = qkv if qkv is not None else (q, k, v)
    att = decode_attention(qa, ka, va, k_cache_bits, v_cache_bits, pos, n_kv_heads, 128)
    attn_bits = f64_to_bf16(att["out"])
    h1 = round_f32(np.asarray(h, np.float64) + gemv(blk["Wo"], bf16_to_f64(attn_bits), threads))
    m = round_bf16(rmsnorm(h1, g2, eps))
    s_bits = f64_to_bf16(swiglu(gemv(blk["Wg"], m, threads), gemv(blk["Wu"], m, threads)))
    h2 = round_f32(h1 + gemv(blk["Wd"], bf16_to_f64(s_bits), threads))
    return {"q": q, "k": k, "v": v, "attn": attn_bits, "h_mid": h1, "s": s_bits, "h": h2,
            "k_cache": att["k_cache"], "v_cache": att["v_cache"]}


def qwen_chain(h0, blocks, attns, gamma_f, Wlm_bits, eps: float,
               threads: int = 1, keep_blocks: bool = False) -> dict:
    """The full decode weight chain: blocks in order, then the final RMSNorm,
    the LM head and the argmax of every row (ties to the lowest index)."""
    h = round_f32(h0)
    per_block = []
    for blk, attn in zip(blocks, attns):
        out = qwen_block(h, blk, attn, eps, threads)
        h = out["h"]
        if keep_blocks:
            per_block.append(out)
    logits = lmhead_logits(h, bf16_to_f64(gamma_f), Wlm_bits, eps, threads)
    idx = argmax_rows(logits)
    return {"h": h, "logits": logits, "idx": idx, "blocks": per_block}


def mlp_block(x_bits, blk: dict, eps: float = 1e-5, threads: int = 1,
              exact: bool = False, linear: bool = False) -> np.ndarray:
    """bf16 LayerNorm -> Linear(+bias) -> GELU, each module's output rounded to bf16.

    Returns the bf16 bits of z = bf16(gelu(bf16(bf16(LN(x)).W^T + b))); with
    exact=True the value of gelu(...) before its final rounding (double); with
    linear=True the Linear output bf16(LN(x)).W^T + b before its rounding."""
    x = bf16_to_f64(x_bits)
    a = round_bf16(layernorm(x, bf16_to_f64(blk["gamma"]), bf16_to_f64(blk["beta"]), eps))
    lin = gemv(blk["W"], a, threads) + bf16_to_f64(blk["b"])[None, :]
    if linear:
        return lin
    z = gelu(round_bf16(lin))
    return z if exact else f64_to_bf16(z)


def mlp_chain(x_bits, blocks, eps: float = 1e-5, threads: int = 1) -> np.ndarray:
    z = _u16(x_bits)
    for blk in blocks:
        z = mlp_block(z, blk, eps, threads)
    return z


def rmsnorm_rows(x_bits, gamma_bits, eps: float, dtype: str = "fp16") -> np.ndarray:
    """Standalone RMSNorm of [R, N] rows stored in fp16 or bf16; one rounding."""
    dec = fp16_to_f64 if dtype == "fp16" else bf16_to_f64
    enc = f64_to_fp16 if dtype == "fp16" else f64_to_bf16
    return enc(rmsnorm(dec(x_bits), dec(gamma_bits), eps))


# --------------------------------------------------------------------------
# decode attention with a key-value cache
# --------------------------------------------------------------------------

def decode_attention(q, k_new, v_new, k_cache_bits, v_cache_bits, pos, n_kv_heads: int,
                     head_dim: int) -> dict:
    """One decode step of grouped-query attention over a key-value cache, in
    double ("Making small PyTorch ops faster on a laptop GPU", "A full decode
    step is a different story": the new key and value are appended to the
    cache and the softmax is taken over every cached position; "One Token,
    Kernel by Kernel", "The fix: Part 10's split-KV kernel": the cache layout
    (batch, key-value head, slot, dimension), the valid length read at run
    time, one key-value head serving n_heads / n_kv_heads query heads).

    q: [B, n_heads * d] (fp32 values); k_new, v_new: [B, n_kv * d]; the
    caches: bf16 bits [B, n_kv, S, d]; pos: [B] slot of the new token.
    Steps, per batch row b:
      1. the new key and value, rounded to bf16 (the cache's type), are
         written at slot pos[b] of their head;
      2. for query head h, with key-value head g = h // (n_heads / n_kv):
         s_j = (q_h . k_j) / sqrt(d) for slots j = 0 .. pos[b],
         p = exp(s - max s) / sum exp(s - max s),
         out_h = sum_j p_j v_j.
    Returns the output [B, n_heads * d] (double) and the updated caches."""
    q = np.asarray(q, np.float64)
    B = q.shape[0]
    d = head_dim
    nh = q.shape[1] // d
    group = nh // n_kv_heads
    kc = _u16(k_cache_bits).copy()
    vc = _u16(v_cache_bits).copy()
    kn = f64_to_bf16(np.asarray(k_new, np.float64))
    vn = f64_to_bf16(np.asarray(v_new, np.float64))
    out = np.zeros((B, nh * d), np.float64)
    for b in range(B):
        p_b = int(pos[b])
        for g in range(n_kv_heads):
            kc[b, g, p_b] = kn[b, g * d:(g + 1) * d]
            vc[b, g, p_b] = vn[b, g * d:(g + 1) * d]
        for h in range(nh):
            g = h // group
            K = bf16_to_f64(kc[b, g, :p_b + 1])      # [n, d]
            V = bf16_to_f64(vc[b, g, :p_b + 1])
            s = K @ q[b, h * d:(h + 1) * d] / np.sqrt(d)
            e = np.exp(s - s.max())
            out[b, h * d:(h + 1) * d] = (e / e.sum()) @ V
    return {"out": out, "k_cache": kc, "v_cache": vc}


def openmp_threads() -> int:
    return int(_load().ws_oracle_openmp_threads())

