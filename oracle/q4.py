"""4-bit group-128 weights for the oracle: the packed format, its
dequantisation, the GEMV over it in double, and the quantiser.

TEST INFRASTRUCTURE ONLY (see the package docstring): shares no code with the
CUDA library.

"One Token, Kernel by Kernel: A Decode Step on a Laptop GPU", "4-bit
weights": every linear layer, the LM head included, is quantised to 4-bit
integers in groups of 128, 0.82 GB of weights instead of 3.09 (3.76 times
smaller).  Readings where the pages are silent:

* a group is 128 consecutive weights of one row (along K); it carries a bf16
  scale s and a bf16 zero z, and code q in 0..15 stands for s * (q - 8) + z
  (the zero-point-in-the-float-domain form of the tinygemm kernel the pages
  name).  4 bits per weight plus 32 bits per 128 weights is 4.25 bits, which
  gives the pages' 0.82 GB and 3.76 times for Qwen2.5-1.5B;
* the quantiser is min-max per group, its decisions in fp32:
  s = bf16((max - min) / 15), z = bf16(min + 8 s),
  q = clamp(rint((w - z) / s) + 8, 0, 15) (q = 8 when s is 0);
* the byte layout is this project's own (the pages' kernel uses its own tiled
  layout): a row is a run of super-groups of four groups; a super-group holds
  its groups' codes (64 bytes each, in group order) followed by its groups'
  (s, z) pairs (4 bytes each, s first), zero-padded to a multiple of 16 bytes
  (272 bytes for four groups).  Within a group, 32-bit little-endian word i
  holds k = 8i .. 8i + 7: bits 4j .. 4j+3 hold k = 8i + 2j and bits
  16 + 4j .. 16 + 4j + 3 hold k = 8i + 2j + 1 (j = 0..3).
"""
from __future__ import annotations

import numpy as np

GROUP = 128
SUPER = 4  # groups per super-group


def _pad16(n: int) -> int:
    return (n + 15) // 16 * 16


def super_group_bytes(n_groups: int) -> int:
    """Bytes of a super-group of n_groups (1..4) groups."""
    return _pad16(n_groups * (GROUP // 2 + 4))


def row_bytes(K: int) -> int:
    """Bytes of one packed row of K weights (K a multiple of 128)."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    ng = K // GROUP
    full, tail = divmod(ng, SUPER)
    return full * super_group_bytes(SUPER) + (super_group_bytes(tail) if tail else 0)


def _bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _f32_to_bf16_bits(v) -> np.ndarray:
    """Round-to-nearest-even of fp32 values to bf16 bit patterns."""
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def unpack(packed, K: int):
    """Codes [M][K] (uint8, 0..15), scale bits and zero bits [M][K/128]
    (uint16) of packed rows [M][row_bytes(K)] (uint8)."""
    P = np.ascontiguousarray(packed, np.uint8)
    M = P.shape[0]
    if P.shape[1] != row_bytes(K):
        raise ValueError("packed row length does not match K")
    ng = K // GROUP
    codes = np.zeros((M, K), np.uint8)
    s = np.zeros((M, ng), np.uint16)
    z = np.zeros((M, ng), np.uint16)
    off = 0
    for g0 in range(0, ng, SUPER):
        n = min(SUPER, ng - g0)
        sg = P[:, off:off + super_group_bytes(n)]
        for gi in range(n):
            words = sg[:, gi * 64:(gi + 1) * 64].copy().view("<u4")  # [M][16]
            for i in range(16):
                w = words[:, i]
                for j in range(4):
                    k = (g0 + gi) * GROUP + 8 * i + 2 * j
                    codes[:, k] = (w >> (4 * j)) & 0xF
                    codes[:, k + 1] = (w >> (16 + 4 * j)) & 0xF
            pair = sg[:, n * 64 + gi * 4:n * 64 + gi * 4 + 4].copy().view("<u2")  # [M][2]
            s[:, g0 + gi] = pair[:, 0]
            z[:, g0 + gi] = pair[:, 1]
        off += super_group_bytes(n)
    return codes, s, z


def pack(codes, s_bits, z_bits) -> np.ndarray:
    """Packed rows from codes [M][K] and scale / zero bits [M][K/128]."""
    codes = np.asarray(codes, np.uint8)
    M, K = codes.shape
    ng = K // GROUP
    out = np.zeros((M, row_bytes(K)), np.uint8)
    off = 0
    for g0 in range(0, ng, SUPER):
        n = min(SUPER, ng - g0)
        for gi in range(n):
            c = codes[:, (g0 + gi) * GROUP:(g0 + gi + 1) * GROUP].astype(np.uint32)
            words = np.zeros((M, 16), np.uint32)
            for i in range(16):
                for j in range(4):
                    words[:, i] |= c[:, 8 * i + 2 * j] << (4 * j)
                    words[:, i] |= c[:, 8 * i + 2 * j + 1] << (16 + 4 * j)
            out[:, off + gi * 64:off + (gi + 1) * 64] = words.astype("<u4").view(np.uint8)
            pair = np.stack([np.asarray(s_bits)[:, g0 + gi], np.asarray(z_bits)[:, g0 + gi]],
                            axis=1).astype("<u2")
            out[:, off + n * 64 + gi * 4:off + n * 64 + gi * 4 + 4] = pair.view(np.uint8)
        off += super_group_bytes(n)
    return out


def dequant(packed, K: int) -> np.ndarray:
    """W [M][K] in double: s * (q - 8) + z per group (exact in double)."""
    codes, s, z = unpack(packed, K)
    S = np.repeat(_bf16_bits_to_f64(s), GROUP, axis=1)
    Z = np.repeat(_bf16_bits_to_f64(z), GROUP, axis=1)
    return S * (codes.astype(np.float64) - 8.0) + Z


def gemv(packed, K: int, x) -> np.ndarray:
    """y [B][M] = x W^T with W = dequant(packed): double products and sums."""
    W = dequant(packed, K)
    return np.asarray(x, np.float64) @ W.T


def quantize(W_bits):
    """Min-max 4-bit quantisation of bf16 weights [M][K] in groups of 128,
    every decision in fp32 (see the module docstring).  Returns codes
    [M][K] (uint8) and scale / zero bits [M][K/128] (uint16)."""
    Wb = np.asarray(W_bits, np.uint16)
    M, K = Wb.shape
    ng = K // GROUP
    w = (Wb.astype(np.uint32) << 16).view(np.float32).reshape(M, ng, GROUP)
    lo = w.min(axis=2)
    hi = w.max(axis=2)
    s32 = (hi - lo) / np.float32(15.0)
    s_bits = _f32_to_bf16_bits(s32)
    s_f = (s_bits.astype(np.uint32) << 16).view(np.float32)
    z32 = lo + np.float32(8.0) * s_f
    z_bits = _f32_to_bf16_bits(z32)
    z_f = (z_bits.astype(np.uint32) << 16).view(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        d = (w - z_f[:, :, None]) / s_f[:, :, None]
    q = np.rint(d) + np.float32(8.0)
    q = np.where(s_f[:, :, None] == 0, np.float32(8.0), q)
    q = np.clip(q, 0, 15).astype(np.uint8).reshape(M, K)
    return q, s_bits, z_bits


def qwen_block(h, blk: dict, attn, eps: float) -> dict:
    """One decoder block with 4-bit weights (the module docstring's reading),
    the same steps as the bf16 block with every product over the dequantised
    rows: blk holds bf16 bits gamma1, gamma2 and packed rows Wq, Wk, Wv, Wo,
    Wg, Wu, Wd with their K in blk["K"] (hidden) and blk["KI"] (inter)."""
    from . import bf16_to_f64, f64_to_bf16, rmsnorm, round_bf16, round_f32, swiglu
    H, I = blk["K"], blk["KI"]
    a = round_bf16(rmsnorm(h, bf16_to_f64(blk["gamma1"]), eps))
    q, k, v = (gemv(blk[n], H, a) for n in ("Wq", "Wk", "Wv"))
    h1 = round_f32(np.asarray(h, np.float64) + gemv(blk["Wo"], H, attn))
    m = round_bf16(rmsnorm(h1, bf16_to_f64(blk["gamma2"]), eps))
    s_bits = f64_to_bf16(swiglu(gemv(blk["Wg"], H, m), gemv(blk["Wu"], H, m)))
    h2 = round_f32(h1 + gemv(blk["Wd"], I, bf16_to_f64(s_bits)))
    return {"q": q, "k": k, "v": v, "h_mid": h1, "s": s_bits, "h": h2}


def lmhead_logits(h, gamma_bits, Wlm, K: int, eps: float) -> np.ndarray:
    from . import bf16_to_f64, rmsnorm, round_bf16
    return gemv(Wlm, K, round_bf16(rmsnorm(h, bf16_to_f64(gamma_bits), eps)))
