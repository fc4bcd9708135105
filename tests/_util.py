"""Shared helpers for the tests: device transfer of bit patterns and the
comparison metrics (fp32: |g - r| / max(|r|, rms(r)) <= 2e-3 per row; bf16 and
fp16: at most 1 unit in the last place)."""
import contextlib

import numpy as np
import torch

FP32_TOL = 2e-3
ULP_TOL = 1

# The largest ulp distance each bf16-criterion check accepted (an element past
# 1 ulp passes only under the fp32 bound); printed at the end of the session
# so that drift in that margin shows.
ULP_SEEN: dict = {}


def note_ulps(what: str, max_ulp: int, frac_1ulp: float):
    import re
    key = re.sub(r"\s*block \d+\s*", " ", what).strip()
    old = ULP_SEEN.get(key)
    if old is None or max_ulp > old[0] or frac_1ulp < old[1]:
        ULP_SEEN[key] = (max(max_ulp, old[0] if old else 0), min(frac_1ulp, old[1] if old else 1.0))


@contextlib.contextmanager
def tuning(**fields):
    """The library's tuning with the given fields changed, restored after."""
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    base = wb.get_tuning()
    t = wb.Tuning()
    for f, _ in wb.Tuning._fields_:
        setattr(t, f, getattr(base, f))
    for k, v in fields.items():
        setattr(t, k, v)
    wb.set_tuning(t)
    try:
        yield
    finally:
        wb.set_tuning(base)


def dev_bf16(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dev_fp16(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).to(device)


def dev_f32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def host_bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16/fp16 tensor."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def rel_err_rows(got, ref) -> float:
    """max_i |g_i - r_i| / max(|r_i|, rms(r_row)) over every row."""
    got = np.asarray(got, np.float64).reshape(-1, np.asarray(ref).shape[-1])
    ref = np.asarray(ref, np.float64).reshape(got.shape)
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    scale = np.maximum(np.abs(ref), np.maximum(rms, 1e-30))
    return float(np.max(np.abs(got - ref) / scale))


def _ordered(bits):
    b = np.asarray(bits, np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_dist(a_bits, b_bits) -> np.ndarray:
    """Distance in units in the last place between two 16-bit float patterns."""
    return np.abs(_ordered(a_bits) - _ordered(b_bits))


def assert_fp32(got, ref, tol=FP32_TOL, what=""):
    e = rel_err_rows(got, ref)
    assert e <= tol, f"{what}: max relative error {e:.3g} > {tol}"
    return e


def assert_ulp(got_bits, ref_bits, tol=ULP_TOL, what=""):
    d = ulp_dist(got_bits, ref_bits)
    assert int(d.max()) <= tol, f"{what}: {int((d > tol).sum())} elements beyond {tol} ulp (max {int(d.max())})"
    return int(d.max())


def bf16_bits_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def fp16_bits_to_f64(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _bf16_neighbours(v):
    """The bf16 values just below and just above each double v."""
    import oracle
    bits = oracle.f64_to_bf16(v)
    r = bf16_bits_to_f64(bits)
    o = _ordered(bits)
    up = np.where(r >= v, o, o + 1)
    lo = np.where(r <= v, o, o - 1)

    def unorder(q):
        q = np.asarray(q, np.int32)
        return np.where(q < 0, (-q) | 0x8000, q).astype(np.uint16)
    return bf16_bits_to_f64(unorder(lo)), bf16_bits_to_f64(unorder(up))


def assert_mlp_block_close(got_bits, x_bits, blk, eps, what="", rel=FP32_TOL):
    """A LayerNorm -> Linear -> GELU block output.  The block rounds the Linear
    output t = x.W^T + b to bf16 before the GELU; that rounding is a decision
    on an fp32 value the oracle only knows to the fp32 tolerance.  Where t
    lies within that tolerance of a rounding boundary, either neighbour is a
    correct intermediate, and the GPU output must be within 1 ulp of the GELU
    of one of them (or, near a cancellation, within the fp32 bound)."""
    import oracle
    lin = oracle.mlp_block(x_bits, blk, eps, 8, linear=True)
    lo, hi = _bf16_neighbours(lin)
    rms = np.sqrt(np.mean(lin * lin, axis=1, keepdims=True))
    near = np.abs(lin - 0.5 * (lo + hi)) <= rel * np.maximum(np.abs(lin), rms)
    t_main = oracle.round_bf16(lin)
    t_alt = np.where(t_main == lo, hi, lo)
    got = np.asarray(got_bits, np.uint16).reshape(lin.shape)
    g = bf16_bits_to_f64(got)
    ok = np.zeros(lin.shape, bool)
    for t, allowed in ((t_main, np.ones_like(near)), (t_alt, near)):
        z = oracle.gelu(t)
        d = ulp_dist(got, oracle.f64_to_bf16(z)).reshape(lin.shape)
        zr = np.sqrt(np.mean(z * z, axis=1, keepdims=True))
        close = (d <= 1) | (np.abs(g - z) <= rel * np.maximum(np.abs(z), zr))
        ok |= allowed & close
    assert ok.all(), f"{what}: {int((~ok).sum())} elements off"
    d_main = ulp_dist(got, oracle.f64_to_bf16(oracle.gelu(t_main))).reshape(lin.shape)
    frac = float(np.mean(d_main <= 1))
    note_ulps(what or "mlp block", int(d_main.max()), frac)
    return frac


def assert_bf16_close(got_bits, exact, what="", rel=FP32_TOL, min_frac_1ulp=0.995):
    """bf16 outputs that are functions of fp32 dot products: each element is
    within 1 ulp of the correctly rounded oracle value, or -- where the value
    sits near a cancellation and fp32 accumulation legitimately moves it by
    more -- within the fp32 tolerance |g - r| <= rel * max(|r|, rms(row)).
    At least `min_frac_1ulp` of the elements must be within 1 ulp."""
    import oracle
    exact = np.asarray(exact, np.float64)
    ref_bits = oracle.f64_to_bf16(exact)
    d = ulp_dist(got_bits, ref_bits).reshape(exact.shape)
    g = bf16_bits_to_f64(got_bits).reshape(exact.shape)
    e2 = exact.reshape(-1, exact.shape[-1])
    rms = np.sqrt(np.mean(e2 * e2, axis=1, keepdims=True))
    scale = np.maximum(np.abs(e2), rms).reshape(exact.shape)
    ok = (d <= 1) | (np.abs(g - exact) <= rel * scale)
    frac = float(np.mean(d <= 1))
    note_ulps(what or "bf16", int(d.max()), frac)
    assert ok.all(), f"{what}: {int((~ok).sum())} elements outside both bounds"
    assert frac >= min_frac_1ulp, f"{what}: only {frac:.4f} of elements within 1 ulp"
    return frac
