"""Pins of the CPU oracle against facts that do not come from the oracle itself:
library conversions, closed forms, invariants, brute force in exact rational
arithmetic, and the figures the pages print.  No GPU needed."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from weight_streaming_gemv_bf16_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- formats

def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_encode_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(1)
    # normals over a wide exponent range, subnormals, exact ties
    v = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.integers(-140, 120, 20000)),
        rng.standard_normal(2000) * 1e-39,
        (np.arange(-300, 300) * 2.0 + 1.0) * 2.0 ** -8,  # halfway between bf16 steps near 1
    ]).astype(np.float32)
    ours = oracle.f64_to_bf16(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("value,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),          # tie -> even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),      # tie -> even (up)
    (-2.0, 0xC000),
    (2.0 ** -133, 0x0001),              # smallest subnormal
    (2.0 ** -134, 0x0000),              # tie with zero -> even (zero)
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),   # largest finite
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),   # tie above largest -> infinity
])
def test_bf16_encode_ieee_cases(value, bits):
    assert int(oracle.f64_to_bf16(np.array([value]))[0]) == bits


def test_fp16_decode_and_encode_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.fp16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.integers(-30, 18, 20000)),
        (np.arange(-500, 500) * 2.0 + 1.0) * 2.0 ** -11,   # ties near 1
        np.array([65504.0, 65519.99, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26]),
    ])
    assert np.array_equal(oracle.f64_to_fp16(v), v.astype(np.float16).view(np.uint16))


# ---------------------------------------------------------------- GEMV

def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_gemv_identity_and_permutation_are_exact():
    K = 64
    x = oracle.round_bf16(np.random.default_rng(3).standard_normal((3, K)))
    assert np.array_equal(oracle.gemv(_bf16(np.eye(K)), x), x)
    perm = np.random.default_rng(4).permutation(K)
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), perm] = 1.0                      # row m picks x[perm[m]]
    assert np.array_equal(oracle.gemv(_bf16(P), x), x[:, perm])


def test_gemv_one_hot_picks_the_column():
    M, K = 5, 40
    W = np.zeros((M, K), np.float32)
    cols = [0, 7, 39, 12, 7]
    for m, c in enumerate(cols):
        W[m, c] = 2.0 ** m
    x = oracle.round_bf16(np.random.default_rng(5).standard_normal((2, K)))
    y = oracle.gemv(_bf16(W), x)
    for m, c in enumerate(cols):
        assert np.array_equal(y[:, m], x[:, c] * 2.0 ** m)


def test_gemv_all_ones():
    for K in (8, 1536, 8960):
        y = oracle.gemv(_bf16(np.ones((3, K))), np.ones((2, K)))
        assert np.all(y == K)


def test_gemv_brute_force_exact_rational():
    """16x16 and a non-square 12x20 case, summed exactly with Fractions."""
    for (M, K, B, seed) in [(16, 16, 1, 6), (16, 16, 4, 7), (12, 20, 3, 8)]:
        W = synth.normal_bf16((M, K), 1.0, seed, "bf")
        xb = synth.normal_bf16((B, K), 1.0, seed, "bx")
        Wd, xd = oracle.bf16_to_f64(W), oracle.bf16_to_f64(xb)
        y = oracle.gemv(W, xd)
        for b in range(B):
            for m in range(M):
                exact = sum(Fraction(float(Wd[m, k])) * Fraction(float(xd[b, k])) for k in range(K))
                scale = sum(abs(Fraction(float(Wd[m, k])) * Fraction(float(xd[b, k]))) for k in range(K))
                assert abs(Fraction(float(y[b, m])) - exact) <= scale * Fraction(1, 2 ** 50)
                # both round to the same binary32 value
                assert np.float32(float(exact)) == np.float32(y[b, m]) or \
                    abs(float(exact) - y[b, m]) <= 2 ** -40 * float(scale)


def test_gemv_linearity():
    M, K = 64, 1536
    W = synth.normal_bf16((M, K), 0.02, 0, "lin/W")
    x = oracle.bf16_to_f64(synth.normal_bf16((1, K), 1.0, 0, "lin/x"))
    z = oracle.bf16_to_f64(synth.normal_bf16((1, K), 1.0, 0, "lin/z"))
    lhs = oracle.gemv(W, 2 * x + z / 4)
    rhs = 2 * oracle.gemv(W, x) + oracle.gemv(W, z) / 4
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-13)


def test_gemv_thread_count_does_not_change_result():
    W = synth.normal_bf16((257, 96), 0.02, 0, "thr/W")
    x = oracle.bf16_to_f64(synth.normal_bf16((3, 96), 1.0, 0, "thr/x"))
    assert np.array_equal(oracle.gemv(W, x, threads=1), oracle.gemv(W, x, threads=4))


# ---------------------------------------------------------------- norms

def test_rmsnorm_unit_rms_invariant():
    x = np.random.default_rng(9).standard_normal((4, 1536)) * 3.0
    eps = 1e-6
    out = oracle.rmsnorm(x, np.ones(1536), eps)
    ms = np.mean(x * x, axis=1)
    assert np.allclose(np.sqrt(np.mean(out * out, axis=1)), np.sqrt(ms / (ms + eps)), rtol=1e-12)


def test_rmsnorm_eps_inside_the_square_root_and_gamma_per_column():
    # constant rows: out = c / sqrt(c^2 + eps) * gamma  (eps inside the root)
    c, eps = 0.01, 1e-4
    g = np.linspace(0.5, 1.5, 8)
    out = oracle.rmsnorm(np.full((1, 8), c), g, eps)
    assert np.allclose(out[0], c / math.sqrt(c * c + eps) * g, rtol=1e-14)
    # gamma multiplies column-wise
    x = np.random.default_rng(10).standard_normal((2, 8))
    assert np.allclose(oracle.rmsnorm(x, g, eps), oracle.rmsnorm(x, np.ones(8), eps) * g, rtol=1e-14)


def test_rmsnorm_scale_invariance_without_eps():
    x = np.random.default_rng(11).standard_normal((3, 896))
    g = np.random.default_rng(12).uniform(0.5, 1.5, 896)
    assert np.allclose(oracle.rmsnorm(x * 1024.0, g, 0.0), oracle.rmsnorm(x, g, 0.0), rtol=1e-13)


def test_layernorm_moments_and_shift_invariance():
    x = np.random.default_rng(13).standard_normal((4, 768)) * 2 + 5
    out = oracle.layernorm(x, np.full(768, 3.0), np.full(768, -0.25), 0.0)
    assert np.allclose(out.mean(axis=1), -0.25, atol=1e-12)
    assert np.allclose(out.var(axis=1), 9.0, rtol=1e-12)
    g = np.random.default_rng(14).uniform(0.5, 1.5, 768)
    bt = np.random.default_rng(15).standard_normal(768) * 0.02
    assert np.allclose(oracle.layernorm(x + 7.0, g, bt, 1e-5), oracle.layernorm(x, g, bt, 1e-5), atol=1e-12)
    # two elements: (x - mean) / sqrt(var + eps) = +-d / sqrt(d^2 + eps)
    d, eps = 0.5, 1e-5
    out2 = oracle.layernorm(np.array([[1.0 - d, 1.0 + d]]), np.ones(2), np.zeros(2), eps)
    assert np.allclose(out2[0], [-d / math.sqrt(d * d + eps), d / math.sqrt(d * d + eps)], rtol=1e-14)


# ---------------------------------------------------------------- activations

def test_gelu_against_the_normal_table():
    for z, phi in _golden("normal_cdf.txt"):
        z, phi = float(z), float(phi)
        assert abs(oracle.gelu(np.array([z]))[0] - z * phi) <= z * 6e-10
        assert abs(oracle.gelu(np.array([-z]))[0] - (-z) * (1 - phi)) <= z * 6e-10
    assert oracle.gelu(np.array([0.0]))[0] == 0.0


def test_gelu_odd_part_identity():
    z = np.random.default_rng(16).standard_normal(1000) * 4
    assert np.allclose(oracle.gelu(z) - oracle.gelu(-z), z, atol=1e-14)


def test_swiglu_closed_forms():
    # silu(ln 3) = ln 3 * 3/4 ; silu(0) = 0 ; silu(g) - silu(-g) = g ; u scales linearly
    ln3 = math.log(3.0)
    assert abs(oracle.swiglu(np.array([ln3]), np.array([1.0]))[0] - 0.75 * ln3) < 1e-15
    assert oracle.swiglu(np.array([0.0]), np.array([5.0]))[0] == 0.0
    g = np.random.default_rng(17).standard_normal(1000) * 6
    one = np.ones_like(g)
    assert np.allclose(oracle.swiglu(g, one) - oracle.swiglu(-g, one), g, atol=1e-13)
    assert np.allclose(oracle.swiglu(g, 3 * one), 3 * oracle.swiglu(g, one), rtol=1e-15)
    assert abs(oracle.swiglu(np.array([40.0]), np.array([1.0]))[0] - 40.0) < 1e-15


# ---------------------------------------------------------------- argmax

def test_argmax_planted_and_ties():
    v = np.random.default_rng(18).standard_normal((3, 151936))
    v[0, 123456] = 10.0
    v[1, 5] = v[1, 99] = v[1, 151935] = 10.0     # ties -> lowest index
    v[2, :] = -1.0                               # all equal -> 0
    assert list(oracle.argmax_rows(v)) == [123456, 5, 0]


# ---------------------------------------------------------------- block structure

def _tiny_block(H, KV, I, seed):
    t = f"tiny{seed}/"
    return {
        "gamma1": synth.uniform_bf16((H,), 0.5, 1.5, seed, t + "g1"),
        "Wq": synth.normal_bf16((H, H), 0.02, seed, t + "Wq"),
        "Wk": synth.normal_bf16((KV, H), 0.02, seed, t + "Wk"),
        "Wv": synth.normal_bf16((KV, H), 0.02, seed, t + "Wv"),
        "Wo": synth.normal_bf16((H, H), 0.02, seed, t + "Wo"),
        "gamma2": synth.uniform_bf16((H,), 0.5, 1.5, seed, t + "g2"),
        "Wg": synth.normal_bf16((I, H), 0.02, seed, t + "Wg"),
        "Wu": synth.normal_bf16((I, H), 0.02, seed, t + "Wu"),
        "Wd": synth.normal_bf16((H, I), 0.02, seed, t + "Wd"),
    }


def test_block_special_cases_expose_each_step():
    H, KV, I, B = 32, 8, 32, 2
    eps = 1e-6
    blk = _tiny_block(H, KV, I, 0)
    h = oracle.bf16_to_f64(synth.normal_bf16((B, H), 1.0, 0, "tiny/h"))
    attn = oracle.bf16_to_f64(synth.normal_bf16((B, H), 1.0, 0, "tiny/attn"))
    g1 = oracle.bf16_to_f64(blk["gamma1"])
    g2 = oracle.bf16_to_f64(blk["gamma2"])
    zero = lambda a: np.zeros_like(a)
    eye = _bf16(np.eye(H))

    # zero Wo and Wd: the residual passes through unchanged
    z = dict(blk, Wo=zero(blk["Wo"]), Wd=zero(blk["Wd"]))
    out = oracle.qwen_block(h, z, attn, eps)
    assert np.array_equal(out["h"], h)

    # Wq = I: q is the bf16-rounded RMSNorm of h with gamma1 (not gamma2)
    out = oracle.qwen_block(h, dict(blk, Wq=eye), attn, eps)
    ms = np.mean(h * h, axis=1, keepdims=True)
    a_ref = torch.from_numpy(h / np.sqrt(ms + eps) * g1).to(torch.bfloat16).double().numpy()
    assert np.allclose(out["q"], a_ref, rtol=0, atol=0) or np.max(np.abs(out["q"] - a_ref)) <= 2 ** -8 * np.max(np.abs(a_ref))

    # Wo = I, Wd = 0: h_mid = h + attn (the attention stand-in, not a)
    out = oracle.qwen_block(h, dict(blk, Wo=eye, Wd=zero(blk["Wd"])), attn, eps)
    assert np.allclose(out["h"], h + attn, rtol=1e-7)

    # Wg = Wu = I, Wd = I (I == H): h = h_mid + bf16(silu(m) * m), m from gamma2
    out = oracle.qwen_block(h, dict(blk, Wg=eye, Wu=eye, Wd=eye), attn, eps)
    hm = out["h_mid"]
    ms = np.mean(hm * hm, axis=1, keepdims=True)
    m = torch.from_numpy(hm / np.sqrt(ms + eps) * g2).to(torch.bfloat16).double().numpy()
    s = torch.from_numpy(m * m / (1 + np.exp(-m))).to(torch.bfloat16).double().numpy()
    assert np.max(np.abs(out["h"] - (hm + s))) <= 2 ** -7 * np.max(np.abs(s)) + 1e-6


def test_chain_identity_head_picks_the_largest_normalised_element():
    H, KV, I, B, L = 32, 8, 32, 3, 2
    blocks = [_tiny_block(H, KV, I, s) for s in range(L)]
    attns = [oracle.bf16_to_f64(synth.normal_bf16((B, H), 1.0, s, "tiny/attn")) for s in range(L)]
    h0 = oracle.bf16_to_f64(synth.normal_bf16((B, H), 1.0, 0, "tiny/h"))
    gf = _bf16(np.ones(H))
    out = oracle.qwen_chain(h0, blocks, attns, gf, _bf16(np.eye(H)), 1e-6, keep_blocks=True)
    a = oracle.round_bf16(oracle.rmsnorm(out["h"], np.ones(H), 1e-6))
    assert np.array_equal(out["logits"], a)
    assert list(out["idx"]) == [int(np.argmax(r)) for r in a]
    assert np.array_equal(out["blocks"][-1]["h"], out["h"])
    # block l's output is block l+1's input
    again = oracle.qwen_block(out["blocks"][0]["h"], blocks[1], attns[1], 1e-6)
    assert np.array_equal(again["h"], out["h"])


def test_mlp_block_zero_weight_reduces_to_gelu_of_bias():
    w, B = 16, 2
    blk = {"gamma": _bf16(np.ones(w)), "beta": _bf16(np.zeros(w)),
           "W": _bf16(np.zeros((w, w))), "b": synth.normal_bf16((w,), 1.0, 0, "mlpz/b")}
    x = synth.normal_bf16((B, w), 1.0, 0, "mlpz/x")
    z = oracle.mlp_block(x, blk)
    bvals = oracle.bf16_to_f64(blk["b"])
    ref = torch.from_numpy(bvals).to(torch.bfloat16).float()
    ref = torch.nn.functional.gelu(ref.double()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(z, np.broadcast_to(ref, (B, w)))


def test_mlp_block_identity_weight_reduces_to_gelu_of_layernorm():
    w, B = 16, 2
    g = synth.uniform_bf16((w,), 0.5, 1.5, 0, "mlpi/g")
    bt = synth.normal_bf16((w,), 0.02, 0, "mlpi/bt")
    blk = {"gamma": g, "beta": bt, "W": _bf16(np.eye(w)), "b": _bf16(np.zeros(w))}
    x = synth.normal_bf16((B, w), 1.0, 0, "mlpi/x")
    z = oracle.bf16_to_f64(oracle.mlp_block(x, blk))
    xt = torch.from_numpy(oracle.bf16_to_f64(x))
    ln = torch.nn.functional.layer_norm(xt, (w,), torch.from_numpy(oracle.bf16_to_f64(g)),
                                        torch.from_numpy(oracle.bf16_to_f64(bt)), 1e-5)
    ref = torch.nn.functional.gelu(ln.to(torch.bfloat16).double()).to(torch.bfloat16).double().numpy()
    assert np.array_equal(z, ref)


# ---------------------------------------------------------------- the pages' figures

def test_workload_shapes_reproduce_the_pages_byte_counts():
    s = synth.QWEN2_5_1_5B
    vals = {}
    for key, value, _unit, digits, *_where in _golden("qwen2_5_1_5b_bytes.txt"):
        vals[key] = (float(value), int(digits))

    def close(x, key):
        v, d = vals[key]
        if d == 0:
            return x == v
        return abs(x - v) <= 0.5 * 10 ** (math.floor(math.log10(v)) - d + 1)

    assert close(s.chain_weight_bytes(), "chain_weight_bytes")
    assert close(s.lm_head_bytes(), "lm_head_bytes")
    assert close(2 * s.kv_dim * s.hidden, "kv_proj_bytes")
    assert close(7 * s.layers + 1, "gemv_count")
    assert close(s.vocab, "lm_head_rows") and close(s.hidden, "lm_head_cols")


# --------------------------------------------------------------------------
# decode attention over a key-value cache
# --------------------------------------------------------------------------

def _attn_case(rng, B, nkv, S, d, nh, ints=False):
    def draw(shape):
        v = rng.integers(-8, 9, size=shape).astype(np.float64) if ints else rng.standard_normal(shape)
        return v
    q = draw((B, nh * d))
    kn, vn = draw((B, nkv * d)), draw((B, nkv * d))
    kc = oracle.f64_to_bf16(draw((B, nkv, S, d)))
    vc = oracle.f64_to_bf16(draw((B, nkv, S, d)))
    return q, kn, vn, kc, vc


def test_attention_single_slot_returns_the_new_value():
    """pos = 0: the softmax has one term, so every query head returns its
    group's new value, rounded to bf16 (the cache's type), exactly."""
    rng = np.random.default_rng(1)
    B, nkv, S, d, nh = 2, 2, 8, 16, 6
    q, kn, vn, kc, vc = _attn_case(rng, B, nkv, S, d, nh)
    r = oracle.decode_attention(q, kn, vn, kc, vc, np.zeros(B, np.int32), nkv, d)
    group = nh // nkv
    for b in range(B):
        for h in range(nh):
            g = h // group
            want = oracle.bf16_to_f64(oracle.f64_to_bf16(vn[b, g * d:(g + 1) * d]))
            assert np.array_equal(r["out"][b, h * d:(h + 1) * d], want)


def test_attention_appends_at_pos_and_leaves_other_slots():
    rng = np.random.default_rng(2)
    B, nkv, S, d, nh = 3, 2, 16, 8, 4
    q, kn, vn, kc, vc = _attn_case(rng, B, nkv, S, d, nh)
    pos = np.array([0, 7, 15])
    r = oracle.decode_attention(q, kn, vn, kc, vc, pos, nkv, d)
    for b in range(B):
        for g in range(nkv):
            assert np.array_equal(r["k_cache"][b, g, pos[b]], oracle.f64_to_bf16(kn[b, g * d:(g + 1) * d]))
            assert np.array_equal(r["v_cache"][b, g, pos[b]], oracle.f64_to_bf16(vn[b, g * d:(g + 1) * d]))
            keep = np.arange(S) != pos[b]
            assert np.array_equal(r["k_cache"][b, g][keep], kc[b, g][keep])
            assert np.array_equal(r["v_cache"][b, g][keep], vc[b, g][keep])


def test_attention_zero_query_averages_the_values():
    """q = 0: every score is 0, the weights are uniform and the output is the
    mean of the group's value rows over slots 0 .. pos."""
    rng = np.random.default_rng(3)
    B, nkv, S, d, nh = 2, 2, 32, 8, 4
    _, kn, vn, kc, vc = _attn_case(rng, B, nkv, S, d, nh)
    q = np.zeros((B, nh * d))
    pos = np.array([9, 31])
    r = oracle.decode_attention(q, kn, vn, kc, vc, pos, nkv, d)
    for b in range(B):
        for h in range(nh):
            g = h // (nh // nkv)
            V = oracle.bf16_to_f64(r["v_cache"][b, g, :pos[b] + 1])
            assert np.allclose(r["out"][b, h * d:(h + 1) * d], V.mean(axis=0), rtol=0, atol=1e-12)


def test_attention_two_slots_closed_form():
    """Two slots: the weight of slot 0 is the logistic function of the score
    difference divided by sqrt(d) (pins the scale and the sign)."""
    d = 16
    q = np.zeros((1, d)); q[0, 0] = 2.0
    k0 = np.zeros(d); k0[0] = 1.5
    k1 = np.zeros(d); k1[0] = -0.5
    v0 = np.arange(d, dtype=np.float64)
    v1 = -2.0 * np.ones(d)
    kc = oracle.f64_to_bf16(np.stack([k0, np.zeros(d)])[None, None])
    vc = oracle.f64_to_bf16(np.stack([v0, np.zeros(d)])[None, None])
    r = oracle.decode_attention(q, k1[None], v1[None], kc, vc, np.array([1]), 1, d)
    s0, s1 = q[0] @ k0, q[0] @ k1
    p0 = 1.0 / (1.0 + math.exp((s1 - s0) / math.sqrt(d)))
    assert np.allclose(r["out"][0], p0 * v0 + (1 - p0) * v1, rtol=0, atol=1e-12)


def test_attention_slot_order_does_not_matter():
    rng = np.random.default_rng(4)
    B, nkv, S, d, nh = 1, 2, 24, 8, 6
    q, kn, vn, kc, vc = _attn_case(rng, B, nkv, S, d, nh)
    pos = np.array([20])
    r1 = oracle.decode_attention(q, kn, vn, kc, vc, pos, nkv, d)
    perm = np.concatenate([rng.permutation(20), np.arange(20, S)])
    r2 = oracle.decode_attention(q, kn, vn, kc[:, :, perm], vc[:, :, perm], pos, nkv, d)
    assert np.allclose(r1["out"], r2["out"], rtol=0, atol=1e-12)


def test_attention_is_linear_in_the_values():
    """With integer-valued caches (exact in bf16) the output for V1 + V2 is
    the sum of the outputs for V1 and V2 (same keys, same weights)."""
    rng = np.random.default_rng(5)
    B, nkv, S, d, nh = 2, 2, 16, 8, 4
    q, kn, vn1, kc, vc1 = _attn_case(rng, B, nkv, S, d, nh, ints=True)
    _, _, vn2, _, vc2 = _attn_case(rng, B, nkv, S, d, nh, ints=True)
    pos = np.array([5, 15])
    vc12 = oracle.f64_to_bf16(oracle.bf16_to_f64(vc1) + oracle.bf16_to_f64(vc2))
    r1 = oracle.decode_attention(q, kn, vn1, kc, vc1, pos, nkv, d)
    r2 = oracle.decode_attention(q, kn, vn2, kc, vc2, pos, nkv, d)
    r12 = oracle.decode_attention(q, kn, vn1 + vn2, kc, vc12, pos, nkv, d)
    assert np.allclose(r12["out"], r1["out"] + r2["out"], rtol=0, atol=1e-9)


def test_attention_query_heads_share_their_group():
    """Query heads of one group with equal queries give equal outputs; heads
    of another group read the other key-value head."""
    rng = np.random.default_rng(6)
    B, nkv, S, d, nh = 1, 2, 16, 8, 4   # groups of 2 heads
    q, kn, vn, kc, vc = _attn_case(rng, B, nkv, S, d, nh)
    q[0, d:2 * d] = q[0, 0:d]            # heads 0 and 1 (group 0) equal
    q[0, 2 * d:3 * d] = q[0, 0:d]        # head 2 (group 1) equal too
    r = oracle.decode_attention(q, kn, vn, kc, vc, np.array([10]), nkv, d)
    o = r["out"][0].reshape(nh, d)
    assert np.array_equal(o[0], o[1])
    assert not np.allclose(o[0], o[2])


# ---- 4-bit group-128 weights ("One Token, Kernel by Kernel", "4-bit weights")

from oracle import q4 as oq4  # noqa: E402


def _bf16_value(bits):
    import struct
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def test_q4_golden_group_layout_and_dequant():
    """One group (K = 128) written byte by byte from the format: codes
    q_k = k mod 16 give word 0x75316420 for k = 0..7 (even k in the low
    half's nibbles 0..3, odd k in the high half's) and 0xFDB9ECA8 for
    k = 8..15; scale 0.5 (0x3F00), zero -1.0 (0xBF80) right after the 64
    bytes of codes, padded to 80 bytes.  Weight k is 0.5 (k mod 16 - 8) - 1."""
    import struct
    row = b"".join(struct.pack("<II", 0x75316420, 0xFDB9ECA8) for _ in range(8))
    row += struct.pack("<HH", 0x3F00, 0xBF80) + bytes(12)
    assert len(row) == 80 == oq4.row_bytes(128)
    P = np.frombuffer(row, np.uint8)[None, :]
    W = oq4.dequant(P, 128)
    assert np.array_equal(W[0], [0.5 * (k % 16 - 8) - 1.0 for k in range(128)])


def test_q4_super_group_and_tail_layout():
    """K = 640: one super-group of four groups (4 x 64 bytes of codes, then
    the four (s, z) pairs, 272 bytes) and a tail of one group (64 + 4 bytes
    padded to 80).  All codes 8, so each weight is its group's zero, here
    g + 1 for group g; scale 1."""
    import struct
    zero_bits = [0x3F80, 0x4000, 0x4040, 0x4080, 0x40A0]  # 1, 2, 3, 4, 5
    codes8 = struct.pack("<I", 0x88888888) * 16
    row = codes8 * 4 + b"".join(struct.pack("<HH", 0x3F80, z) for z in zero_bits[:4])
    row += codes8 + struct.pack("<HH", 0x3F80, zero_bits[4]) + bytes(12)
    assert len(row) == 352 == oq4.row_bytes(640)
    W = oq4.dequant(np.frombuffer(row, np.uint8)[None, :], 640)
    for g in range(5):
        assert np.all(W[0, g * 128:(g + 1) * 128] == g + 1)
    # the Qwen2.5-1.5B row lengths: 3 super-groups; 17 and a tail of two groups
    assert oq4.row_bytes(1536) == 3 * 272
    assert oq4.row_bytes(8960) == 17 * 272 + 144


def _brute_q4_row(row_bytes, K):
    """Weights of one packed row by plain loops over bytes (nibble m of a
    32-bit word, m = 0..7 from the least significant bits, is weight 2m for
    m < 4 and 2(m - 4) + 1 for m >= 4 of the word's eight)."""
    out = [0.0] * K
    ng = K // 128
    off = 0
    for g0 in range(0, ng, 4):
        n = min(4, ng - g0)
        for gi in range(n):
            g = g0 + gi
            sb = row_bytes[off + 64 * n + 4 * gi] | (row_bytes[off + 64 * n + 4 * gi + 1] << 8)
            zb = row_bytes[off + 64 * n + 4 * gi + 2] | (row_bytes[off + 64 * n + 4 * gi + 3] << 8)
            s, z = _bf16_value(sb), _bf16_value(zb)
            for i in range(16):
                b0 = off + 64 * gi + 4 * i
                word = sum(row_bytes[b0 + t] << (8 * t) for t in range(4))
                for m in range(8):
                    q = (word >> (4 * m)) & 15
                    kk = 2 * m if m < 4 else 2 * (m - 4) + 1
                    out[g * 128 + 8 * i + kk] = s * (q - 8) + z
        off += ((64 + 4) * n + 15) // 16 * 16
    return out


def test_q4_gemv_matches_brute_force():
    rng = np.random.default_rng(5)
    M, K, B = 3, 640, 2
    codes = rng.integers(0, 16, size=(M, K), dtype=np.uint8)
    s = oracle.f64_to_bf16(rng.uniform(0.001, 0.01, size=(M, K // 128)))
    z = oracle.f64_to_bf16(rng.normal(0, 0.01, size=(M, K // 128)))
    P = oq4.pack(codes, s, z)
    x = oracle.bf16_to_f64(oracle.f64_to_bf16(rng.normal(size=(B, K))))
    y = oq4.gemv(P, K, x)
    for m in range(M):
        w = _brute_q4_row([int(v) for v in P[m]], K)
        for b in range(B):
            ref = sum(w[k] * x[b, k] for k in range(K))
            assert abs(y[b, m] - ref) <= 1e-12 * max(1.0, abs(ref))
    cu, su, zu = oq4.unpack(P, K)
    assert np.array_equal(cu, codes) and np.array_equal(su, s) and np.array_equal(zu, z)


def test_q4_gemv_all_codes_eight_is_zero_times_group_sums():
    rng = np.random.default_rng(6)
    M, K = 4, 512
    z = oracle.f64_to_bf16(rng.normal(0, 1, size=(M, K // 128)))
    s = oracle.f64_to_bf16(rng.uniform(0.1, 1, size=(M, K // 128)))
    P = oq4.pack(np.full((M, K), 8, np.uint8), s, z)
    x = rng.normal(size=(1, K))
    zg = oracle.bf16_to_f64(z)
    ref = [sum(zg[m, g] * x[0, g * 128:(g + 1) * 128].sum() for g in range(K // 128))
           for m in range(M)]
    assert np.allclose(oq4.gemv(P, K, x)[0], ref, rtol=1e-12, atol=1e-12)


def test_q4_quantizer_error_bound_and_special_groups():
    rng = np.random.default_rng(7)
    M, K = 6, 512
    W = rng.normal(0, 0.02, size=(M, K))
    W[1, :128] = 0.25            # a constant group: scale 0, codes 8, exact
    W[2, 128:256] = np.linspace(-1, 1, 128)
    Wb = oracle.f64_to_bf16(W)
    codes, s, z = oq4.quantize(Wb)
    assert codes.min() >= 0 and codes.max() <= 15
    assert s[1, 0] == 0 and np.all(codes[1, :128] == 8)
    Wq = oq4.dequant(oq4.pack(codes, s, z), K)
    w = oracle.bf16_to_f64(Wb)
    sg = np.repeat(oracle.bf16_to_f64(s), 128, axis=1)
    zg = np.repeat(oracle.bf16_to_f64(z), 128, axis=1)
    # half a step, plus what rounding s and z to bf16 moves the grid's ends by
    bound = 0.5 * sg + 2.0 ** -8 * (np.abs(zg) + 8 * sg) + 1e-30
    assert np.all(np.abs(Wq - w) <= bound)
    assert np.all(Wq[1, :128] == 0.25)
    # a group's minimum and maximum land on the end codes (within one step)
    g = codes[2, 128:256]
    assert g[0] <= 1 and g[-1] >= 14


def test_q4_model_size_matches_the_pages():
    """Qwen2.5-1.5B's linear layers and LM head: 3.09 GB in bf16, 0.82 GB in
    this format, 3.76 times smaller (the pages' figures)."""
    blk = [(1536, 1536), (256, 1536), (256, 1536), (1536, 1536), (8960, 1536),
           (8960, 1536), (1536, 8960)]
    bf16 = 28 * sum(M * K * 2 for M, K in blk) + 151936 * 1536 * 2
    q4b = 28 * sum(M * oq4.row_bytes(K) for M, K in blk) + 151936 * oq4.row_bytes(1536)
    assert round(bf16 / 1e9, 2) == 3.09
    assert round(q4b / 1e9, 2) == 0.82
    assert round(bf16 / q4b, 2) == 3.76


def test_qwen_block_attention_with_constant_values_reduces_to_wo_of_that_row():
    """Every value row (cached and new) equal to one row c: attention returns
    c whatever the scores, so the block equals h + bf16(c).Wo^T followed by
    the MLP, as the stand-in block computes it with attn = c; the new key
    lands at pos."""
    rng = np.random.default_rng(31)
    H, KV, I, B, S = 256, 128, 256, 2, 64
    blk = {
        "gamma1": oracle.f64_to_bf16(rng.uniform(0.5, 1.5, H)),
        "gamma2": oracle.f64_to_bf16(rng.uniform(0.5, 1.5, H)),
        "Wq": oracle.f64_to_bf16(rng.normal(0, 0.05, (H, H))),
        "Wk": oracle.f64_to_bf16(rng.normal(0, 0.05, (KV, H))),
        "Wv": np.zeros((KV, H), np.uint16),          # v = 0 for the new token
        "Wo": oracle.f64_to_bf16(rng.normal(0, 0.05, (H, H))),
        "Wg": oracle.f64_to_bf16(rng.normal(0, 0.05, (I, H))),
        "Wu": oracle.f64_to_bf16(rng.normal(0, 0.05, (I, H))),
        "Wd": oracle.f64_to_bf16(rng.normal(0, 0.05, (H, I))),
    }
    h = rng.normal(size=(B, H))
    kc = oracle.f64_to_bf16(rng.normal(size=(B, 1, S, 128)))
    vc = np.zeros((B, 1, S, 128), np.uint16)        # every cached value row is 0
    pos = [10, 63]
    out = oracle.qwen_block_attention(h, blk, kc, vc, pos, 1, 1e-6)
    assert np.all(out["attn"] == 0)                 # attention of constant 0 rows
    ref = oracle.qwen_block(h, blk, np.zeros((B, H)), 1e-6)
    assert np.array_equal(out["h"], ref["h"])
    a = oracle.round_bf16(oracle.rmsnorm(h, oracle.bf16_to_f64(blk["gamma1"]), 1e-6))
    k_new = oracle.f64_to_bf16(oracle.gemv(blk["Wk"], a))
    for b, p in enumerate(pos):
        assert np.array_equal(out["k_cache"][b, 0, p], k_new[b])
        assert np.array_equal(np.delete(out["k_cache"][b, 0], p, axis=0),
                              np.delete(kc[b, 0], p, axis=0))


def test_q4_block_with_all_codes_eight_is_the_bf16_block_of_the_zeros():
    """Every code 8: each 4-bit weight equals its group's bf16 zero, so the
    4-bit block equals the bf16 block whose matrices hold those zeros (the
    steps and roundings of the two oracles must agree)."""
    rng = np.random.default_rng(41)
    H, KV, I, B = 256, 128, 384, 2
    shapes = {"Wq": (H, H), "Wk": (KV, H), "Wv": (KV, H), "Wo": (H, H), "Wg": (I, H),
              "Wu": (I, H), "Wd": (H, I)}
    q4blk, bfblk = {"K": H, "KI": I}, {}
    for n in ("gamma1", "gamma2"):
        q4blk[n] = bfblk[n] = oracle.f64_to_bf16(rng.uniform(0.5, 1.5, H))
    for n, (M, K) in shapes.items():
        z = oracle.f64_to_bf16(rng.normal(0, 0.05, (M, K // 128)))
        s = oracle.f64_to_bf16(rng.uniform(0.001, 0.01, (M, K // 128)))
        q4blk[n] = oq4.pack(np.full((M, K), 8, np.uint8), s, z)
        bfblk[n] = np.repeat(z, 128, axis=1)
    h = rng.normal(size=(B, H))
    attn = oracle.bf16_to_f64(oracle.f64_to_bf16(rng.normal(size=(B, H))))
    a = oq4.qwen_block(h, q4blk, attn, 1e-6)
    b = oracle.qwen_block(h, bfblk, attn, 1e-6)
    for k in ("q", "k", "v", "h_mid", "h"):
        assert np.allclose(a[k], b[k], rtol=1e-12, atol=1e-12), k
    assert np.array_equal(a["s"], b["s"])


# ---- the LayerNorm -> Linear -> GELU block's backward ("It works in training too")

from oracle import train as otr  # noqa: E402


def _bf16_round(v):
    return oracle.bf16_to_f64(oracle.f64_to_bf16(v))


def test_gelu_grad_is_the_derivative_of_gelu():
    t = np.linspace(-6, 6, 241)
    h = 1e-5
    fd = (oracle.gelu(t + h) - oracle.gelu(t - h)) / (2 * h)
    assert np.max(np.abs(otr.gelu_grad(t) - fd)) < 1e-8
    assert abs(otr.gelu_grad(np.array([0.0]))[0] - 0.5) < 1e-15


def test_exact_block_backward_matches_finite_differences():
    """L = sum(dz * z) of the exact block (no roundings): every gradient of
    the exact backward against central differences of L."""
    rng = np.random.default_rng(51)
    B, w = 2, 8
    x = rng.normal(size=(B, w))
    gamma, beta, b = rng.uniform(0.5, 1.5, w), rng.normal(0, 0.1, w), rng.normal(0, 0.1, w)
    W = rng.normal(0, 0.4, (w, w))
    dz = rng.normal(size=(B, w))
    g = otr.mlp_block_backward(x, gamma, beta, W, b, dz)

    def loss(x_, gamma_, beta_, W_, b_):
        return float((dz * otr.mlp_block_forward(x_, gamma_, beta_, W_, b_)["z"]).sum())
    args = [x, gamma, beta, W, b]
    names = ["dx", "dgamma", "dbeta", "dW", "db"]
    h = 1e-6
    for a, name in enumerate(names):
        fd = np.zeros_like(args[a])
        for idx in np.ndindex(args[a].shape):
            p = [v.copy() for v in args]
            m = [v.copy() for v in args]
            p[a][idx] += h
            m[a][idx] -= h
            fd[idx] = (loss(*p) - loss(*m)) / (2 * h)
        assert np.allclose(g[name], fd, rtol=1e-6, atol=1e-8), name


def test_layernorm_gradient_sums_to_zero_per_row():
    """LN(x + c) = LN(x): the exact input gradient has zero row sums."""
    rng = np.random.default_rng(52)
    x = rng.normal(size=(3, 16))
    w = 16
    g = otr.mlp_block_backward(x, rng.uniform(0.5, 1.5, w), rng.normal(0, 0.1, w),
                               rng.normal(0, 0.3, (w, w)), rng.normal(0, 0.1, w),
                               rng.normal(size=(3, w)))
    assert np.max(np.abs(g["dx"].sum(axis=1))) < 1e-12


def test_rounded_forward_is_the_bf16_block():
    """The backward's saved forward with bf16 roundings is the forward block
    of the C oracle bit for bit."""
    rng = np.random.default_rng(53)
    B, w = 4, 64
    xb = oracle.f64_to_bf16(rng.normal(size=(B, w)))
    blk = {"gamma": oracle.f64_to_bf16(rng.uniform(0.5, 1.5, w)),
           "beta": oracle.f64_to_bf16(rng.normal(0, 0.1, w)),
           "W": oracle.f64_to_bf16(rng.normal(0, 0.05, (w, w))),
           "b": oracle.f64_to_bf16(rng.normal(0, 0.1, w))}
    f = otr.mlp_block_forward(oracle.bf16_to_f64(xb), *(oracle.bf16_to_f64(blk[k])
                              for k in ("gamma", "beta", "W", "b")), rounding=_bf16_round)
    assert np.array_equal(oracle.f64_to_bf16(f["z"]), oracle.mlp_block(xb, blk))


def test_backward_prefetch_order_fetches_the_previous_block():
    assert otr.chain_prefetch_order(3, backward=False) == [(0, 1), (1, 2), (2, None)]
    assert otr.chain_prefetch_order(3, backward=True) == [(2, 1), (1, 0), (0, None)]


def test_chain_backward_matches_finite_differences_of_the_mean_square_loss():
    """Two exact blocks chained, loss mean(z^2) of the last output: every
    gradient of mlp_chain_backward against central differences of the loss
    (a dropped link between blocks, a wrong loss gradient or a swapped
    block order fails here)."""
    rng = np.random.default_rng(54)
    B, w, L = 2, 8, 2
    x = rng.normal(size=(B, w))
    blocks = [{"gamma": rng.uniform(0.5, 1.5, w), "beta": rng.normal(0, 0.1, w),
               "W": rng.normal(0, 0.4, (w, w)), "b": rng.normal(0, 0.1, w)} for _ in range(L)]
    res = otr.mlp_chain_backward(x, blocks)

    def loss(x_, blocks_):
        h = x_
        for blk in blocks_:
            h = otr.mlp_block_forward(h, blk["gamma"], blk["beta"], blk["W"], blk["b"])["z"]
        return float(np.mean(h * h))
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (loss(xp, blocks) - loss(xm, blocks)) / (2 * h)
    assert np.allclose(res["dx"], fd, rtol=1e-6, atol=1e-9)
    for i, name, key in ((0, "W", "dW"), (1, "gamma", "dgamma"), (0, "b", "db"), (1, "beta", "dbeta")):
        fd = np.zeros_like(blocks[i][name])
        for idx in np.ndindex(fd.shape):
            bp = [dict(b) for b in blocks]
            bm = [dict(b) for b in blocks]
            bp[i][name] = blocks[i][name].copy()
            bm[i][name] = blocks[i][name].copy()
            bp[i][name][idx] += h
            bm[i][name][idx] -= h
            fd[idx] = (loss(x, bp) - loss(x, bm)) / (2 * h)
        assert np.allclose(res["grads"][i][key], fd, rtol=1e-6, atol=1e-9), (i, key)


def test_mean_square_loss_grad_closed_form():
    z = np.array([[1.0, -2.0], [0.5, 0.0]])
    assert np.array_equal(otr.mean_square_loss_grad(z), np.array([[0.5, -1.0], [0.25, 0.0]]))


def test_forced_module_inputs_equal_to_its_own_change_nothing():
    """Teacher forcing plumbing: forcing each module input with the value the
    oracle computes itself reproduces the unforced gradients bit for bit,
    and forcing dlin changes exactly the gradients downstream of it."""
    rng = np.random.default_rng(55)
    B, w = 3, 16
    x = oracle.bf16_to_f64(oracle.f64_to_bf16(rng.normal(size=(B, w))))
    args = [_bf16_round(rng.uniform(0.5, 1.5, w)), _bf16_round(rng.normal(0, 0.1, w)),
            _bf16_round(rng.normal(0, 0.2, (w, w))), _bf16_round(rng.normal(0, 0.1, w))]
    dz = _bf16_round(rng.normal(size=(B, w)))
    g = otr.mlp_block_backward(x, *args, dz, rounding=_bf16_round)
    f = otr.mlp_block_forward(x, *args, rounding=_bf16_round)
    g2 = otr.mlp_block_backward(x, *args, dz, rounding=_bf16_round,
                                forced={"ln": f["ln"], "lin": f["lin"], "dlin": g["dlin"],
                                        "dln": g["dln"]})
    for k in ("dx", "dW", "db", "dgamma", "dbeta", "dlin", "dln"):
        assert np.array_equal(g[k], g2[k]), k
    g3 = otr.mlp_block_backward(x, *args, dz, rounding=_bf16_round,
                                forced={"dlin": np.zeros((B, w))})
    assert not np.any(g3["dW"]) and not np.any(g3["db"]) and not np.any(g3["dx"])
