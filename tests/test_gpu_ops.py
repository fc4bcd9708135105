"""GPU parity of every single-op entry point against the CPU oracle, element by
element, through the C ABI.  Sizes span several row groups, K splits and a
ragged tail; the full-size shapes are checked on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from weight_streaming_gemv_bf16_gb300 import binding as wb
from weight_streaming_gemv_bf16_gb300 import synth
from _util import (assert_bf16_close, assert_fp32, assert_mlp_block_close, assert_ulp, dev_bf16,
                   dev_f32, dev_fp16, host_bits, tuning)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    assert wb.device_error(reset=True) == 0
    yield
    torch.cuda.synchronize()
    assert wb.device_error() == 0


def _ws(op, M, K, B):
    return wb.new_workspace(op, M, K, B)


def _inputs(M, K, B, seed, tag, xstd=1.0):
    W = synth.normal_bf16((M, K), 0.02, seed, tag + "/W")
    x = synth.normal_bf16((B, K), xstd, seed, tag + "/x")
    return W, x


# ------------------------------------------------------------------ gemv_bf16

@pytest.mark.parametrize("M,K,B,split", [
    (256, 256, 1, False), (37, 40, 3, True), (1000, 1536, 5, True), (2048, 1536, 2, False),
    (1536, 8960, 1, True), (256, 1536, 1, True), (256, 1536, 16, True), (1, 8, 1, True),
    (1536, 8960, 16, True), (513, 1536, 8, False), (768, 768, 4, True), (8960, 1536, 7, False),
])
def test_gemv_bf16_matches_oracle(M, K, B, split):
    W, x = _inputs(M, K, B, 1, f"gemv{M}x{K}x{B}")
    y = torch.full((B, M), float("nan"), device="cuda")
    ws = _ws(wb.OP_GEMV, M, K, B) if split else None
    wb.gemv_bf16(dev_bf16(W), dev_bf16(x), y, workspace=ws)
    ref = oracle.gemv(W, oracle.bf16_to_f64(x), threads=8)
    assert_fp32(y.cpu().numpy(), ref, what=f"gemv {M}x{K} B={B}")


def test_gemv_identity_and_one_hot_are_bit_exact():
    K = 1536
    x = synth.normal_bf16((4, K), 1.0, 2, "eye/x")
    eye = torch.eye(K, dtype=torch.bfloat16, device="cuda")
    y = torch.empty((4, K), device="cuda")
    wb.gemv_bf16(eye, dev_bf16(x), y)
    assert torch.equal(y.cpu(), torch.from_numpy(oracle.bf16_to_f64(x)).float())
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(3))
    P = torch.zeros((K, K), dtype=torch.bfloat16)
    P[torch.arange(K), perm] = 1.0
    wb.gemv_bf16(P.cuda(), dev_bf16(x), y)
    assert torch.equal(y.cpu(), torch.from_numpy(oracle.bf16_to_f64(x)).float()[:, perm])


def test_gemv_all_ones_exact():
    for K in (8, 1536, 8960):
        W = torch.ones((300, K), dtype=torch.bfloat16, device="cuda")
        x = torch.ones((2, K), dtype=torch.bfloat16, device="cuda")
        y = torch.empty((2, 300), device="cuda")
        wb.gemv_bf16(W, x, y)
        assert torch.all(y == K)


def test_split_k_is_deterministic_and_leaves_workspace_zeroed():
    M, K, B = 256, 1536, 3
    W, x = _inputs(M, K, B, 4, "det")
    ws = _ws(wb.OP_GEMV, M, K, B)
    assert ws is not None
    outs = []
    for _ in range(5):
        y = torch.empty((B, M), device="cuda")
        wb.gemv_bf16(dev_bf16(W), dev_bf16(x), y, workspace=ws)
        outs.append(y)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    sc = wb.gemv_plan(M, K, B)
    assert sc["S"] > 1
    tickets = ws[: sc["RG"] * 4]
    assert int(tickets.count_nonzero()) == 0


def test_large_gemv_sampled_rows():
    """The LM-head-sized GEMV at B = 1..16, checked on 2048 sampled rows."""
    M, K = 151936, 1536
    W = synth.normal_bf16((M, K), 0.02, 5, "big/W")
    Wd = dev_bf16(W)
    rows = np.sort(np.random.default_rng(5).choice(M, 2048, replace=False))
    for B in (1, 2, 4, 8, 16):
        x = synth.normal_bf16((B, K), 1.0, 5, f"big/x{B}")
        y = torch.empty((B, M), device="cuda")
        wb.gemv_bf16(Wd, dev_bf16(x), y)
        ref = oracle.gemv(W[rows], oracle.bf16_to_f64(x), threads=8)
        got = y.cpu().numpy()[:, rows]
        assert_fp32(got, ref, what=f"151936x1536 B={B}")


# ------------------------------------------------------------------ fused ops

def test_rmsnorm_gemv_fused_config():
    """x bf16[1,256] ~ N(0,1), gamma ~ U(0.5,1.5), W[256,256] ~ N(0,0.02), eps 1e-6."""
    x = synth.normal_bf16((1, 256), 1.0, 0, "cfg1/x")
    g = synth.uniform_bf16((256,), 0.5, 1.5, 0, "cfg1/gamma")
    W = synth.normal_bf16((256, 256), 0.02, 0, "cfg1/W")
    y = torch.empty((1, 256), device="cuda")
    wb.rmsnorm_gemv(dev_bf16(x), dev_bf16(g), dev_bf16(W), y, 1e-6)
    ref = oracle.rmsnorm_gemv(oracle.bf16_to_f64(x), oracle.bf16_to_f64(g), W, 1e-6)
    assert_fp32(y.cpu().numpy(), ref, what="rmsnorm_gemv 256")


@pytest.mark.parametrize("B,xdt", [(1, "f32"), (3, "bf16"), (16, "f32")])
def test_rmsnorm_gemv_wider(B, xdt):
    M, K = 1000, 1536
    W = synth.normal_bf16((M, K), 0.02, 6, "rg/W")
    g = synth.uniform_bf16((K,), 0.5, 1.5, 6, "rg/g")
    if xdt == "f32":
        xh = synth.normal_f32((B, K), 1.0, 6, "rg/x") * 3
        xd, xo = dev_f32(xh), xh.astype(np.float64)
    else:
        xb = synth.normal_bf16((B, K), 1.0, 6, "rg/x")
        xd, xo = dev_bf16(xb), oracle.bf16_to_f64(xb)
    y = torch.empty((B, M), device="cuda")
    wb.rmsnorm_gemv(xd, dev_bf16(g), dev_bf16(W), y, 1e-6, workspace=_ws(wb.OP_GEMV, M, K, B))
    ref = oracle.rmsnorm_gemv(xo, oracle.bf16_to_f64(g), W, 1e-6)
    assert_fp32(y.cpu().numpy(), ref, what=f"rmsnorm_gemv B={B}")


@pytest.mark.parametrize("B", [1, 2, 16])
def test_qkv_gemv(B):
    H, KV = 1536, 256
    sh = synth.QwenShape()
    blk = synth.qwen_block_weights(sh, 7, 0)
    h = synth.qwen_hidden(sh, B, 7)
    q = torch.empty((B, H), device="cuda")
    k = torch.empty((B, KV), device="cuda")
    v = torch.empty((B, KV), device="cuda")
    wb.qkv_gemv(dev_f32(h), dev_bf16(blk["gamma1"]), dev_bf16(blk["Wq"]), dev_bf16(blk["Wk"]),
                dev_bf16(blk["Wv"]), q, k, v, 1e-6, workspace=_ws(wb.OP_QKV_GEMV, H + 2 * KV, H, B))
    a = oracle.round_bf16(oracle.rmsnorm(h.astype(np.float64), oracle.bf16_to_f64(blk["gamma1"]), 1e-6))
    for name, t in (("Wq", q), ("Wk", k), ("Wv", v)):
        assert_fp32(t.cpu().numpy(), oracle.gemv(blk[name], a, 8), what=f"qkv {name} B={B}")


@pytest.mark.parametrize("B,norm", [(1, True), (4, True), (16, True), (2, False)])
def test_swiglu_gemv(B, norm):
    M, K = 8960, 1536
    Wg = synth.normal_bf16((M, K), 0.02, 8, "sw/Wg")
    Wu = synth.normal_bf16((M, K), 0.02, 8, "sw/Wu")
    g = synth.uniform_bf16((K,), 0.5, 1.5, 8, "sw/g")
    s = torch.empty((B, M), dtype=torch.bfloat16, device="cuda")
    if norm:
        xh = synth.normal_f32((B, K), 1.0, 8, "sw/x")
        wb.swiglu_gemv(dev_f32(xh), dev_bf16(g), dev_bf16(Wg), dev_bf16(Wu), s, 1e-6,
                       workspace=_ws(wb.OP_SWIGLU_GEMV, M, K, B))
        ref = oracle.swiglu_gemv(xh.astype(np.float64), oracle.bf16_to_f64(g), Wg, Wu, 1e-6, 8,
                                 exact=True)
    else:
        xb = synth.normal_bf16((B, K), 1.0, 8, "sw/x")
        wb.swiglu_gemv(dev_bf16(xb), None, dev_bf16(Wg), dev_bf16(Wu), s, 1e-6)
        ref = oracle.swiglu_gemv(oracle.bf16_to_f64(xb), None, Wg, Wu, 1e-6, 8, exact=True)
    assert_bf16_close(host_bits(s), ref, what=f"swiglu B={B}")


@pytest.mark.parametrize("B,in_place", [(1, True), (3, False), (16, True)])
def test_gemv_residual(B, in_place):
    M, K = 1536, 8960
    W, x = _inputs(M, K, B, 9, "res")
    h0 = synth.normal_f32((B, M), 1.0, 9, "res/h")
    h_out = dev_f32(h0)
    h_in = None if in_place else dev_f32(h0)
    if not in_place:
        h_out.fill_(float("nan"))
    wb.gemv_residual(dev_bf16(W), dev_bf16(x), h_out, h_in=h_in,
                     workspace=_ws(wb.OP_GEMV, M, K, B))
    ref = h0.astype(np.float64) + oracle.gemv(W, oracle.bf16_to_f64(x), 8)
    assert_fp32(h_out.cpu().numpy(), ref, what=f"residual B={B}")


@pytest.mark.parametrize("B", [4, 16])
def test_ln_gemv_gelu(B):
    sh = synth.MlpShape()
    blk = synth.mlp_block_weights(sh, 10, 0)
    x = synth.mlp_input(sh, B, 10)
    z = torch.empty((B, sh.width), dtype=torch.bfloat16, device="cuda")
    wb.ln_gemv_gelu(dev_bf16(x), dev_bf16(blk["gamma"]), dev_bf16(blk["beta"]), dev_bf16(blk["W"]),
                    dev_bf16(blk["b"]), z, 1e-5, workspace=_ws(wb.OP_GEMV, sh.width, sh.width, B))
    assert_mlp_block_close(host_bits(z), x, blk, 1e-5, what=f"ln_gemv_gelu B={B}")


@pytest.mark.parametrize("B,K", [(16, 1536), (16, 1544), (13, 1536), (9, 2048), (8, 2048),
                                 (8, 2056), (5, 3072), (4, 1536), (3, 1536)])
def test_rmsnorm_staging_by_rows_and_cta_wide(B, K):
    """The RMSNorm-fused GEMV on fp32 activations on both sides of the widths
    the row-wise staging takes (from batch tile 8 at most 6 chunks of 8
    columns a lane at tile 16 and 8 at tile 8; the fp32-output form at tile
    4), ragged batches inside the tile included; one-round CTA-wide staging
    past them (9 x 2048, 5 x 3072) and the two-pass general kernel past
    that (16 x 1544, 8 x 2056): all against the oracle."""
    M = 700
    W = synth.normal_bf16((M, K), 0.02, K + B, "rs/W")
    g = synth.uniform_bf16((K,), 0.5, 1.5, K + B, "rs/g")
    xh = synth.normal_f32((B, K), 1.0, K + B, "rs/x") * 3
    y = torch.empty((B, M), device="cuda")
    wb.rmsnorm_gemv(dev_f32(xh), dev_bf16(g), dev_bf16(W), y, 1e-6,
                    workspace=_ws(wb.OP_GEMV, M, K, B))
    ref = oracle.rmsnorm_gemv(xh.astype(np.float64), oracle.bf16_to_f64(g), W, 1e-6)
    assert_fp32(y.cpu().numpy(), ref, what=f"rmsnorm_gemv B={B} K={K}")


@pytest.mark.parametrize("B,K,split", [(16, 768, 0), (13, 768, 0), (5, 768, 0), (16, 1536, 0),
                                       (16, 1536, 2), (9, 2048, 0), (8, 2048, 0), (4, 768, 0),
                                       (3, 768, 0), (4, 2048, 0), (2, 768, 0), (1, 768, 0)])
def test_layernorm_staging_by_rows_and_cta_wide(B, K, split):
    """The LayerNorm + GEMV + bias + GELU block by rows (768 and 1536 wide at
    batch tile 16, ragged batches, 2048 at tile 8, 768 and 2048 at tile 4 with
    warps 0-3 staging a row each), by rows with a forced K split (each CTA
    staging its half of the columns), and CTA-wide past the row limit
    (9 x 2048) and below tile 4 (batch 2 and 1), against the oracle."""
    sh = synth.MlpShape(width=K)
    blk = synth.mlp_block_weights(sh, 12, 0)
    x = synth.mlp_input(sh, B, 12)
    z = torch.empty((B, K), dtype=torch.bfloat16, device="cuda")
    with tuning(force_ksplit=split):
        wb.ln_gemv_gelu(dev_bf16(x), dev_bf16(blk["gamma"]), dev_bf16(blk["beta"]),
                        dev_bf16(blk["W"]), dev_bf16(blk["b"]), z, 1e-5,
                        workspace=_ws(wb.OP_GEMV, K, K, B))
        torch.cuda.synchronize()
    assert_mlp_block_close(host_bits(z), x, blk, 1e-5, what=f"ln_gemv_gelu B={B} K={K} S={split}")


def _margin_ok(logits):
    top2 = np.sort(logits, axis=1)[:, -2:]
    rms = np.sqrt(np.mean(logits * logits, axis=1))
    return (top2[:, 1] - top2[:, 0]) > 2 * 2e-3 * np.maximum(np.abs(top2[:, 1]), rms)


@pytest.mark.parametrize("B,logits_out", [(1, True), (4, False), (16, True)])
def test_lmhead_argmax_sampled(B, logits_out):
    V, K = 151936, 1536
    W = synth.normal_bf16((V, K), 0.02, 11, "lm/W")
    g = synth.uniform_bf16((K,), 0.5, 1.5, 11, "lm/g")
    h = synth.normal_f32((B, K), 1.0, 11, "lm/h")
    idx = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    logits = torch.empty((B, V), device="cuda") if logits_out else None
    ws = _ws(wb.OP_LMHEAD_ARGMAX, V, K, B)
    wb.lmhead_argmax(dev_f32(h), dev_bf16(g), dev_bf16(W), idx, 1e-6, ws, logits=logits)
    full = oracle.lmhead_logits(h.astype(np.float64), oracle.bf16_to_f64(g), W, 1e-6, threads=8)
    ref_idx = oracle.argmax_rows(full)
    ok = _margin_ok(full)
    got = idx.cpu().numpy()
    assert ok.sum() >= 1
    assert np.array_equal(got[ok], ref_idx[ok])
    if logits_out:
        assert_fp32(logits.cpu().numpy(), full, what="lm logits")
        # the fused argmax equals the argmax of the kernel's own logits
        assert np.array_equal(got, np.argmax(logits.cpu().numpy(), axis=1))


def test_lmhead_argmax_planted_ties():
    """Identity-like head: logits are the normalised h, with planted ties."""
    K, V, B = 64, 64, 2
    W = torch.eye(K, dtype=torch.bfloat16)
    h = np.zeros((B, K), np.float32)
    h[0, [5, 9, 40]] = 3.0          # tie of three -> lowest index
    h[1, :] = -1.0
    h[1, 63] = 0.5                  # unique max at the end
    idx = torch.empty((B,), dtype=torch.int32, device="cuda")
    g = torch.ones(K, dtype=torch.bfloat16, device="cuda")
    ws = _ws(wb.OP_LMHEAD_ARGMAX, V, K, B)
    wb.lmhead_argmax(dev_f32(h), g, W.cuda(), idx, 1e-6, ws)
    assert idx.cpu().tolist() == [5, 63]


@pytest.mark.parametrize("rows,cols", [(1, 151936), (16, 151936), (3, 1000), (2, 1)])
def test_argmax_rows(rows, cols):
    v = np.random.default_rng(12).standard_normal((rows, cols)).astype(np.float32)
    if cols > 10:
        v[0, 7] = v[0, cols - 1] = 50.0   # tie: lowest index wins
    idx = torch.empty((rows,), dtype=torch.int32, device="cuda")
    ws = _ws(wb.OP_ARGMAX_ROWS, rows, cols, 1)
    for _ in range(2):  # twice: the tickets must have been reset
        wb.argmax_rows(dev_f32(v), idx, ws)
        assert np.array_equal(idx.cpu().numpy(), oracle.argmax_rows(v.astype(np.float64)))


@pytest.mark.parametrize("R,dtype", [(1, "fp16"), (128, "fp16"), (4096, "fp16"), (33, "bf16")])
def test_rmsnorm_rows(R, dtype):
    N = 896
    if dtype == "fp16":
        x = synth.normal_fp16((R, N), 1.0, 13, "rn/x")
        g = synth.uniform_fp16((N,), 0.5, 1.5, 13, "rn/g")
        xd, gd = dev_fp16(x), dev_fp16(g)
    else:
        x = synth.normal_bf16((R, N), 1.0, 13, "rn/x")
        g = synth.uniform_bf16((N,), 0.5, 1.5, 13, "rn/g")
        xd, gd = dev_bf16(x), dev_bf16(g)
    y = torch.empty_like(xd)
    wb.rmsnorm(xd, gd, y, 1e-6)
    assert_ulp(host_bits(y), oracle.rmsnorm_rows(x, g, 1e-6, dtype), what=f"rmsnorm {dtype} R={R}")


# ------------------------------------------------------------------ prefetch, probes, waits

def test_l2_prefetch_leaves_memory_untouched():
    buf = torch.randint(0, 2 ** 15, (1 << 22,), dtype=torch.int16, device="cuda")
    before = buf.clone()
    for mode, stride in ((1, 128), (2, 128), (3, 16384)):
        wb.l2_prefetch(buf, buf.numel() * 2, wb.PrefetchPlan(8, 256, stride, mode))
        wb.l2_prefetch(buf.data_ptr() + 4096, buf.numel() * 2 - 4096 - 48,
                       wb.PrefetchPlan(3, 128, stride, mode))
    torch.cuda.synchronize()
    assert torch.equal(buf, before)


def test_probes_run():
    buf = torch.ones(1 << 20, dtype=torch.int32, device="cuda")
    sink = torch.zeros(64, dtype=torch.int32, device="cuda")
    wb.read_probe(buf, buf.numel() * 4, 64, sink)
    wb.empty_probe(0)
    wb.empty_probe(1, buf, sink)
    torch.cuda.synchronize()
    assert int(sink[0]) == 1


def test_bounded_wait_times_out_and_reports():
    assert wb.device_error(reset=True) == 0
    wb.test_bounded_wait(50_000_000)  # 50 ms
    assert wb.device_error(reset=True) == 1
    assert wb.device_error() == 0
    # the context is still usable
    y = torch.empty((1, 8), device="cuda")
    wb.gemv_bf16(torch.ones((8, 8), dtype=torch.bfloat16, device="cuda"),
                 torch.ones((1, 8), dtype=torch.bfloat16, device="cuda"), y)
    assert torch.all(y.cpu() == 8)
