"""GPU parity of the 4-bit group-128 weight path ("One Token, Kernel by
Kernel", "4-bit weights") against the oracle: the quantiser bit for bit (its
decisions in fp32 on both sides), the GEMV over the packed rows within the
fp32 bound (double oracle on the same bytes), the decode chain on 4-bit
weights block by block (teacher-forced on the GPU's h trace) and its argmax."""
import numpy as np
import pytest
import torch

import oracle
from oracle import q4 as oq4
from weight_streaming_gemv_bf16_gb300 import binding as wb
from weight_streaming_gemv_bf16_gb300 import chain as wc
from weight_streaming_gemv_bf16_gb300 import synth
from _util import assert_fp32, dev_bf16, dev_f32, host_bits, tuning

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


def _quantize_both(W_bits):
    """(GPU packed rows, oracle packed rows); asserts they are the same bytes."""
    M, K = W_bits.shape
    Wq = torch.zeros((M, wb.q4_row_bytes(K)), dtype=torch.uint8, device="cuda")
    wb.quantize_q4(dev_bf16(W_bits), Wq)
    torch.cuda.synchronize()
    ref = oq4.pack(*oq4.quantize(W_bits))
    got = Wq.cpu().numpy()
    assert got.shape == ref.shape
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:4].tolist()}"
    return Wq, ref


@pytest.mark.parametrize("M,K", [(37, 640), (64, 1536), (9, 8960), (5, 1408), (3, 128)])
def test_quantizer_matches_oracle_bitwise(M, K):
    W = synth.normal_bf16((M, K), 0.02, M * 7 + K, "q4/W")
    W[0, :128] = W[0, 0]  # a constant group: scale 0
    _quantize_both(W)


def _with_forms(forms):
    base = wb.get_tuning()
    t = wb.Tuning()
    for f, _ in wb.Tuning._fields_:
        setattr(t, f, getattr(base, f))
    t.forms = forms
    wb.set_tuning(t)
    return base


@pytest.mark.parametrize("kernel", ["mma", "cuda_cores"])
@pytest.mark.parametrize("M,K,B", [(37, 640, 1), (37, 640, 3), (300, 1408, 2), (2048, 1536, 1),
                                   (1536, 8960, 1), (1536, 8960, 4), (8960, 1536, 1),
                                   (5, 128, 4), (151936 // 8, 1536, 2)])
def test_gemv_q4_matches_oracle(M, K, B, kernel):
    """Both 4-bit kernels: the tensor-core one (chain forms) and the CUDA-core
    one (taken with the chain forms switched off)."""
    W = synth.normal_bf16((M, K), 0.02, M + K + B, "q4/W")
    Wq, ref = _quantize_both(W)
    x = synth.normal_bf16((B, K), 1.0, M + K + B, "q4/x")
    y = torch.full((B, M), float("nan"), device="cuda")
    base = _with_forms(1 if kernel == "mma" else 0)
    try:
        wb.gemv_q4(Wq, dev_bf16(x), y, K)
        torch.cuda.synchronize()
    finally:
        wb.set_tuning(base)
    assert_fp32(y.cpu().numpy(), oq4.gemv(ref, K, oracle.bf16_to_f64(x)), what=f"{M}x{K} B={B}")


SMALL = synth.QwenShape(hidden=256, kv_dim=64, inter=512, vocab=1000, layers=3)
MID = synth.QwenShape(hidden=512, kv_dim=128, inter=1408, vocab=4096, layers=2)


@pytest.mark.parametrize("B,shape", [(1, SMALL), (2, SMALL), (4, SMALL), (1, MID), (3, MID)])
def test_q4_chain_matches_oracle(B, shape):
    _q4_chain_check(B, shape)


def _q4_chain_check(B, shape):
    seed = 11 * B + shape.hidden
    blocks = [synth.qwen_block_weights(shape, seed, l) for l in range(shape.layers)]
    head = synth.qwen_head_weights(shape, seed)
    attn = np.stack([synth.qwen_attn(shape, B, seed, l) for l in range(shape.layers)])
    h0 = synth.qwen_hidden(shape, B, seed)
    mats = ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")
    dblocks, rblocks = [], []
    for blk in blocks:
        d = {n: dev_bf16(blk[n]) for n in ("gamma1", "gamma2")}
        r = {n: blk[n] for n in ("gamma1", "gamma2")}
        for n in mats:
            d[n], r[n] = _quantize_both(blk[n])
        r["K"], r["KI"] = shape.hidden, shape.inter
        dblocks.append(d)
        rblocks.append(r)
    Wlm, Wlm_ref = _quantize_both(head["Wlm"])
    dhead = {"gamma_f": dev_bf16(head["gamma_f"]), "Wlm": Wlm}
    ch = wc.qwen_chain(dblocks, dhead, dev_bf16(attn), dev_f32(h0), eps=shape.eps, trace=True,
                       logits=True, q4=True)
    ch.chain.capture()
    ch.run()
    torch.cuda.synchronize()
    trace = ch.h_trace.cpu().numpy().astype(np.float64)
    h = h0.astype(np.float64)
    for l in range(shape.layers):
        out = oq4.qwen_block(h, rblocks[l], oracle.bf16_to_f64(attn[l]), shape.eps)
        assert_fp32(trace[l], out["h"], what=f"block {l}")
        h = trace[l]
    logits = oq4.lmhead_logits(h, head["gamma_f"], Wlm_ref, shape.hidden, shape.eps)
    assert_fp32(ch.logits.cpu().numpy(), logits, what="logits")
    idx = ch.idx.cpu().numpy()
    top2 = np.sort(logits, axis=1)[:, -2:]
    rms = np.sqrt(np.mean(logits * logits, axis=1))
    clear = (top2[:, 1] - top2[:, 0]) > 2 * 2e-3 * np.maximum(np.abs(top2[:, 1]), rms)
    ref_idx = oracle.argmax_rows(logits)
    assert np.array_equal(idx[clear], ref_idx[clear])


@pytest.mark.parametrize("M,K,B", [(40000, 640, 1), (40000, 640, 3), (39000, 1408, 4)])
def test_gemv_q4_tensor_core_kernel(M, K, B):
    """Shapes with at least two 16-row tasks per warp take the tensor-core
    4-bit kernel; every output against the oracle on a sample of rows (every
    seventh, and the last 40: the ragged final task)."""
    W = synth.normal_bf16((M, K), 0.02, M + K + B, "q4/Wbig")
    Wq = torch.zeros((M, wb.q4_row_bytes(K)), dtype=torch.uint8, device="cuda")
    wb.quantize_q4(dev_bf16(W), Wq)
    rows = np.unique(np.concatenate([np.arange(0, M, 7), np.arange(M - 40, M)]))
    codes, s, z = oq4.quantize(W[rows])
    ref = oq4.pack(codes, s, z)
    assert np.array_equal(Wq.cpu().numpy()[rows], ref)
    x = synth.normal_bf16((B, K), 1.0, M + B, "q4/xbig")
    y = torch.full((B, M), float("nan"), device="cuda")
    with tuning(q4_mma=2):  # batch 1 too
        wb.gemv_q4(Wq, dev_bf16(x), y, K)
        torch.cuda.synchronize()
    assert_fp32(y.cpu().numpy()[:, rows], oq4.gemv(ref, K, oracle.bf16_to_f64(x)),
                what=f"{M}x{K} B={B}")


@pytest.mark.parametrize("B", [1, 4])
def test_q4_chain_with_a_tensor_core_lm_head(B):
    """A vocabulary of 40000 rows puts the LM head (RMSNorm, argmax) on the
    tensor-core 4-bit kernel (at batch 1 only when asked for)."""
    shape = synth.QwenShape(hidden=256, kv_dim=64, inter=512, vocab=40000, layers=1)
    with tuning(q4_mma=2):
        _q4_chain_check(B, shape)


@pytest.mark.parametrize("cps", [1, 2, 3])
@pytest.mark.parametrize("B", [1, 4])
def test_q4_chain_at_every_residency(B, cps):
    """The CUDA-core 4-bit plans for one, two and three CTAs per SM (rings
    and grids sized for each; a vocabulary of 40000 on CUDA cores too) all
    match the oracle."""
    shape = synth.QwenShape(hidden=256, kv_dim=64, inter=1408, vocab=40000, layers=2)
    with tuning(ctas_per_sm=cps, q4_mma=0):
        _q4_chain_check(B, shape)


@pytest.mark.parametrize("B", [1, 4])
def test_q4_full_size_block_and_vocabulary(B):
    """One Qwen2.5-1.5B-sized block and the full 151936-row LM head on 4-bit
    weights, as the decode step runs them (batch 1: the CUDA-core kernel at
    two CTAs per SM, 304 CTAs, the head included; batch 4: one CTA per SM and
    the tensor-core head).  The block against the oracle; the head's packed
    rows and logits on sampled rows (every 97th and the last 40) against the
    oracle on the GPU's final h; the fused argmax over all rows equal to the
    first maximum of the GPU's own logits."""
    shape = synth.QwenShape(layers=1)
    seed = 101 + B
    blk = synth.qwen_block_weights(shape, seed, 0)
    head = synth.qwen_head_weights(shape, seed)
    attn = synth.qwen_attn(shape, B, seed, 0)[None]
    h0 = synth.qwen_hidden(shape, B, seed)
    d = {n: dev_bf16(blk[n]) for n in ("gamma1", "gamma2")}
    r = {n: blk[n] for n in ("gamma1", "gamma2")}
    for n in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd"):
        d[n], r[n] = _quantize_both(blk[n])
    r["K"], r["KI"] = shape.hidden, shape.inter
    V, H = shape.vocab, shape.hidden
    Wlm = torch.zeros((V, wb.q4_row_bytes(H)), dtype=torch.uint8, device="cuda")
    wb.quantize_q4(dev_bf16(head["Wlm"]), Wlm)
    rows = np.unique(np.concatenate([np.arange(0, V, 97), np.arange(V - 40, V)]))
    ref_rows = oq4.pack(*oq4.quantize(head["Wlm"][rows]))
    assert np.array_equal(Wlm.cpu().numpy()[rows], ref_rows)
    ch = wc.qwen_chain([d], {"gamma_f": dev_bf16(head["gamma_f"]), "Wlm": Wlm}, dev_bf16(attn),
                       dev_f32(h0), eps=shape.eps, trace=True, logits=True, q4=True)
    ch.chain.capture()
    ch.run()
    torch.cuda.synchronize()
    trace = ch.h_trace.cpu().numpy().astype(np.float64)
    ref = oq4.qwen_block(h0.astype(np.float64), r, oracle.bf16_to_f64(attn[0]), shape.eps)
    assert_fp32(trace[0], ref["h"], what="full-size 4-bit block")
    logits = ch.logits.cpu().numpy()
    ref_logits = oq4.lmhead_logits(trace[0], head["gamma_f"], ref_rows, H, shape.eps)
    assert_fp32(logits[:, rows], ref_logits, what="4-bit LM head, sampled rows")
    assert np.array_equal(ch.idx.cpu().numpy(), np.argmax(logits, axis=1))


def test_stamp_rows_cover_two_ctas_per_sm():
    """Per-CTA diagnostics of a chain whose ops run more CTAs than SMs (4-bit
    rows at batch 1: two CTAs per SM): the stamp buffer's CTA dimension is the
    widest op's grid, every CTA of every op writes its own row and no row
    past an op's grid, and a buffer one row short is refused."""
    shape = synth.QwenShape(hidden=512, kv_dim=128, inter=1408, vocab=40000, layers=2)
    blocks = [synth.qwen_block_weights(shape, 3, l) for l in range(shape.layers)]
    head = synth.qwen_head_weights(shape, 3)
    mats = ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")
    dblocks = []
    for blk in blocks:
        d = {n: dev_bf16(blk[n]) for n in ("gamma1", "gamma2")}
        for n in mats:
            d[n], _ = _quantize_both(blk[n])
        dblocks.append(d)
    Wlm, _ = _quantize_both(head["Wlm"])
    attn = np.stack([synth.qwen_attn(shape, 1, 3, l) for l in range(shape.layers)])
    h0 = synth.qwen_hidden(shape, 1, 3)
    ch = wc.qwen_chain(dblocks, {"gamma_f": dev_bf16(head["gamma_f"]), "Wlm": Wlm},
                       dev_bf16(attn), dev_f32(h0), eps=shape.eps, q4=True)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    g, nops = ch.chain.grid(), ch.chain.n_ops
    assert g == 2 * nsm  # the widest op: two CTAs per SM
    short = torch.zeros((g - 1, nops, 44), dtype=torch.int64, device="cuda")
    with pytest.raises(wb.WsError):
        ch.chain.debug_stamps(short)
    buf = torch.zeros((g, nops, 44), dtype=torch.int64, device="cuda")
    ch.chain.debug_stamps(buf)
    ch.chain.capture()
    ch.run()
    torch.cuda.synchronize()
    written = (buf[:, :, 0] > 0).cpu().numpy()  # [cta, op]
    per_op = written.sum(axis=0)
    # every op's CTAs are a prefix of the rows: rows past its grid untouched
    for f in range(nops):
        n = int(per_op[f])
        assert n > 0 and written[:n, f].all() and not written[n:, f].any(), (f, n)
    assert per_op.max() == g
    ch.chain.debug_stamps(None)
