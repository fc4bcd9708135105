"""GPU parity of the chain executor (one CUDA graph per step) against the
oracle: per-block teacher-forced checks through the h trace, end-to-end argmax
where the oracle's top-2 margin exceeds the tolerance, bit-identity between
graph/eager/PDL on/off and prefetch on/off/decoy, and the host-buffer step."""
import numpy as np
import pytest
import torch

import oracle
from weight_streaming_gemv_bf16_gb300 import binding as wb
from weight_streaming_gemv_bf16_gb300 import chain as wc
from weight_streaming_gemv_bf16_gb300 import synth
from _util import (assert_fp32, assert_mlp_block_close, bf16_bits_to_f64, dev_bf16, dev_f32,
                   host_bits, rel_err_rows)

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


SMALL = synth.QwenShape(hidden=256, kv_dim=64, inter=512, vocab=1000, layers=3)


def _host_weights(shape, seed):
    blocks = [synth.qwen_block_weights(shape, seed, l) for l in range(shape.layers)]
    head = synth.qwen_head_weights(shape, seed)
    return blocks, head


def _dev(ws):
    return {k: dev_bf16(v) for k, v in ws.items()}


def _make(shape, B, seed, **kw):
    blocks, head = _host_weights(shape, seed)
    attn = np.stack([synth.qwen_attn(shape, B, seed, l) for l in range(shape.layers)])
    h0 = synth.qwen_hidden(shape, B, seed)
    ch = wc.qwen_chain([_dev(b) for b in blocks], _dev(head), dev_bf16(attn), dev_f32(h0), **kw)
    return ch, blocks, head, attn, h0


def _margin_ok(logits):
    top2 = np.sort(logits, axis=1)[:, -2:]
    rms = np.sqrt(np.mean(logits * logits, axis=1))
    return (top2[:, 1] - top2[:, 0]) > 2 * 2e-3 * np.maximum(np.abs(top2[:, 1]), rms)


def _check_chain(ch, blocks, head, attn, h0, eps=1e-6):
    """Teacher-forced per-block parity on the h trace, q/k/v of every block,
    then the head on the GPU's final h, and the end-to-end oracle argmax."""
    L = len(blocks)
    trace = ch.h_trace.cpu().numpy().astype(np.float64)
    h_prev = h0.astype(np.float64)
    for l in range(L):
        ref = oracle.qwen_block(h_prev, blocks[l], bf16_bits_to_f64(attn[l]), eps, threads=8)
        assert_fp32(trace[l], ref["h"], what=f"block {l} h")
        if ch.qkv:
            for name, t in zip("qkv", ch.qkv[l]):
                assert_fp32(t.cpu().numpy(), ref[name], what=f"block {l} {name}")
        h_prev = trace[l]
    assert np.array_equal(ch.h_out.cpu().numpy(), trace[-1].astype(np.float32))
    logits = oracle.lmhead_logits(trace[-1], oracle.bf16_to_f64(head["gamma_f"]), head["Wlm"],
                                  eps, threads=8)
    got = ch.idx.cpu().numpy()
    ok = _margin_ok(logits)
    assert np.array_equal(got[ok], oracle.argmax_rows(logits)[ok])
    if ch.logits is not None:
        assert_fp32(ch.logits.cpu().numpy(), logits, what="logits")
    # end to end from h0 (no teacher forcing): the argmax where the margin allows
    full = oracle.qwen_chain(h0, blocks, [bf16_bits_to_f64(a) for a in attn], head["gamma_f"],
                             head["Wlm"], eps, threads=8)
    ok2 = _margin_ok(full["logits"])
    assert np.array_equal(got[ok2], full["idx"][ok2])
    # Without teacher forcing, rounding differences compound through the
    # blocks; the end-to-end drift is reported and only bounded against gross
    # errors (a wrong block would be off by O(1)).
    drift = rel_err_rows(trace[-1], full["h"])
    print(f"end-to-end final-h relative drift after {L} blocks: {drift:.3g}")
    assert drift < 0.05
    return int(ok2.sum())


SMALL_SPLIT = synth.QwenShape(hidden=256, kv_dim=64, inter=2048, vocab=1000, layers=2)
# gate/up and the LM head large enough (8 Mi weights) for the optional
# tensor-core kernel
MID = synth.QwenShape(hidden=512, kv_dim=128, inter=8192, vocab=16384, layers=2)


@pytest.mark.parametrize("persistent", [False, True])
@pytest.mark.parametrize("B,shape", [(1, SMALL), (3, SMALL), (8, SMALL), (12, SMALL), (16, SMALL),
                                     (1, SMALL_SPLIT), (4, SMALL_SPLIT), (16, SMALL_SPLIT),
                                     (5, MID), (12, MID), (16, MID)])
def test_small_chain_matches_oracle(B, shape, persistent):
    """SMALL_SPLIT's down projection (K = 2048 over 256 rows) is split in K."""
    ch, blocks, head, attn, h0 = _make(shape, B, 21, trace=True, keep_qkv=True, logits=True,
                                       persistent=persistent)
    # the persistent kernel takes batch <= 4; larger batches run op by op
    assert ch.chain.persistent == (persistent and B <= 4)
    ch.chain.capture()
    ch.run()
    ch.run()  # a second replay: barrier counters and tickets were reset
    torch.cuda.synchronize()
    _check_chain(ch, blocks, head, attn, h0)


def test_persistent_graph_and_launch_are_bit_identical():
    outs = []
    for graph in (True, False):
        ch, *_ = _make(SMALL, 2, 26, trace=True, logits=True, persistent=True)
        assert ch.chain.persistent
        if graph:
            ch.chain.capture()
            for _ in range(3):
                ch.run()
        else:
            ch.chain.run_eager()
        torch.cuda.synchronize()
        outs.append((ch.h_out.cpu(), ch.logits.cpu(), ch.idx.cpu(), ch.h_trace.cpu()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_graph_eager_and_pdl_are_bit_identical():
    B = 2
    outs = []
    for use_pdl, graph in ((True, True), (False, True), (True, False)):
        ch, *_ = _make(SMALL, B, 22, use_pdl=use_pdl, trace=True, logits=True)
        if graph:
            ch.chain.capture()
            for _ in range(3):
                ch.run()  # replays start again from h_in
        else:
            ch.chain.run_eager()
        torch.cuda.synchronize()
        outs.append((ch.h_out.cpu(), ch.logits.cpu(), ch.idx.cpu(), ch.h_trace.cpu()))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)


@pytest.mark.parametrize("B,shape", [(1, SMALL), (4, SMALL), (16, SMALL), (2, SMALL_SPLIT),
                                     (16, SMALL_SPLIT), (5, MID)])
def test_untraced_pdl_graph_matches_traced_build(B, shape):
    """The chain without trace copies (programmatic-dependent-launch edges at
    every op boundary, as timed) against the traced build of the same weights
    (whose blocks the oracle checks): final h, logits and argmax bit for bit,
    replay after replay, and the argmax against the oracle end to end."""
    blocks, head = _host_weights(shape, 27)
    attn = np.stack([synth.qwen_attn(shape, B, 27, l) for l in range(shape.layers)])
    h0 = synth.qwen_hidden(shape, B, 27)
    db, dh, da, dx = [_dev(b) for b in blocks], _dev(head), dev_bf16(attn), dev_f32(h0)
    traced = wc.qwen_chain(db, dh, da, dx, trace=True, logits=True)
    traced.chain.capture()
    traced.run()
    timed = wc.qwen_chain(db, dh, da, dx, use_pdl=True, logits=True)
    timed.chain.capture()
    for _ in range(3):
        timed.h_out.fill_(float("nan"))
        timed.run()
        torch.cuda.synchronize()
        assert torch.equal(timed.h_out.cpu(), traced.h_out.cpu())
        assert torch.equal(timed.logits.cpu(), traced.logits.cpu())
        assert torch.equal(timed.idx.cpu(), traced.idx.cpu())
    _oracle_end_to_end(timed.h_out.cpu().numpy(), timed.idx.cpu().numpy(),
                       timed.logits.cpu().numpy(), blocks, head, attn, h0, 1e-6)


def _set_tuning(**kw):
    base = wb.get_tuning()
    t = wb.Tuning()
    for f, _ in wb.Tuning._fields_:
        setattr(t, f, getattr(base, f))
    for k, v in kw.items():
        setattr(t, k, v)
    wb.set_tuning(t)
    return base


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16])
def test_form_kernels_match_general_kernel_bitwise(B):
    """The per-form kernels (each holding only its op's staging path and
    epilogue) compute exactly what the general kernel computes."""
    outs = []
    for forms in (0, 1):
        base = _set_tuning(forms=forms, mma=0)  # the CUDA-core forms
        try:
            ch, *_ = _make(SMALL, B, 24, trace=True, logits=True, keep_qkv=True)
            ch.chain.capture()
            ch.run()
            torch.cuda.synchronize()
            outs.append((ch.h_out.cpu(), ch.logits.cpu(), ch.idx.cpu(), ch.h_trace.cpu(),
                         *[t.cpu() for t in ch.qkv[-1]]))
        finally:
            wb.set_tuning(base)
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("mode,stride", [(1, 128), (2, 128), (3, 16384)])
def test_prefetch_and_decoy_leave_outputs_bit_identical(mode, stride):
    B = 1
    base, *_ = _make(SMALL, B, 23, logits=True)
    base.chain.capture()
    base.run()
    plan = wb.PrefetchPlan(8, 256, stride, mode)
    for decoy in (False, True):
        ch, *_ = _make(SMALL, B, 23, logits=True, prefetch=2, fixed_plan=plan, decoy=decoy)
        ch.chain.capture()
        ch.run()
        ch.run()
        torch.cuda.synchronize()
        assert torch.equal(ch.h_out.cpu(), base.h_out.cpu())
        assert torch.equal(ch.logits.cpu(), base.logits.cpu())
        assert torch.equal(ch.idx.cpu(), base.idx.cpu())


def test_tuner_measures_plans_and_keeps_bits():
    B = 1
    base, *_ = _make(SMALL, B, 24, logits=True)
    base.chain.capture()
    base.run()
    ch, *_ = _make(SMALL, B, 24, logits=True, prefetch=1, tune_pairs=8)
    ch.chain.tune()
    plans = ch.chain.plans()
    assert len(plans) == 4 * SMALL.layers + 1
    for (mode, blocks, threads, stride), lo, mean in plans:
        assert mode in (0, 1, 2, 3)
        assert np.isfinite(lo) and np.isfinite(mean)
        if mode:
            assert lo > 0.01  # kept only when the CI lower bound clears +1%
    ch.chain.capture()
    ch.run()
    torch.cuda.synchronize()
    assert torch.equal(ch.logits.cpu(), base.logits.cpu())


def test_step_host_matches_device_run():
    B = 4
    ch, blocks, head, attn, h0 = _make(SMALL, B, 25)
    ch.chain.capture()
    ch.run()
    torch.cuda.synchronize()
    ref_idx = ch.idx.cpu().numpy().copy()
    h_host = torch.from_numpy(h0).pin_memory()
    attn_host = torch.from_numpy(attn.view(np.int16)).pin_memory()
    out = torch.full((B,), -1, dtype=torch.int32).pin_memory()
    ch.h_out.fill_(float("nan"))
    ch.chain.step_host(h_host, attn_host, out)
    assert np.array_equal(out.numpy(), ref_idx)
    # the host-staged step against the oracle: argmax where the margin allows,
    # the final h it left on the device within the end-to-end drift bound
    _oracle_end_to_end(ch.h_out.cpu().numpy(), out.numpy(), None, blocks, head, attn, h0, 1e-6)
    # new inputs through the host path change the answer the same way a device run does
    h2 = (h0[::-1].copy())
    ch.chain.step_host(torch.from_numpy(h2).pin_memory(), attn_host, out)
    ch.h_in.copy_(torch.from_numpy(h2))
    ch.run()
    torch.cuda.synchronize()
    assert np.array_equal(out.numpy(), ch.idx.cpu().numpy())
    # the same host buffers with new contents (the step's graph reads them anew)
    h3 = synth.qwen_hidden(SMALL, B, 99)
    h_host.copy_(torch.from_numpy(h3))
    out.fill_(-1)
    ch.chain.step_host(h_host, attn_host, out)
    ch.h_in.copy_(torch.from_numpy(h3))
    ch.run()
    torch.cuda.synchronize()
    assert np.array_equal(out.numpy(), ch.idx.cpu().numpy())


@pytest.mark.parametrize("mma", [0, 1])
@pytest.mark.parametrize("B,shape", [(32, SMALL), (128, SMALL), (40, MID), (128, MID)])
def test_large_batch_chain_in_tiles_matches_oracle(B, shape, mma):
    """Batches past the kernels' 16-row tile ("One Token, Kernel by Kernel",
    "Batching: when does decode stop being memory-bound?"): every op runs
    once per 16-row tile (40 = two full tiles and one of 8); per-block
    teacher-forced parity, the end-to-end argmax, and the graph without trace
    copies equal to the traced one bit for bit."""
    base = _set_tuning(mma=mma)
    try:
        ch, blocks, head, attn, h0 = _make(shape, B, 28, trace=True, keep_qkv=True, logits=True)
        ch.chain.capture()
        ch.run()
        ch.run()
        plain = wc.qwen_chain([_dev(b) for b in blocks], _dev(head), dev_bf16(attn), dev_f32(h0),
                              logits=True)
        plain.chain.capture()
        plain.run()
        torch.cuda.synchronize()
    finally:
        wb.set_tuning(base)
    assert wb.device_error() == 0
    assert torch.equal(plain.h_out.cpu(), ch.h_out.cpu())
    assert torch.equal(plain.idx.cpu(), ch.idx.cpu())
    assert torch.equal(plain.logits.cpu(), ch.logits.cpu())
    _check_chain(ch, blocks, head, attn, h0)


@pytest.mark.parametrize("persistent", [False, True])
def test_one_full_size_block_matches_oracle(persistent):
    """One Qwen2.5-1.5B-shaped block at batch 1 (hidden 1536, KV 256, MLP 8960)."""
    shape = synth.QwenShape(layers=1)
    ch, blocks, head, attn, h0 = _make(shape, 1, 0, trace=True, keep_qkv=True,
                                       persistent=persistent)
    assert ch.chain.persistent == persistent
    ch.chain.capture()
    ch.run()
    torch.cuda.synchronize()
    ref = oracle.qwen_block(h0.astype(np.float64), blocks[0], bf16_bits_to_f64(attn[0]), 1e-6,
                            threads=8)
    for name, t in zip("qkv", ch.qkv[0]):
        assert_fp32(t.cpu().numpy(), ref[name], what=name)
    assert_fp32(ch.h_out.cpu().numpy(), ref["h"], what="h")


@pytest.mark.parametrize("B", [8, 16])
def test_one_full_size_block_tensor_cores_match_oracle(B):
    """One full-size block at batch 8 and 16 with the optional tensor-core
    kernel (gate/up, Wd with its K = 8960 split, the LM head and its
    argmax), against the oracle."""
    base = _set_tuning(mma=1)
    try:
        shape = synth.QwenShape(layers=1)
        ch, blocks, head, attn, h0 = _make(shape, B, 3, trace=True, keep_qkv=True, logits=True)
        ch.chain.capture()
        ch.run()
        ch.run()
        torch.cuda.synchronize()
    finally:
        wb.set_tuning(base)
    assert wb.device_error() == 0
    _check_chain(ch, blocks, head, attn, h0)


@pytest.mark.parametrize("B", [5, 12, 16])
def test_mid_chain_tensor_cores_match_oracle(B):
    """The optional tensor-core kernel on MID (gate/up and the LM head large
    enough for it), batch tiles 8 and 16 with padded batch rows."""
    base = _set_tuning(mma=1)
    try:
        ch, blocks, head, attn, h0 = _make(MID, B, 21, trace=True, keep_qkv=True, logits=True)
        ch.chain.capture()
        ch.run()
        torch.cuda.synchronize()
    finally:
        wb.set_tuning(base)
    _check_chain(ch, blocks, head, attn, h0)


@pytest.fixture(scope="module")
def full_chain():
    """The full-size chain's seeded inputs (Qwen2.5-1.5B shapes, batch 1, seed
    0: the weights the benchmark times), on the host and on the device."""
    sh = synth.QWEN2_5_1_5B
    blocks, head = _host_weights(sh, 0)
    attn = np.stack([synth.qwen_attn(sh, 1, 0, l) for l in range(sh.layers)])
    h0 = synth.qwen_hidden(sh, 1, 0)
    dev = ([_dev(b) for b in blocks], _dev(head), dev_bf16(attn), dev_f32(h0))
    return sh, blocks, head, attn, h0, dev


def _chain_on(full, **kw):
    sh, blocks, head, attn, h0, (dblocks, dhead, dattn, dh0) = full
    return wc.qwen_chain(dblocks, dhead, dattn, dh0, eps=sh.eps, **kw)


@pytest.mark.parametrize("persistent", [False, True])
def test_full_chain_28_blocks_matches_oracle(full_chain, persistent):
    """The full 28-block chain + final RMSNorm + LM head 151936 x 1536 + argmax,
    batch 1, one CUDA graph: per-block teacher forcing and the end-to-end argmax."""
    sh, blocks, head, attn, h0, _ = full_chain
    ch = _chain_on(full_chain, trace=True, logits=True, persistent=persistent)
    assert ch.chain.persistent == persistent
    ch.chain.capture()
    ch.run()
    ch.run()  # a replay computes the same step again from the same inputs
    torch.cuda.synchronize()
    assert wb.device_error() == 0
    eligible = _check_chain(ch, blocks, head, attn, h0)
    assert eligible == 1


def _oracle_end_to_end(h_gpu, idx_gpu, logits_gpu, blocks, head, attn, h0, eps):
    """The oracle's whole step from h0 against a GPU step's final h, argmax
    and (when given) logits: the logits of the oracle's LM head on the GPU's
    own final h within the fp32 bound, the argmax where the oracle's top-2
    margin exceeds the tolerance, and the final h within the end-to-end drift
    bound (bf16 rounding points compound over the blocks)."""
    full = oracle.qwen_chain(h0, blocks, [bf16_bits_to_f64(a) for a in attn], head["gamma_f"],
                             head["Wlm"], eps, threads=8)
    ok = _margin_ok(full["logits"])
    assert np.array_equal(idx_gpu[ok], full["idx"][ok])
    drift = rel_err_rows(h_gpu, full["h"])
    assert drift < 0.05, f"final h drift {drift:.3g}"
    own = oracle.lmhead_logits(np.asarray(h_gpu, np.float64), oracle.bf16_to_f64(head["gamma_f"]),
                               head["Wlm"], eps, threads=8)
    ok_own = _margin_ok(own)
    assert np.array_equal(idx_gpu[ok_own], oracle.argmax_rows(own)[ok_own])
    if logits_gpu is not None:
        e = assert_fp32(logits_gpu, own, what="logits of the timed graph")
        print(f"timed graph: logits max rel err {e:.3g}, final-h drift {drift:.3g}")
    return int(ok.sum())


@pytest.mark.parametrize("prefetch", ["tuned", "off"])
def test_timed_graph_matches_traced_build_and_oracle(full_chain, prefetch):
    """The graph the benchmark times -- no trace copies, so every op boundary
    (Wd -> next block's QKV and the last Wd -> LM head included) carries a
    programmatic-dependent-launch edge, and prefetch plans tuned or none --
    replayed several times.  Every replay's final h and argmax equal the
    traced build's bit for bit (the traced build's blocks are checked against
    the oracle one by one), and the step agrees with the oracle end to end.
    The same graph with the logits written gives the logits for the fp32
    check ("One Token, Kernel by Kernel", "The whole step")."""
    sh, blocks, head, attn, h0, _ = full_chain
    pf = 1 if prefetch == "tuned" else 0
    timed = _chain_on(full_chain, use_pdl=True, prefetch=pf, tune_pairs=30, min_gain=0.01)
    timed.chain.tune()
    timed.chain.capture()
    withlog = _chain_on(full_chain, use_pdl=True, prefetch=pf, logits=True, tune_pairs=30,
                        min_gain=0.01)
    withlog.chain.tune()
    withlog.chain.capture()
    traced = _chain_on(full_chain, trace=True, logits=True)
    traced.chain.capture()
    traced.run()
    torch.cuda.synchronize()
    ref_h, ref_idx = traced.h_out.cpu(), traced.idx.cpu()
    assert torch.equal(ref_h, traced.h_trace[-1].cpu())
    for rep in range(4):
        timed.h_out.fill_(float("nan"))
        timed.idx.fill_(-1)
        timed.run()
        withlog.run()
        torch.cuda.synchronize()
        assert torch.equal(timed.h_out.cpu(), ref_h), f"replay {rep}: final h differs"
        assert torch.equal(timed.idx.cpu(), ref_idx), f"replay {rep}: argmax differs"
        assert torch.equal(withlog.h_out.cpu(), ref_h)
        assert torch.equal(withlog.logits.cpu(), traced.logits.cpu())
    assert wb.device_error() == 0
    eligible = _oracle_end_to_end(timed.h_out.cpu().numpy(), timed.idx.cpu().numpy(),
                                  withlog.logits.cpu().numpy(), blocks, head, attn, h0, sh.eps)
    assert eligible == 1


def test_host_step_full_chain_matches_oracle(full_chain):
    """ws_chain_step_host on the benchmark's chain: h and the 28 attention
    inputs from pinned host buffers, the argmax back to a host buffer, all in
    one graph launch.  The host result equals the oracle's argmax, and the
    device-side final h it left behind agrees with the oracle end to end and
    with the device-input run bit for bit."""
    sh, blocks, head, attn, h0, _ = full_chain
    ch = _chain_on(full_chain, use_pdl=True, prefetch=1, tune_pairs=30, min_gain=0.01)
    ch.chain.tune()
    ch.chain.capture()
    ch.run()
    torch.cuda.synchronize()
    dev_h, dev_idx = ch.h_out.cpu(), ch.idx.cpu()
    h_host = torch.from_numpy(h0).pin_memory()
    a_host = torch.from_numpy(np.ascontiguousarray(attn).view(np.int16)).pin_memory()
    out = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    for _ in range(3):
        ch.h_out.fill_(float("nan"))
        out.fill_(-1)
        ch.chain.step_host(h_host, a_host, out)
        assert torch.equal(out, dev_idx)
        assert torch.equal(ch.h_out.cpu(), dev_h)
    assert wb.device_error() == 0
    _oracle_end_to_end(ch.h_out.cpu().numpy(), out.numpy(), None, blocks, head, attn, h0, sh.eps)


@pytest.mark.parametrize("B", [4, 16])
def test_mlp_chain_72_blocks(B):
    sh = synth.MlpShape()
    blocks = [synth.mlp_block_weights(sh, 0, i) for i in range(sh.blocks)]
    x = synth.mlp_input(sh, B, 0)
    dblocks = [_dev(b) for b in blocks]
    ch = wc.mlp_chain(dblocks, dev_bf16(x))
    ch.chain.capture()
    ch.run()
    # teacher-forced: the same kernel launched op by op, each op against the oracle
    cur = dev_bf16(x)
    ws = wb.new_workspace(wb.OP_GEMV, sh.width, sh.width, B)
    for i, (hb, db) in enumerate(zip(blocks, dblocks)):
        z = torch.empty_like(cur)
        wb.ln_gemv_gelu(cur, db["gamma"], db["beta"], db["W"], db["b"], z, sh.eps, workspace=ws)
        if i % 12 == 0 or i == sh.blocks - 1:
            assert_mlp_block_close(host_bits(z), host_bits(cur), hb, sh.eps, what=f"mlp block {i}")
        cur = z
    torch.cuda.synchronize()
    assert torch.equal(ch.y_out.cpu(), cur.cpu())
    # prefetch with a fixed plan and with a decoy: same bits
    for decoy in (False, True):
        pch = wc.mlp_chain(dblocks, dev_bf16(x), prefetch=2,
                           fixed_plan=wb.PrefetchPlan(8, 256, 128, 1), decoy=decoy)
        pch.chain.capture()
        pch.run()
        torch.cuda.synchronize()
        assert torch.equal(pch.y_out.cpu(), ch.y_out.cpu())


@pytest.mark.parametrize("B", [4, 16])
def test_mlp_step_host_matches_device_run(B):
    """The LayerNorm chain's host step: x from a pinned host buffer, the
    output back to one, one graph launch (the word copies chained to the
    first and last op), equal bit for bit to the device-input run."""
    sh = synth.MlpShape(blocks=12)
    blocks = [synth.mlp_block_weights(sh, 4, i) for i in range(sh.blocks)]
    x = synth.mlp_input(sh, B, 4)
    ch = wc.mlp_chain([_dev(b) for b in blocks], dev_bf16(x))
    ch.chain.capture()
    ch.run()
    torch.cuda.synchronize()
    ref = ch.y_out.cpu().clone()
    x_host = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
    out = torch.zeros((B, sh.width), dtype=torch.int16).pin_memory()
    for _ in range(3):
        out.fill_(0)
        ch.chain.step_host(x_host, None, out)
        assert torch.equal(out.view(torch.bfloat16), ref)
    x2 = synth.mlp_input(sh, B, 5)
    x_host.copy_(torch.from_numpy(np.ascontiguousarray(x2).view(np.int16)))
    ch.chain.step_host(x_host, None, out)
    ch.x_in.copy_(dev_bf16(x2))
    ch.run()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.bfloat16), ch.y_out.cpu())


@pytest.mark.parametrize("persistent,B", [(False, 4), (True, 4), (True, 1), (False, 16)])
def test_mlp_chain_72_blocks_trace(persistent, B):
    """Every block of the 72-block chain, teacher-forced on the chain's own
    trace: block i's oracle is fed the GPU's output of block i-1."""
    sh = synth.MlpShape()
    blocks = [synth.mlp_block_weights(sh, 1, i) for i in range(sh.blocks)]
    x = synth.mlp_input(sh, B, 1)
    ch = wc.mlp_chain([_dev(b) for b in blocks], dev_bf16(x), persistent=persistent, trace=True)
    assert ch.chain.persistent == persistent
    ch.chain.capture()
    ch.run()
    ch.run()
    torch.cuda.synchronize()
    tr = host_bits(ch.trace)
    prev = x
    for i, hb in enumerate(blocks):
        frac = assert_mlp_block_close(tr[i], prev, hb, sh.eps, what=f"mlp block {i}")
        assert frac >= 0.97
        prev = tr[i]
    assert np.array_equal(host_bits(ch.y_out), tr[-1])
