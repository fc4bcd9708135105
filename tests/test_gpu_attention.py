"""GPU parity of the decode-attention entry point against the oracle's double
attention: the key-value append (bit-exact cache contents), the fp32 output
(within 2e-3 of the row's rms, the FP64-reference error bar of the split-KV
kernel of "One Token, Kernel by Kernel"), the bf16 output (the kernel's own
fp32 result rounded to nearest even), cache lengths on and around the
128-slot chunk boundary up to the full cache, every supported group size,
ragged positions across the batch, graph replay with advancing positions, and
an out-of-range position turned into the device error flag, and stale
non-finite values in the cache past the new token (never read)."""
import numpy as np
import pytest
import torch

import oracle
from weight_streaming_gemv_bf16_gb300 import binding as wb
from weight_streaming_gemv_bf16_gb300 import synth
from _util import assert_fp32, dev_bf16, dev_f32, host_bits

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    assert wb.device_error(reset=True) == 0
    yield
    torch.cuda.synchronize()
    assert wb.device_error() == 0


def _inputs(B, nh, nkv, S, seed, q_std=1.0):
    q = synth.normal_f32((B, nh * D), q_std, seed, "attn_q")
    kn = synth.normal_f32((B, nkv * D), 1.0, seed, "attn_k_new")
    vn = synth.normal_f32((B, nkv * D), 1.0, seed, "attn_v_new")
    kc = synth.normal_bf16((B, nkv, S, D), 1.0, seed, "attn_k_cache")
    vc = synth.normal_bf16((B, nkv, S, D), 1.0, seed, "attn_v_cache")
    return q, kn, vn, kc, vc


def _run(q, kn, vn, kc, vc, pos, nkv, both=True):
    B = q.shape[0]
    nh = q.shape[1] // D
    S = kc.shape[2]
    dk, dv = dev_bf16(kc), dev_bf16(vc)
    dpos = torch.tensor(np.asarray(pos, np.int32), device="cuda")
    ws = torch.empty(wb.attention_workspace_bytes(B, nh, nkv, S), dtype=torch.uint8, device="cuda").zero_()
    o32 = torch.full((B, nh * D), float("nan"), device="cuda")
    o16 = torch.zeros((B, nh * D), dtype=torch.bfloat16, device="cuda") if both else None
    wb.decode_attention(dev_f32(q), dev_f32(kn), dev_f32(vn), dk, dv, dpos, ws, o32, o16)
    torch.cuda.synchronize()
    return o32, o16, dk, dv


def _check(q, kn, vn, kc, vc, pos, nkv, what):
    o32, o16, dk, dv = _run(q, kn, vn, kc, vc, pos, nkv)
    ref = oracle.decode_attention(q, kn, vn, kc, vc, pos, nkv, D)
    assert np.array_equal(host_bits(dk), ref["k_cache"]), f"{what}: key cache"
    assert np.array_equal(host_bits(dv), ref["v_cache"]), f"{what}: value cache"
    got = o32.cpu().numpy()
    e = assert_fp32(got, ref["out"], what=what)
    assert torch.equal(o16, o32.to(torch.bfloat16)), f"{what}: bf16 output is not the fp32 rounded"
    return e


@pytest.mark.parametrize("n_valid", [1, 127, 128, 129, 1000, 1024])
def test_qwen_heads_cache_lengths(n_valid):
    # 12 query heads over 2 key-value heads of 128 (Qwen2.5-1.5B), cache 1024
    B, nh, nkv, S = 2, 12, 2, 1024
    args = _inputs(B, nh, nkv, S, seed=40 + n_valid)
    _check(*args, [n_valid - 1] * B, nkv, f"n_valid={n_valid}")


@pytest.mark.parametrize("B", [1, 4, 16])
def test_ragged_positions_across_the_batch(B):
    nh, nkv, S = 12, 2, 640
    rng = np.random.default_rng(B)
    pos = rng.integers(0, S, size=B)
    pos[0] = S - 1
    if B > 1:
        pos[1] = 0
    args = _inputs(B, nh, nkv, S, seed=7 * B)
    _check(*args, pos, nkv, f"B={B}")


@pytest.mark.parametrize("nh,nkv", [(4, 4), (8, 4), (12, 4), (8, 2), (12, 2), (16, 2)])
def test_group_sizes(nh, nkv):
    B, S = 3, 384
    args = _inputs(B, nh, nkv, S, seed=nh * 10 + nkv)
    _check(*args, [300, 129, 5], nkv, f"{nh}/{nkv}")


def test_sharp_softmax():
    # queries scaled by 8: scores of standard deviation 8, a softmax dominated
    # by a few slots in different chunks, so the merge's rescaling matters
    B, nh, nkv, S = 2, 12, 2, 1024
    args = _inputs(B, nh, nkv, S, seed=5, q_std=8.0)
    _check(*args, [1023, 700], nkv, "sharp")


def test_long_cache():
    # 32k slots: 256 chunks per (row, head) merged by the last one
    B, nh, nkv, S = 1, 12, 2, 32768
    args = _inputs(B, nh, nkv, S, seed=11)
    _check(*args, [S - 1], nkv, "32k")


def test_graph_replay_advances_positions():
    """Three decode steps replayed from one captured graph: the positions are
    read on the device, the ticket is reset for each replay, and every step
    matches the oracle run on the cache the previous steps left."""
    B, nh, nkv, S = 2, 12, 2, 512
    q, kn, vn, kc, vc = _inputs(B, nh, nkv, S, seed=3)
    dq, dkn, dvn = dev_f32(q), dev_f32(kn), dev_f32(vn)
    dk, dv = dev_bf16(kc), dev_bf16(vc)
    pos = np.array([126, 300], np.int32)
    dpos = torch.tensor(pos, device="cuda")
    ws = torch.empty(wb.attention_workspace_bytes(B, nh, nkv, S), dtype=torch.uint8, device="cuda").zero_()
    o32 = torch.empty((B, nh * D), device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        wb.decode_attention(dq, dkn, dvn, dk, dv, dpos, ws, o32, None, stream=s)  # warm
    torch.cuda.synchronize()
    kc_ref, vc_ref = host_bits(dk), host_bits(dv)
    with torch.cuda.graph(g, stream=s):
        wb.decode_attention(dq, dkn, dvn, dk, dv, dpos, ws, o32, None, stream=s)
    for step in range(3):
        pos = pos + 1
        q, kn, vn = (synth.normal_f32(a.shape, 1.0, 100 + step, t)
                     for a, t in ((q, "rq"), (kn, "rk"), (vn, "rv")))
        dq.copy_(torch.from_numpy(q))
        dkn.copy_(torch.from_numpy(kn))
        dvn.copy_(torch.from_numpy(vn))
        dpos.copy_(torch.from_numpy(pos))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.decode_attention(q, kn, vn, kc_ref, vc_ref, pos, nkv, D)
        kc_ref, vc_ref = ref["k_cache"], ref["v_cache"]
        assert np.array_equal(host_bits(dk), kc_ref)
        assert np.array_equal(host_bits(dv), vc_ref)
        assert_fp32(o32.cpu().numpy(), ref["out"], what=f"replay {step}")


def test_position_outside_the_cache_raises_the_device_flag():
    """Row 1 names slot S (one past the cache): the kernel touches nothing for
    that row and raises the flag; row 0 is still computed."""
    B, nh, nkv, S = 2, 12, 2, 256
    q, kn, vn, kc, vc = _inputs(B, nh, nkv, S, seed=9)
    o32, _, dk, dv = _run(q, kn, vn, kc, vc, [17, S], nkv, both=False)
    assert wb.device_error(reset=True) == 2
    ref = oracle.decode_attention(q[:1], kn[:1], vn[:1], kc[:1], vc[:1], [17], nkv, D)
    assert_fp32(o32[:1].cpu().numpy(), ref["out"], what="valid row")
    assert np.array_equal(host_bits(dk)[1], kc[1]) and np.array_equal(host_bits(dv)[1], vc[1])
    assert torch.isnan(o32[1]).all()


def test_group_merges():
    """17 chunks (a group of 16 and a group of 1, merged by the last group),
    exactly 16 chunks (one group), and 33 chunks, across three rows."""
    B, nh, nkv, S = 3, 12, 2, 4224
    args = _inputs(B, nh, nkv, S, seed=21)
    _check(*args, [2175, 2047, 4223], nkv, "groups")


def test_slots_past_the_token_are_never_read():
    """Cache slots after pos hold NaN and infinity bit patterns (stale or
    uninitialised memory): the output is the oracle's over slots 0..pos."""
    B, nh, nkv, S = 2, 12, 2, 512
    q, kn, vn, kc, vc = _inputs(B, nh, nkv, S, seed=13)
    pos = [200, 37]
    for b, p in enumerate(pos):
        kc[b, :, p + 1:] = 0x7FC0  # NaN
        vc[b, :, p + 1:] = 0x7F80  # +inf
    _check(q, kn, vn, kc, vc, pos, nkv, "stale tail")
