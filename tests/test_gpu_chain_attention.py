"""GPU parity of the decode chain with decode attention in every block (the
seeded attention stand-in replaced, "One Token, Kernel by Kernel", "The fix:
Part 10's split-KV kernel"): two steps replayed from one captured graph with
the positions advanced on the device; per block and step the h trace against
the oracle block with attention (teacher-forced on the GPU's input h and on
its q, k, v), the caches bit for bit, and the argmax."""
import numpy as np
import pytest
import torch

import oracle
from weight_streaming_gemv_bf16_gb300 import binding as wb
from weight_streaming_gemv_bf16_gb300 import chain as wc
from weight_streaming_gemv_bf16_gb300 import synth
from _util import assert_fp32, dev_bf16, dev_f32, host_bits

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


# 6 query heads of 128 over 2 key-value heads
SHAPE = synth.QwenShape(hidden=768, kv_dim=256, inter=512, vocab=1000, layers=2)


@pytest.mark.parametrize("B,pos0", [(1, [100]), (3, [100, 37, 253])])
def test_chain_with_attention_matches_oracle(B, pos0):
    sh, S = SHAPE, 256
    nkv = sh.kv_dim // 128
    seed = 5 + B
    blocks = [synth.qwen_block_weights(sh, seed, l) for l in range(sh.layers)]
    head = synth.qwen_head_weights(sh, seed)
    h0 = synth.qwen_hidden(sh, B, seed)
    kc = [synth.normal_bf16((B, nkv, S, 128), 1.0, seed + l, "chain/kc") for l in range(sh.layers)]
    vc = [synth.normal_bf16((B, nkv, S, 128), 1.0, seed + l, "chain/vc") for l in range(sh.layers)]
    dk = [dev_bf16(c) for c in kc]
    dv = [dev_bf16(c) for c in vc]
    pos = torch.tensor(np.asarray(pos0, np.int32), device="cuda")
    dblocks = [{k: dev_bf16(v) for k, v in b.items()} for b in blocks]
    dhead = {k: dev_bf16(v) for k, v in head.items()}
    ch = wc.qwen_chain(dblocks, dhead, None, dev_f32(h0), eps=sh.eps, trace=True, keep_qkv=True,
                       logits=True, caches=list(zip(dk, dv)), pos=pos)
    ch.chain.capture()
    for step in range(2):
        kc_before = [host_bits(t) for t in dk]
        vc_before = [host_bits(t) for t in dv]
        p = pos.cpu().numpy()
        ch.run()
        torch.cuda.synchronize()
        trace = ch.h_trace.cpu().numpy().astype(np.float64)
        h = h0.astype(np.float64)
        for l in range(sh.layers):
            q, k, v = (t.cpu().numpy().astype(np.float64) for t in ch.qkv[l])
            out = oracle.qwen_block_attention(h, blocks[l], kc_before[l], vc_before[l], p, nkv,
                                              sh.eps, qkv=(q, k, v))
            assert_fp32(trace[l], out["h"], what=f"step {step} block {l}")
            assert np.array_equal(host_bits(dk[l]), out["k_cache"]), f"step {step} k cache {l}"
            assert np.array_equal(host_bits(dv[l]), out["v_cache"]), f"step {step} v cache {l}"
            h = trace[l]
        logits = oracle.lmhead_logits(h, oracle.bf16_to_f64(head["gamma_f"]), head["Wlm"], sh.eps)
        assert_fp32(ch.logits.cpu().numpy(), logits, what=f"step {step} logits")
        pos += 1  # the next token of every row; the captured graph reads it on the device
