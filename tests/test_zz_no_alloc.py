"""ws_gemv_bf16_noalloc: the GEMV entry point for callers that cannot allocate
device memory when they need it (code running during CUDA graph capture,
serving loops that must not allocate after start-up, hosts that hand over only
their own buffers).  It keeps its split-K scratch in a fixed device array owned
by the library instead of asking for a workspace.

This file is collected last on purpose.  Each check runs the no-allocation
call twice in a row (the second call reuses the scratch array the first one
left behind) and compares it with ws_gemv_bf16 given its own workspace and
with the double-accumulating oracle GEMV, within the fp32 tolerance the other
GEMV tests use.  It passes alone in a fresh process and after the other
tests."""
import numpy as np
import pytest
import torch

import oracle
from weight_streaming_gemv_bf16_gb300 import binding as wb
from weight_streaming_gemv_bf16_gb300 import synth
from _util import assert_fp32, bf16_bits_to_f64, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("M,K,B", [
    (256, 1536, 1),     # a skinny K/V-projection shape: the schedule splits K
    (256, 1536, 16),
    (1536, 8960, 16),   # activations too large for shared memory: split needed
    (1000, 1536, 3),    # no split: no scratch used at all
])
def test_noalloc_matches_workspace_entry_point_twice(M, K, B):
    Wh = synth.normal_bf16((M, K), 0.02, 31, f"na/W{M}x{K}")
    W = dev_bf16(Wh)
    xs = [synth.normal_bf16((B, K), 1.0, s, f"na/x{s - 30}/{B}") for s in (31, 32)]
    ws = wb.new_workspace(wb.OP_GEMV, M, K, B)
    for xh in xs:
        x = dev_bf16(xh)
        ref = torch.empty((B, M), device="cuda")
        wb.gemv_bf16(W, x, ref, workspace=ws)
        got = torch.full((B, M), float("nan"), device="cuda")
        wb.gemv_bf16_noalloc(W, x, got)
        torch.cuda.synchronize()
        g = got.cpu().numpy()
        assert_fp32(g, ref.cpu().numpy().astype(np.float64), what=f"noalloc {M}x{K} B={B}")
        exact = oracle.gemv(Wh, bf16_bits_to_f64(xh), threads=8)
        assert_fp32(g, exact, what=f"noalloc {M}x{K} B={B} vs oracle")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # a split-K scratch larger than the fixed 1 MiB array: clear error, no launch
    M, K, B = 8192, 8960, 16
    W = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    x = torch.empty((B, K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((B, M), device="cuda")
    with pytest.raises(wb.WsError) as e:
        wb.gemv_bf16_noalloc(W, x, y)
    assert e.value.status == -3 and "scratch" in str(e.value)
