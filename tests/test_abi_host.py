"""Host-side checks of the C ABI that need no GPU: the library loads and exports
every function include/wsgemv.h declares; argument validation rejects bad
calls before anything is launched; every bulk copy the GEMV schedule issues
stays inside its source matrix and its ring stage, is 16-byte aligned, and the
copies of all CTAs cover every weight byte exactly once."""
import os
import re

import numpy as np
import pytest

from weight_streaming_gemv_bf16_gb300 import binding as wb
from _util import tuning

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from weight_streaming_gemv_bf16_gb300 import _build
    _build.build()
    return wb.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "wsgemv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(ws_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 30
    for n in names:
        assert hasattr(lib, n), n


def test_library_is_built_for_sm_103a(lib):
    assert "sm_103a" in wb.version()


# fake device addresses: the validation fails before any of them is touched
A = 0x7F0000000000
MIS = A + 8


@pytest.mark.parametrize("args,status", [
    ((A, A, A, 64, 12, 1), -3),     # K % 8 != 0
    ((A, A, A, 64, 16, 0), -3),     # B = 0
    ((A, A, A, 64, 16, 17), -3),    # B > 16
    ((A, A, A, 0, 16, 1), -3),      # M = 0
    ((None, A, A, 64, 16, 1), -1),  # null W
    ((MIS, A, A, 64, 16, 1), -2),   # misaligned W
    ((A, MIS, A, 64, 16, 1), -2),   # misaligned x
])
def test_gemv_argument_validation(lib, args, status):
    W, x, y, M, K, B = args
    assert lib.ws_gemv_bf16(W, x, y, M, K, B, None, 0, None) == status
    assert lib.ws_last_error()


def test_other_entry_points_validate(lib):
    assert lib.ws_rmsnorm_gemv(A, 7, A, A, A, 64, 16, 1, 1e-6, None, 0, None) == -1  # dtype
    assert lib.ws_swiglu_gemv(A, 0, None, A, A, A, 64, 16, 1, 1e-6, None, 0, None) == -1  # fp32 w/o norm
    assert lib.ws_lmhead_argmax(A, 0, A, A, A, None, 64, 16, 1, 1e-6, None, 0, None) == -1  # no workspace
    assert lib.ws_argmax_rows(A, A, 0, 10, A, 4096, None) == -3
    assert lib.ws_argmax_rows(A, A, 2, 10, A, 1, None) == -1  # workspace too small
    assert lib.ws_rmsnorm(A, A, A, 4, 12, 2, 1e-6, None) == -3
    assert lib.ws_rmsnorm(A, A, A, 4, 16, 5, 1e-6, None) == -1
    bad = wb.PrefetchPlan(0, 256, 128, 1)
    assert lib.ws_l2_prefetch(A, 4096, bad, None) == -1
    bulk = wb.PrefetchPlan(4, 256, 100, 3)
    assert lib.ws_l2_prefetch(A, 4096, bulk, None) == -2
    none = wb.PrefetchPlan(0, 0, 0, 0)
    assert lib.ws_l2_prefetch(A, 4096, none, None) == 0  # enqueues nothing
    assert lib.ws_test_bounded_wait(0, None) == -1
    t = wb.Tuning(96 * 1024, 0, 0, 0, 1, 0)
    assert lib.ws_set_tuning(wb.ctypes.byref(t)) == -1


@pytest.mark.parametrize("field,value", [("ctas_per_sm", 4), ("ctas_per_sm", -1), ("q4_mma", 3),
                                         ("q4_mma", -1)])
def test_tuning_rejects_out_of_range_residency_fields(lib, field, value):
    t = wb.get_tuning()
    setattr(t, field, value)
    assert lib.ws_set_tuning(wb.ctypes.byref(t)) == -1
    assert wb.get_tuning().ctas_per_sm == 0 and wb.get_tuning().q4_mma == 1  # unchanged


@pytest.mark.parametrize("B,nh,nkv,d,S,kc,wsb,status", [
    (2, 12, 2, 64, 256, A, 1 << 20, -3),     # head_dim != 128
    (2, 12, 1, 128, 256, A, 1 << 20, -3),    # 12 query heads per key-value head (> 8)
    (2, 12, 5, 128, 256, A, 1 << 20, -3),    # n_heads not a multiple of n_kv_heads
    (2, 12, 2, 128, 200, A, 1 << 20, -3),    # s_max not a multiple of 64
    (17, 12, 2, 128, 256, A, 1 << 20, -3),   # B > 16
    (0, 12, 2, 128, 256, A, 1 << 20, -3),    # B = 0
    (2, 12, 2, 128, 256, MIS + 2, 1 << 20, -2),  # misaligned cache
    (2, 12, 2, 128, 256, A, 64, -1),         # workspace too small
])
def test_decode_attention_validation(lib, B, nh, nkv, d, S, kc, wsb, status):
    assert lib.ws_decode_attention(A, A, A, kc, A, A, A, None, B, nh, nkv, d, S, A, wsb,
                                   None) == status
    assert lib.ws_last_error()


def test_decode_attention_alignment_checks(lib):
    # q 8-byte aligned, k_new and v_new 16-byte aligned, checked before anything runs
    args = dict(B=2, nh=12, nkv=2, d=128, S=256)
    def call(q=A, kn=A, vn=A):
        return lib.ws_decode_attention(q, kn, vn, A, A, A, A, None, args["B"], args["nh"],
                                       args["nkv"], args["d"], args["S"], A, 1 << 20, None)
    assert call(q=A + 4) == -2
    assert call(kn=A + 8) == -2
    assert call(vn=A + 8) == -2


def test_decode_attention_workspace(lib):
    def expect(B, nh, nkv, S):
        # tickets per group of 16 splits, per (row, head); G x 130 floats per
        # split (at most one per 64 slots) and per group; each part 256-byte aligned
        a = lambda v: -(-v // 256) * 256
        G, chunks = nh // nkv, S // 64
        groups = -(-chunks // 16)
        bg = B * nkv
        return (a(bg * groups * 4) + a(bg * 4) + a(bg * chunks * G * 130 * 4)
                + bg * groups * G * 130 * 4)
    for shape in [(1, 12, 2, 1024), (16, 12, 2, 32768), (3, 8, 8, 128), (2, 16, 2, 2176)]:
        assert wb.attention_workspace_bytes(*shape) == expect(*shape), shape
    assert wb.attention_workspace_bytes(1, 12, 2, 1024) == 256 + 256 + 2 * 16 * 6 * 520 + 2 * 6 * 520
    assert wb.attention_workspace_bytes(1, 12, 2, 1000) == 0
    assert wb.attention_workspace_bytes(1, 12, 1, 1024) == 0
    assert wb.attention_workspace_bytes(1, 12, 2, 1024, head_dim=64) == 0


def test_chain_create_rejects_bad_block_lists(lib):
    opts = wb.ChainOpts(batch=1, hidden=64, kv_dim=16, inter=128, vocab=100, eps=1e-6,
                        h_in=A, h_out=A + 4096)
    head = wb.BlockDesc(kind=wb.BLOCK_HEAD)
    head.u.head = wb.HeadBlock(A, A, A, None)
    mlp = wb.BlockDesc(kind=wb.BLOCK_MLP)
    mlp.u.mlp = wb.MlpBlock(A, A, A, A)
    h = wb.P()
    two = (wb.BlockDesc * 2)(head, mlp)  # head must be last and alone with MLP
    assert lib.ws_chain_create(two, 2, wb.ctypes.byref(opts), wb.ctypes.byref(h)) == -1
    one = (wb.BlockDesc * 1)(wb.BlockDesc(kind=9))
    assert lib.ws_chain_create(one, 1, wb.ctypes.byref(opts), wb.ctypes.byref(h)) == -1
    opts.batch = 0
    one = (wb.BlockDesc * 1)(head)
    assert lib.ws_chain_create(one, 1, wb.ctypes.byref(opts), wb.ctypes.byref(h)) == -3


SHAPES = [
    # (M, K, B, nmat, allow_split)
    (256, 256, 1, 1, False),      # fused RMSNorm + GEMV config
    (2048, 1536, 1, 1, False),    # merged QKV rows
    (1536, 1536, 1, 1, True),     # Wo
    (8960, 1536, 1, 2, False),    # gate/up pair
    (1536, 8960, 1, 1, True),     # Wd
    (256, 1536, 1, 1, True),      # K/V projection: split-K
    (256, 1536, 16, 1, True),
    (1536, 8960, 16, 1, True),    # activations too big: split needed
    (8960, 1536, 8, 2, True),
    (151936, 1536, 1, 1, False),  # LM head
    (768, 768, 16, 1, True),      # MLP chain block
    (37, 40, 3, 1, True),         # ragged tiny
    (1, 8, 1, 1, True),           # minimal
    (1000, 264, 5, 2, True),
]


@pytest.mark.parametrize("M,K,B,nmat,split", SHAPES)
def test_bulk_copies_in_bounds_aligned_and_covering(lib, M, K, B, nmat, split):
    sc = wb.gemv_plan(M, K, B, nmat=nmat, allow_split=split)
    assert sc["smem_bytes"] <= 227 * 1024
    assert 2 <= sc["NSW"] <= 8
    assert sc["piece_bytes"] % 128 == 0
    assert sc["grid"] % sc["S"] == 0 and sc["grid"] // sc["S"] <= sc["RG"]
    assert sc["KS"] * sc["S"] == K and sc["KS"] % 8 == 0 and sc["PC"] % 8 == 0
    assert sc["NP"] == -(-sc["KS"] // sc["PC"])
    warp_ring = sc["NSW"] * sc["piece_bytes"]
    covered = np.zeros(nmat * M * K * 2 // 16, np.int32)
    for cta in range(sc["grid"]):
        for src, dst, n in wb.debug_gemv_copies(M, K, B, nmat, split, cta):
            assert n > 0 and n % 16 == 0 and src % 16 == 0 and dst % 16 == 0
            assert 0 <= src and src + n <= nmat * M * K * 2
            # a copy never crosses from one matrix of a pair into the other
            assert src // (M * K * 2) == (src + n - 1) // (M * K * 2)
            warp, rest = divmod(dst, warp_ring)
            slot, off = divmod(rest, sc["piece_bytes"])
            assert warp < 8 and slot < sc["NSW"] and off + n <= sc["piece_bytes"]
            covered[src // 16:(src + n) // 16] += 1
    assert covered.min() == 1 and covered.max() == 1


Q4_SHAPES = [
    # (M, K, B, nmat): the Qwen2.5-1.5B products at 4 bits, ragged tails
    (2048, 1536, 1, 1),    # merged QKV rows
    (1536, 1536, 1, 1),    # Wo
    (8960, 1536, 1, 2),    # gate/up pair
    (1536, 8960, 1, 1),    # Wd: 17 super-groups and a tail of two groups
    (1536, 8960, 4, 1),
    (151936, 1536, 1, 1),  # LM head
    (37, 640, 3, 1),       # ragged rows, a one-group tail
    (1000, 1408, 2, 2),    # a three-group tail
    (5, 128, 4, 1),        # one group
]


# the tensor-core 4-bit kernel takes ops of at least two 16-row tasks per warp
Q4_MMA_SHAPES = [
    (151936, 1536, 1, 1),  # LM head
    (40000, 640, 3, 1),    # ragged rows, a one-group tail
    (40000, 1408, 2, 2),   # a pair, a three-group tail
]


@pytest.mark.parametrize("M,K,B,nmat,mma", [s + (False,) for s in Q4_SHAPES] +
                         [s + (True,) for s in Q4_MMA_SHAPES])
def test_q4_bulk_copies_in_bounds_aligned_and_covering(lib, M, K, B, nmat, mma):
    with tuning(q4_mma=2):  # the tensor-core plan at batch 1 too
        _q4_copies_check(M, K, B, nmat, mma)


def _q4_copies_check(M, K, B, nmat, mma):
    rb = wb.q4_row_bytes(K)
    _, sc = wb.debug_gemv_copies_q4(M, K, B, nmat, 0, mma)
    assert sc["smem_bytes"] <= 227 * 1024 and 2 <= sc["NSW"] <= 8
    assert sc["S"] == 1 and sc["KS"] == K
    assert sc["PC"] == K or sc["PC"] % 512 == 0
    assert sc["piece_bytes"] % 128 == 0
    warp_ring = sc["NSW"] * sc["piece_bytes"]
    covered = np.zeros(nmat * M * rb // 16, np.int32)
    for cta in range(sc["grid"]):
        copies, _ = wb.debug_gemv_copies_q4(M, K, B, nmat, cta, mma)
        for src, dst, n in copies:
            assert n > 0 and n % 16 == 0 and src % 16 == 0 and dst % 16 == 0
            assert 0 <= src and src + n <= nmat * M * rb
            assert src // rb == (src + n - 1) // rb  # within one row
            warp, rest = divmod(dst, warp_ring)
            slot, off = divmod(rest, sc["piece_bytes"])
            assert warp < 8 and slot < sc["NSW"] and off + n <= sc["piece_bytes"]
            covered[src // 16:(src + n) // 16] += 1
    assert covered.min() == 1 and covered.max() == 1


@pytest.mark.parametrize("M,K,nmat", [(2048, 1536, 1), (1536, 1536, 1), (8960, 1536, 2),
                                      (1536, 8960, 1), (151936, 1536, 1)])
def test_q4_batch1_plans_hold_two_ctas_per_sm(lib, M, K, nmat):
    """4-bit rows at batch 1 (the decode chain's shapes) plan two CTAs per SM:
    twice the grid of batch 4 and shared memory that leaves room for a
    second CTA (228 KB an SM, 1 KB of it kept per CTA); bf16 rows keep one."""
    _, b1 = wb.debug_gemv_copies_q4(M, K, 1, nmat, 0, 0)
    _, b4 = wb.debug_gemv_copies_q4(M, K, 4, nmat, 0, 0)
    assert b1["grid"] == 2 * b4["grid"]
    assert 2 * (b1["smem_bytes"] + 1024) <= 228 * 1024 and b1["NSW"] >= 2
    with tuning(ctas_per_sm=1):
        _, one = wb.debug_gemv_copies_q4(M, K, 1, nmat, 0, 0)
    assert one["grid"] == b4["grid"]
    bf = wb.gemv_plan(M, K, 1, nmat=nmat, allow_split=False)
    assert bf["grid"] <= b4["grid"]


def test_workspace_sizes(lib):
    assert wb.workspace_bytes(wb.OP_GEMV, 1536, 1536, 1) == 0  # no split needed
    assert wb.workspace_bytes(wb.OP_GEMV, 256, 1536, 1) > 0    # skinny: split
    assert wb.workspace_bytes(wb.OP_LMHEAD_ARGMAX, 151936, 1536, 1) > 0
    assert wb.workspace_bytes(wb.OP_ARGMAX_ROWS, 16, 151936, 1) > 0
    assert wb.workspace_bytes(wb.OP_GEMV, 1536, 8960, 16) > 0  # activations need a split


def test_chain_create_rejects_bad_attention_and_weight_format(lib):
    """Host-side checks of the chain options (nothing is allocated or
    launched): attention needs heads of 128, s_max a multiple of 64 and
    positions; 4-bit weights need batch <= 4 and no persistent mode."""
    blk = wb.BlockDesc(kind=wb.BLOCK_QWEN)
    blk.u.qwen = wb.QwenBlock(*([A] * 9), None, None, None, None, A, A)
    blocks = (wb.BlockDesc * 1)(blk)
    h = wb.P()

    def create(**kw):
        o = wb.ChainOpts(batch=1, hidden=768, kv_dim=256, inter=512, vocab=0, eps=1e-6,
                         h_in=A, h_out=A + 4096)
        for k, v in kw.items():
            setattr(o, k, v)
        return lib.ws_chain_create(blocks, 1, wb.ctypes.byref(o), wb.ctypes.byref(h))
    assert create(attention=1, s_max=256, pos=None) == -1          # no positions
    assert create(attention=1, s_max=200, pos=A) == -1             # s_max not a multiple of 64
    assert create(attention=1, s_max=256, pos=A, kv_dim=64) == -1  # key-value heads not 128
    assert create(attention=1, s_max=256, pos=A, persistent=1) == -1
    assert create(weight_format=2) == -1                           # unknown format
    assert create(weight_format=1, batch=8) == -1                  # 4-bit: batch <= 4
    assert create(weight_format=1, persistent=1) == -1
    assert lib.ws_last_error()


def test_q4_plans_fit_every_k():
    """Every K in 128..12288 (every tail length), batch 1-4, one matrix or a
    pair: a 4-bit plan (CUDA-core kernel, or the tensor-core one where it
    qualifies) fits shared memory, keeps two ring stages or more, cuts pieces
    on super-groups, and CTA 0's copies stay inside the ring."""
    for K in range(128, 12288 + 1, 128):
        for B in (1, 2, 3, 4):
            for nmat in (1, 2):
                for mma, M in ((False, 3000), (True, 40000)):
                    if B * K * 2 > 96 * 1024:
                        continue  # activations of the full K must fit
                    try:
                        copies, sc = wb.debug_gemv_copies_q4(M, K, B, nmat, 0, mma)
                    except wb.WsError:
                        assert mma, (K, B, nmat)  # only the tensor-core plan may decline
                        continue
                    assert sc["smem_bytes"] <= 227 * 1024 and sc["NSW"] >= 2, (K, B, nmat, mma)
                    assert sc["PC"] == K or sc["PC"] % 512 == 0, (K, sc["PC"])
                    ring = 8 * sc["NSW"] * sc["piece_bytes"]
                    assert all(dst + n <= ring for _, dst, n in copies), (K, B, nmat, mma)


def test_bf16_plans_fit_every_k():
    """bf16 plans over K (every 8 up to 1024, every 64 up to 16384), batch
    1-16, one matrix or a pair, with and without a K split: each that plans
    fits shared memory and keeps two ring stages or more."""
    for K in list(range(8, 1024, 8)) + list(range(1024, 16385, 64)):
        for B in (1, 4, 8, 16):
            for nmat in (1, 2):
                for split in (False, True):
                    try:
                        sc = wb.gemv_plan(2000, K, B, nmat=nmat, allow_split=split)
                    except wb.WsError:
                        continue
                    assert sc["smem_bytes"] <= 227 * 1024 and sc["NSW"] >= 2, (K, B, nmat, split)


def test_chain_create_rejects_what_batch_tiles_do_not_cover(lib):
    """Batches above 16 run in 16-row tiles: up to 128 rows, bf16 weights,
    no attention, no training saves (checked before anything is allocated)."""
    blk = wb.BlockDesc(kind=wb.BLOCK_QWEN)
    blk.u.qwen = wb.QwenBlock(*([A] * 9), None, None, None, None, A, A)
    blocks = (wb.BlockDesc * 1)(blk)
    h = wb.P()

    def create(**kw):
        o = wb.ChainOpts(batch=32, hidden=768, kv_dim=256, inter=512, vocab=0, eps=1e-6,
                         h_in=A, h_out=A + 4096)
        for k, v in kw.items():
            setattr(o, k, v)
        return lib.ws_chain_create(blocks, 1, wb.ctypes.byref(o), wb.ctypes.byref(h))
    assert create(batch=129) == -3
    assert create(weight_format=1) == -3
    assert create(attention=1, s_max=256, pos=A) == -3
    mlp = wb.BlockDesc(kind=wb.BLOCK_MLP)
    mlp.u.mlp = wb.MlpBlock(A, A, A, A)
    o = wb.ChainOpts(batch=17, hidden=768, eps=1e-5, x_in=A, y_out=A + 4096, mlp_gelu_grad=A)
    assert lib.ws_chain_create((wb.BlockDesc * 1)(mlp), 1, wb.ctypes.byref(o),
                               wb.ctypes.byref(h)) == -3
    assert b"batch tiles" in lib.ws_last_error()


def test_mlp_backward_create_validates_before_allocating(lib):
    """The backward's shape, alignment and option checks (no GPU needed: they
    come before any device call)."""
    blocks = (wb.MlpBlock * 2)(wb.MlpBlock(A, A, A, A), wb.MlpBlock(A, A, A, A))
    grads = (wb.MlpGrads * 2)(wb.MlpGrads(A, A, A, A), wb.MlpGrads(A, A, A, A))
    h = wb.P()

    def create(n=2, **kw):
        o = wb.MlpBackwardOpts(batch=4, width=768, x_in=A, acts=A, ln=A, gelu_grad=A,
                               ln_stats=A, dx=A, distance=1)
        for k, v in kw.items():
            setattr(o, k, v)
        return lib.ws_mlp_backward_create(blocks, grads, n, wb.ctypes.byref(o), wb.ctypes.byref(h))
    assert create(batch=0) == -3
    assert create(batch=17) == -3
    assert create(width=96) == -3        # not a multiple of 64
    assert create(width=2048) == -3      # wider than 1024
    assert create(distance=0) == -1
    assert create(dx=None) == -2
    assert create(acts=A + 8) == -2      # not 16-byte aligned
    assert create(dln_trace=A + 2) == -2
    assert create(n=0) == -1
    bad = (wb.MlpGrads * 2)(wb.MlpGrads(A, A, A, A), wb.MlpGrads(A, None, A, A))
    o = wb.MlpBackwardOpts(batch=4, width=768, x_in=A, acts=A, ln=A, gelu_grad=A, ln_stats=A,
                           dx=A, distance=1)
    assert lib.ws_mlp_backward_create(blocks, bad, 2, wb.ctypes.byref(o), wb.ctypes.byref(h)) == -2
    assert lib.ws_last_error()
