"""GPU parity of the training path of the LayerNorm -> Linear -> GELU chain
("Making small PyTorch ops faster on a laptop GPU", "It works in training
too"): the training forward's saved tensors, and the backward chain checked
module by module against the oracle on the module's actual inputs (the
GPU's own ln, GELU input, dlin and dln: each rounded intermediate is checked
where it is formed), the loss gradient, bit-identical gradients with and
without the W_(i-1) prefetch (and its decoy) and over replays, and the
end-to-end drift against the oracle's whole training step."""
import numpy as np
import pytest
import torch

import oracle
from oracle import train as otr
from weight_streaming_gemv_bf16_gb300 import binding as wb
from weight_streaming_gemv_bf16_gb300 import chain as wc
from weight_streaming_gemv_bf16_gb300 import synth
from _util import assert_bf16_close, assert_ulp, bf16_bits_to_f64, dev_bf16, host_bits

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


def _setup(sh, B, seed):
    blocks = [synth.mlp_block_weights(sh, seed, i) for i in range(sh.blocks)]
    x = synth.mlp_input(sh, B, seed)
    dblocks = [{k: dev_bf16(v) for k, v in b.items()} for b in blocks]
    return blocks, x, dblocks


def _f64(blk):
    return {k: bf16_bits_to_f64(v) for k, v in blk.items()}


def _check_backward(sh, blocks, x, fwd, bw, dz_bits=None, every=1):
    """Module-by-module parity of every `every`-th block (and the last)."""
    L, (B, w) = sh.blocks, x.shape
    acts = host_bits(fwd.trace)
    lnb, preb = host_bits(fwd.ln), host_bits(fwd.pre)
    dxt, dlt, dnt = host_bits(bw.dx_trace), host_bits(bw.dlin_trace), host_bits(bw.dln_trace)
    # the loss gradient: given, or bf16(2 z / N) of the GPU's chain output
    if dz_bits is None:
        ref = otr.mean_square_loss_grad(bf16_bits_to_f64(acts[L - 1]))
        assert_ulp(dxt[L], oracle.f64_to_bf16(ref), what="loss gradient")
    else:
        assert np.array_equal(dxt[L], dz_bits)
    assert np.array_equal(host_bits(bw.dx), dxt[0])
    for i in range(L):
        if i % every and i != L - 1:
            continue
        b = _f64(blocks[i])
        xi = bf16_bits_to_f64(x if i == 0 else acts[i - 1])
        dz = bf16_bits_to_f64(dxt[i + 1])
        forced = {"ln": bf16_bits_to_f64(lnb[i]), "lin": bf16_bits_to_f64(preb[i]),
                  "dlin": bf16_bits_to_f64(dlt[i]), "dln": bf16_bits_to_f64(dnt[i])}
        # exact values (no rounding) of each module's outputs on its actual inputs
        ex = otr.mlp_block_backward(xi, b["gamma"], b["beta"], b["W"], b["b"], dz, sh.eps,
                                    rounding=None, forced=forced)
        free = otr.mlp_block_backward(xi, b["gamma"], b["beta"], b["W"], b["b"], dz, sh.eps,
                                      rounding=None, forced={"lin": forced["lin"]})
        # dlin: one rounding of dz * gelu'(t) -- within 1 ulp
        assert_ulp(dlt[i], oracle.f64_to_bf16(free["dlin"]), what=f"bwd block {i} dlin")
        g = bw.grads[i]
        assert_bf16_close(dnt[i], ex["dln"], what=f"bwd block {i} dln")
        assert_bf16_close(host_bits(g["dW"]), ex["dW"], what=f"bwd block {i} dW")
        assert_bf16_close(host_bits(g["db"]), ex["db"][None, :], what=f"bwd block {i} db")
        assert_bf16_close(dxt[i], ex["dx"], what=f"bwd block {i} dx")
        assert_bf16_close(host_bits(g["dgamma"]), ex["dgamma"][None, :], what=f"bwd block {i} dgamma")
        assert_bf16_close(host_bits(g["dbeta"]), ex["dbeta"][None, :], what=f"bwd block {i} dbeta")


def _run_training(sh, B, seed, **kw):
    blocks, x, dblocks = _setup(sh, B, seed)
    fwd = wc.mlp_chain(dblocks, dev_bf16(x), eps=sh.eps, training=True)
    fwd.chain.capture()
    fwd.run()
    bw = wc.mlp_backward(dblocks, fwd, traces=True, **kw)
    bw.bwd.capture()
    bw.run()
    bw.run()  # replays write the same gradients
    torch.cuda.synchronize()
    return blocks, x, dblocks, fwd, bw


@pytest.mark.parametrize("B", [4, 16])
def test_training_forward_keeps_outputs_and_saves_module_inputs(B):
    """The 72-block chain: the training forward's outputs equal the plain
    forward's bit for bit; its saved ln, GELU input, gelu' and LayerNorm
    statistics match the oracle on the GPU's own block inputs."""
    sh = synth.MlpShape()
    blocks, x, dblocks = _setup(sh, B, 41)
    plain = wc.mlp_chain(dblocks, dev_bf16(x), eps=sh.eps, trace=True)
    plain.chain.capture()
    plain.run()
    fwd = wc.mlp_chain(dblocks, dev_bf16(x), eps=sh.eps, training=True)
    fwd.chain.capture()
    fwd.run()
    torch.cuda.synchronize()
    assert torch.equal(plain.trace.cpu(), fwd.trace.cpu())
    assert torch.equal(plain.y_out.cpu(), fwd.y_out.cpu())
    acts = host_bits(fwd.trace)
    lnb, preb = host_bits(fwd.ln), host_bits(fwd.pre)
    gg, st = fwd.gelu_grad.cpu().numpy(), fwd.ln_stats.cpu().numpy()
    for i in (0, 1, 35, 71):
        xi = bf16_bits_to_f64(x if i == 0 else acts[i - 1])
        mean = xi.mean(axis=1)
        var = ((xi - mean[:, None]) ** 2).mean(axis=1)
        assert np.allclose(st[i][:, 0], mean, rtol=1e-5, atol=1e-6)
        assert np.allclose(st[i][:, 1], 1.0 / np.sqrt(var + sh.eps), rtol=1e-5)
        b = _f64(blocks[i])
        ln_exact = oracle.layernorm(xi, b["gamma"], b["beta"], sh.eps)
        assert_ulp(lnb[i], oracle.f64_to_bf16(ln_exact), what=f"saved ln block {i}")
        lin = oracle.gemv(blocks[i]["W"], bf16_bits_to_f64(lnb[i]), 8) + b["b"][None, :]
        assert_bf16_close(preb[i], lin, what=f"saved pre-activation block {i}")
        ref = otr.gelu_grad(bf16_bits_to_f64(preb[i]))
        assert np.max(np.abs(gg[i] - ref)) < 2e-6 * max(1.0, float(np.abs(ref).max()))
        # the block's output is the GELU of the saved pre-activation
        assert_ulp(acts[i], oracle.f64_to_bf16(oracle.gelu(bf16_bits_to_f64(preb[i]))),
                   what=f"output block {i}")


@pytest.mark.parametrize("B", [4, 16])
def test_backward_72_blocks_matches_oracle_module_by_module(B):
    sh = synth.MlpShape()
    blocks, x, dblocks, fwd, bw = _run_training(sh, B, 42)
    assert wb.device_error() == 0
    _check_backward(sh, blocks, x, fwd, bw, every=1)


@pytest.mark.parametrize("B,w,L", [(1, 64, 1), (5, 256, 3), (2, 1024, 2), (16, 192, 2),
                                   (3, 320, 2)])
def test_backward_edge_shapes(B, w, L):
    """The smallest and largest widths, batch 1, a partly filled batch tile
    (5 rows of 16), a single block, a width that leaves a partial TMA box
    (320 rows: one box of 256 and one of 64 valid rows)."""
    sh = synth.MlpShape(width=w, blocks=L)
    blocks, x, dblocks, fwd, bw = _run_training(sh, B, 43)
    assert wb.device_error() == 0
    _check_backward(sh, blocks, x, fwd, bw)


def test_backward_with_given_loss_gradient():
    sh = synth.MlpShape(width=256, blocks=3)
    blocks, x, dblocks = _setup(sh, 4, 44)
    fwd = wc.mlp_chain(dblocks, dev_bf16(x), eps=sh.eps, training=True)
    fwd.chain.capture()
    fwd.run()
    dz = synth.normal_bf16((4, 256), 0.01, 44, "bwd/dz")
    bw = wc.mlp_backward(dblocks, fwd, dz=dev_bf16(dz), traces=True)
    bw.bwd.capture()
    bw.run()
    torch.cuda.synchronize()
    _check_backward(sh, blocks, x, fwd, bw, dz_bits=dz)


def _grads_host(bw):
    out = [host_bits(bw.dx)]
    for g in bw.grads:
        out += [host_bits(g[k]) for k in ("dW", "db", "dgamma", "dbeta")]
    return out


@pytest.mark.parametrize("B", [4, 16])
def test_backward_prefetch_and_decoy_leave_gradients_bit_identical(B):
    """W_(i-1) prefetched while block i's gradient runs (a fixed plan, the
    tuned plan, and the decoy aimed at the wrong block): the same bits."""
    sh = synth.MlpShape()
    blocks, x, dblocks = _setup(sh, B, 45)
    fwd = wc.mlp_chain(dblocks, dev_bf16(x), eps=sh.eps, training=True)
    fwd.chain.capture()
    fwd.run()
    base = wc.mlp_backward(dblocks, fwd)
    base.bwd.capture()
    base.run()
    torch.cuda.synchronize()
    ref = _grads_host(base)
    runs = [wc.mlp_backward(dblocks, fwd, prefetch=2, fixed_plan=wb.PrefetchPlan(16, 256, 128, 1)),
            wc.mlp_backward(dblocks, fwd, prefetch=2, fixed_plan=wb.PrefetchPlan(16, 256, 16384, 3),
                            decoy=True),
            wc.mlp_backward(dblocks, fwd, prefetch=1, tune_pairs=8)]
    for r in runs:
        if r.bwd.opts.prefetch == 1:
            r.bwd.tune()
            (mode, *_), lo, mean = r.bwd.plan()
            assert np.isfinite(lo) and (mode == 0 or lo > 0.01)
        r.bwd.capture()
        r.run()
        r.run()
        torch.cuda.synchronize()
        for a, b in zip(_grads_host(r), ref):
            assert np.array_equal(a, b)


def test_backward_end_to_end_against_the_oracle_training_step():
    """No teacher forcing: the oracle's whole training step (rounded forward,
    mean-square loss, rounded backward through 12 blocks of width 768) against
    the GPU's.  Rounding differences compound through the blocks, so the
    drift is reported and bounded against gross errors only; the per-module
    checks above carry the tolerance."""
    sh = synth.MlpShape(blocks=12)
    blocks, x, dblocks, fwd, bw = _run_training(sh, 4, 46)
    ref = otr.mlp_chain_backward(bf16_bits_to_f64(x), [_f64(b) for b in blocks], sh.eps,
                                 rounding=oracle.round_bf16)
    worst = 0.0
    for name, got, exp in [("dx", bw.dx, ref["dx"]),
                           ("dW block 0", bw.grads[0]["dW"], ref["grads"][0]["dW"]),
                           ("dW block 11", bw.grads[11]["dW"], ref["grads"][11]["dW"])]:
        g = bf16_bits_to_f64(host_bits(got))
        rms = np.sqrt(np.mean(exp * exp))
        e = float(np.max(np.abs(g - exp)) / rms)
        print(f"end-to-end {name}: max |gpu - oracle| / rms {e:.3g}")
        worst = max(worst, e)
    assert worst < 0.25
