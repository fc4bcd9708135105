"""Backward pass of the LayerNorm -> Linear(+bias) -> GELU block for the oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring): shares no code with the
CUDA library.

"Making small PyTorch ops faster on a laptop GPU", "It works in training
too": in the backward pass the gradient of layer i reads W_i again, so the
prefetch fetches W_(i-1), and the gradients match plain PyTorch bit for bit
(a prefetch writes nothing).  The block is the one of "Beyond language
models" (72 x [LayerNorm(768) -> Linear(768, 768) -> GELU] in bf16).

Readings where the pages are silent (the same module-by-module bf16 rule as
the forward block):

* forward: ln = bf16(LN(x)), lin = bf16(ln.W^T + b), z = bf16(gelu(lin)),
  LayerNorm statistics exact (double), biased variance, eps inside the root;
* backward, given dz (bf16): every module computes its gradients exactly
  (double here) from its saved bf16 inputs and rounds each gradient it hands
  on or keeps to bf16 once:
  dlin = bf16(dz * gelu'(lin)), gelu'(t) = Phi(t) + t phi(t) (exact erf GELU);
  dln = bf16(dlin . W); dW = bf16(dlin^T . ln); db = bf16(sum_b dlin);
  with xh = (x - mean) * rstd and g = dln * gamma:
  dx = bf16(rstd * (g - mean_k g - xh * mean_k(g * xh))),
  dgamma = bf16(sum_b dln * xh), dbeta = bf16(sum_b dln).
"""
from __future__ import annotations

import math

import numpy as np


def gelu_grad(t) -> np.ndarray:
    """d/dt of t * Phi(t): Phi(t) + t * phi(t), elementwise in double."""
    t = np.asarray(t, np.float64)
    erf = np.vectorize(math.erf)
    Phi = 0.5 * (1.0 + erf(t / math.sqrt(2.0)))
    phi = np.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi)
    return Phi + t * phi


def _gelu(t):
    t = np.asarray(t, np.float64)
    erf = np.vectorize(math.erf)
    return 0.5 * t * (1.0 + erf(t / math.sqrt(2.0)))


def _layernorm_parts(x, eps):
    mean = x.mean(axis=1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    return mean, rstd, (x - mean) * rstd


def mlp_block_forward(x, gamma, beta, W, b, eps: float = 1e-5, rounding=None):
    """The block's forward on double arrays; `rounding` (a callable, or None
    for the exact block) is applied to each module's output."""
    r = rounding if rounding is not None else (lambda v: v)
    _, _, xh = _layernorm_parts(np.asarray(x, np.float64), eps)
    ln = r(xh * gamma + beta)
    lin = r(ln @ W.T + b)
    return {"ln": ln, "lin": lin, "z": r(_gelu(lin))}


def mlp_block_backward(x, gamma, beta, W, b, dz, eps: float = 1e-5, rounding=None,
                       forced=None) -> dict:
    """Gradients of the block (see the module docstring) on double arrays:
    x [B][w], gamma, beta, b [w], W [w_out][w_in], dz [B][w_out].  With
    rounding=None every step is exact (the derivative of the exact block);
    with a rounding callable (bf16) each saved activation and each gradient
    is rounded where the module-by-module reading puts it.

    forced: optional dict of module inputs taken as given instead of
    computed -- "ln" (the Linear's input), "lin" (the GELU's input), "dlin"
    (the Linear's output gradient), "dln" (the LayerNorm's output gradient).
    Each module's outputs then follow from its actual inputs, so a rounded
    intermediate that a GPU took to the other bf16 neighbour is checked
    where it was formed, not in everything after it."""
    r = rounding if rounding is not None else (lambda v: v)
    fz = forced or {}
    x = np.asarray(x, np.float64)
    f = mlp_block_forward(x, gamma, beta, W, b, eps, rounding)
    ln = np.asarray(fz["ln"], np.float64) if "ln" in fz else f["ln"]
    lin = np.asarray(fz["lin"], np.float64) if "lin" in fz else f["lin"]
    dlin = r(np.asarray(dz, np.float64) * gelu_grad(lin))
    if "dlin" in fz:
        dlin = np.asarray(fz["dlin"], np.float64)
    dln = r(dlin @ W)
    if "dln" in fz:
        dln = np.asarray(fz["dln"], np.float64)
    dW = r(dlin.T @ ln)
    db = r(dlin.sum(axis=0))
    _, rstd, xh = _layernorm_parts(x, eps)
    g = dln * gamma
    dx = r(rstd * (g - g.mean(axis=1, keepdims=True)
                   - xh * (g * xh).mean(axis=1, keepdims=True)))
    return {"dx": dx, "dW": dW, "db": db, "dgamma": r((dln * xh).sum(axis=0)),
            "dbeta": r(dln.sum(axis=0)), "dlin": dlin, "dln": dln, "z": f["z"]}


def mean_square_loss_grad(z) -> np.ndarray:
    """d/dz of mean(z^2) over all elements: 2 z / N."""
    z = np.asarray(z, np.float64)
    return 2.0 * z / z.size


def mlp_chain_backward(x, blocks, eps: float = 1e-5, dz=None, rounding=None) -> dict:
    """Forward then backward through a chain of blocks (dicts of double
    arrays gamma, beta, W, b): block i's input gradient is block i-1's output
    gradient.  dz: the loss gradient of the last output, or None for the
    mean-square loss (rounded like every other gradient).  Returns per block
    the gradients of mlp_block_backward and the chain input's dx."""
    r = rounding if rounding is not None else (lambda v: v)
    xs = [np.asarray(x, np.float64)]
    for blk in blocks:
        xs.append(mlp_block_forward(xs[-1], blk["gamma"], blk["beta"], blk["W"], blk["b"], eps,
                                    rounding)["z"])
    g = r(mean_square_loss_grad(xs[-1])) if dz is None else np.asarray(dz, np.float64)
    loss_grad = g
    grads = [None] * len(blocks)
    for i in range(len(blocks) - 1, -1, -1):
        blk = blocks[i]
        grads[i] = mlp_block_backward(xs[i], blk["gamma"], blk["beta"], blk["W"], blk["b"], g,
                                      eps, rounding)
        g = grads[i]["dx"]
    return {"grads": grads, "dx": g, "outputs": xs[1:], "loss_grad": loss_grad}


def chain_prefetch_order(n_blocks: int, backward: bool) -> list:
    """Which block's weights the prefetch fetches while block i runs: block
    i + 1 going forward, block i - 1 going backward (the backward pass visits
    blocks n-1 .. 0, and block i's gradient reads W_i itself); None at the
    end of each pass."""
    if backward:
        return [(i, i - 1 if i > 0 else None) for i in range(n_blocks - 1, -1, -1)]
    return [(i, i + 1 if i + 1 < n_blocks else None) for i in range(n_blocks)]
