"""Seeded synthetic inputs for the decode chain, shared by the tests, the
benchmark and the oracle's callers.

This module draws random numbers and stores them in the formats the chain
reads (bf16 / fp16 bit patterns as uint16, fp32); it holds none of the
method's arithmetic.  Every tensor gets its own independent stream, keyed by
(seed, tag): torch's CPU generator seeded with seed * 2^32 + crc32(tag), so a
tensor does not change when another one is added or resized.  Rounding from
float32 to bf16/fp16 uses torch's own conversions (round to nearest even).

Shapes follow the pages' models:
* Qwen2.5-1.5B decode block ("One Token, Kernel by Kernel: A Decode Step on a
  Laptop GPU", Step 1 "The setup" and "The whole step"): hidden 1536, 2 KV heads
  x 128, MLP 8960 with SwiGLU, 28 blocks, LM head 151,936 x 1,536.
* MLP chain ("Making small PyTorch ops faster on a laptop GPU", "Beyond
  language models"): 72 x [LayerNorm(768) -> Linear(768, 768) -> GELU].
* Qwen2.5-0.5B RMSNorm rows, hidden 896, fp16 ("GPU Kernel Optimization",
  Results).

Distributions (unstated on the pages, chosen): weights ~ N(0, 0.02), norm
scales ~ U(0.5, 1.5), biases and LayerNorm shifts ~ N(0, 0.02), activations and
the attention stand-in ~ N(0, 1).
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np
import torch

WEIGHT_STD = 0.02


def _gen(seed: int, tag: str) -> torch.Generator:
    return torch.Generator().manual_seed((int(seed) << 32) + zlib.crc32(tag.encode()))


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


_CHUNK = 1 << 23


def _normal(shape, std, seed, tag) -> torch.Tensor:
    # large tensors are drawn in chunks of 2^23 values, chunk i from the stream
    # of (seed, tag#i): torch's CPU generator is much slower on huge single draws
    n = int(np.prod(shape)) if len(shape) else 1
    if n <= _CHUNK:
        t = torch.randn(tuple(shape), generator=_gen(seed, tag), dtype=torch.float32)
    else:
        t = torch.empty(n, dtype=torch.float32)
        for i, lo in enumerate(range(0, n, _CHUNK)):
            hi = min(n, lo + _CHUNK)
            t[lo:hi] = torch.randn(hi - lo, generator=_gen(seed, f"{tag}#{i}"))
        t = t.view(tuple(shape))
    return t.mul_(std) if std != 1.0 else t


def _uniform(shape, lo, hi, seed, tag) -> torch.Tensor:
    t = torch.rand(tuple(shape), generator=_gen(seed, tag), dtype=torch.float32)
    return t.mul_(hi - lo).add_(lo)


def normal_f32(shape, std: float, seed: int, tag: str) -> np.ndarray:
    return _normal(shape, std, seed, tag).numpy()


def normal_bf16(shape, std: float, seed: int, tag: str) -> np.ndarray:
    """bf16 bit patterns of N(0, std^2) draws (drawn in fp32, rounded once)."""
    return _bits(_normal(shape, std, seed, tag).to(torch.bfloat16))


def uniform_bf16(shape, lo: float, hi: float, seed: int, tag: str) -> np.ndarray:
    return _bits(_uniform(shape, lo, hi, seed, tag).to(torch.bfloat16))


def normal_fp16(shape, std: float, seed: int, tag: str) -> np.ndarray:
    return _bits(_normal(shape, std, seed, tag).to(torch.float16))


def uniform_fp16(shape, lo: float, hi: float, seed: int, tag: str) -> np.ndarray:
    return _bits(_uniform(shape, lo, hi, seed, tag).to(torch.float16))


def bf16_bits_as_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (a bit move: bf16 is the top half)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# workload shapes
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class QwenShape:
    hidden: int = 1536        # H
    kv_dim: int = 256         # 2 KV heads x 128
    inter: int = 8960         # I
    vocab: int = 151936       # V
    layers: int = 28          # L
    eps: float = 1e-6

    def block_weight_elems(self) -> int:
        H, KV, I = self.hidden, self.kv_dim, self.inter
        return 2 * H * H + 2 * KV * H + 3 * I * H

    def block_weight_bytes(self) -> int:
        return 2 * self.block_weight_elems()

    def lm_head_bytes(self) -> int:
        return 2 * self.vocab * self.hidden

    def chain_weight_bytes(self) -> int:
        return self.layers * self.block_weight_bytes() + self.lm_head_bytes()

    def chain_gamma_bytes(self) -> int:
        return 2 * self.hidden * (2 * self.layers + 1)


QWEN2_5_1_5B = QwenShape()


def qwen_block_weights(shape: QwenShape, seed: int, layer: int) -> dict:
    """bf16 bit arrays of one decoder block: gamma1, Wq, Wk, Wv, Wo, gamma2, Wg, Wu, Wd."""
    H, KV, I = shape.hidden, shape.kv_dim, shape.inter
    t = f"qwen/L{layer}/"
    specs = {
        "gamma1": ("u", (H,)), "Wq": ("n", (H, H)), "Wk": ("n", (KV, H)),
        "Wv": ("n", (KV, H)), "Wo": ("n", (H, H)), "gamma2": ("u", (H,)),
        "Wg": ("n", (I, H)), "Wu": ("n", (I, H)), "Wd": ("n", (H, I)),
    }

    def make(item):
        name, (kind, shp) = item
        if kind == "u":
            return name, uniform_bf16(shp, 0.5, 1.5, seed, t + name)
        return name, normal_bf16(shp, WEIGHT_STD, seed, t + name)

    return dict(make(item) for item in specs.items())


def qwen_head_weights(shape: QwenShape, seed: int) -> dict:
    return {
        "gamma_f": uniform_bf16((shape.hidden,), 0.5, 1.5, seed, "qwen/final/gamma"),
        "Wlm": normal_bf16((shape.vocab, shape.hidden), WEIGHT_STD, seed, "qwen/final/Wlm"),
    }


def qwen_hidden(shape: QwenShape, batch: int, seed: int) -> np.ndarray:
    """Block input x ~ N(0,1) as bf16 values, widened to the fp32 residual."""
    return bf16_bits_as_f32(normal_bf16((batch, shape.hidden), 1.0, seed, "qwen/x"))


def qwen_attn(shape: QwenShape, batch: int, seed: int, layer: int) -> np.ndarray:
    """Seeded N(0,1) stand-in for block `layer`'s attention output, bf16 bits."""
    return normal_bf16((batch, shape.hidden), 1.0, seed, f"qwen/L{layer}/attn")


@dataclass(frozen=True)
class MlpShape:
    width: int = 768
    blocks: int = 72
    eps: float = 1e-5

    def block_bytes(self) -> int:
        w = self.width
        return 2 * (w * w + 3 * w)


def mlp_block_weights(shape: MlpShape, seed: int, block: int) -> dict:
    w = shape.width
    t = f"mlp/B{block}/"
    return {
        "gamma": uniform_bf16((w,), 0.5, 1.5, seed, t + "gamma"),
        "beta": normal_bf16((w,), WEIGHT_STD, seed, t + "beta"),
        "W": normal_bf16((w, w), WEIGHT_STD, seed, t + "W"),
        "b": normal_bf16((w,), WEIGHT_STD, seed, t + "b"),
    }


def mlp_input(shape: MlpShape, batch: int, seed: int) -> np.ndarray:
    return normal_bf16((batch, shape.width), 1.0, seed, "mlp/x")
