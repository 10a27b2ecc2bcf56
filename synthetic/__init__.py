"""Seeded synthetic inputs for the headwise-chunked attention layer.

This module is shared by both sides of every parity check: the fp64 oracle
and the CUDA library read the same bf16 bit patterns produced here.  It holds
none of the method's arithmetic -- only random draws, the float32 -> bfloat16
storage conversion (round to nearest even) and the named layer shapes.

Shapes follow the workloads the UPipe pages train on ("Untied Ulysses",
results section: Llama3-8B and Qwen3-32B); the distributions are
X ~ N(0, 1), W_qkv and W_o ~ N(0, 1/d_model), dY ~ N(0, 1), seed 0.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import numpy as np


@dataclass(frozen=True)
class LayerShape:
    """One attention layer: sequence S, model width d_model, H query heads,
    G key/value heads, head width d_head, U heads per stage, C virtual ranks."""
    S: int
    d_model: int
    H: int
    G: int
    d_head: int
    U: int
    C: int

    def replace(self, **kw) -> "LayerShape":
        d = asdict(self)
        d.update(kw)
        return LayerShape(**d)

    @property
    def qkv_cols(self) -> int:
        return (self.H + 2 * self.G) * self.d_head


# Named workloads.  The first is small enough for the oracle to finish in
# seconds; the others are the Llama3-8B and Qwen3-32B attention-layer shapes.
SHAPES = {
    "tiny": LayerShape(S=1024, d_model=512, H=8, G=2, d_head=64, U=2, C=2),
    "llama3_8b_32k": LayerShape(S=32768, d_model=4096, H=32, G=8, d_head=128, U=8, C=8),
    "qwen3_32b_128k": LayerShape(S=131072, d_model=5120, H=64, G=8, d_head=128, U=8, C=8),
    "llama3_8b_256k_usweep": LayerShape(S=262144, d_model=4096, H=32, G=8, d_head=128, U=8, C=8),
    "llama3_8b_512k_gqa": LayerShape(S=524288, d_model=4096, H=32, G=8, d_head=128, U=8, C=8),
    # Llama3-8B widths at a length the fp64 oracle still finishes in full.
    "llama3_8b_4k": LayerShape(S=4096, d_model=4096, H=32, G=8, d_head=128, U=8, C=8),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


def layer_inputs(shape: LayerShape, seed: int = 0) -> dict:
    """bf16 bit patterns (uint16 arrays) for one layer fwd+bwd:

    X [S, d_model], W_qkv [d_model, (H+2G)*d_head] with columns
    [Q heads 0..H-1 | K heads 0..G-1 | V heads 0..G-1], W_o [H*d_head, d_model],
    dY [S, d_model].  Drawn in that order from numpy's default_rng(seed).
    """
    rng = np.random.default_rng(seed)
    w_std = 1.0 / np.sqrt(shape.d_model)
    X = _normal_bf16(rng, (shape.S, shape.d_model), 1.0)
    W_qkv = _normal_bf16(rng, (shape.d_model, shape.qkv_cols), w_std)
    W_o = _normal_bf16(rng, (shape.H * shape.d_head, shape.d_model), w_std)
    dY = _normal_bf16(rng, (shape.S, shape.d_model), 1.0)
    return {"X": X, "W_qkv": W_qkv, "W_o": W_o, "dY": dY}


def normal_bf16(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """A single seeded N(0, std^2) bf16 tensor (unit-test operands)."""
    return _normal_bf16(np.random.default_rng(seed), shape, std)
