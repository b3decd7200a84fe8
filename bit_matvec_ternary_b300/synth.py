"""Seeded synthetic inputs for the ternary projection linears.

This module draws random numbers and tabulates model shapes.  It holds none
of the method's arithmetic (no packing, no quantisation, no dot products), so
both the CUDA path and the CPU oracle may take their inputs from it.

Everything is numpy ``default_rng(seed)`` (PCG64) on the host.

Sources for the statistics and shapes (Neutrino-1 pages):
  * code statistics 62.63 % zero / 18.68 % plus / 18.69 % minus for the 8B and
    62.26 / 18.87 / 18.86 for the 0.6B -- "Neutrino-1: quantization is a
    training decision", section "Sparsity is learned, not imposed";
  * zero share by depth: attention flat near 62 %, the FFN down/gate spike in
    the earliest layers, densest tensor the first down projection (60.59 %) --
    same section, figure 2; "Neutrino-1" wiki page, "What is actually new";
  * 8B geometry (36 layers, hidden 4096, 32 q / 8 kv heads of 128, SwiGLU
    12288, vocabulary 151,936, untied) -- "Neutrino-1 8B" model page,
    "Architecture"; 0.6B geometry (28 layers, hidden 1024, 16 q / 8 kv heads,
    tied) -- fermionresearch.com/models, "Neutrino-1 0.6B".
"""
from __future__ import annotations

import dataclasses
import numpy as np

# Projection order inside one decoder layer; the per-matrix seed uses it.
PROJ_ORDER = ("q", "k", "v", "o", "gate", "up", "down")


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Geometry of a Qwen3-shaped decoder as far as its linears need it."""
    name: str
    layers: int
    hidden: int
    q_heads: int
    kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    tied_embeddings: bool

    def linear_shapes(self) -> dict[str, tuple[int, int]]:
        """(M, K) = (output rows, input width) of each projection."""
        q = self.q_heads * self.head_dim
        kv = self.kv_heads * self.head_dim
        h, f = self.hidden, self.ffn
        return {"q": (q, h), "k": (kv, h), "v": (kv, h), "o": (h, q),
                "gate": (f, h), "up": (f, h), "down": (h, f)}

    @property
    def linears(self) -> int:
        return self.layers * len(PROJ_ORDER)

    def ternary_weights_per_layer(self) -> int:
        return sum(m * k for m, k in self.linear_shapes().values())

    def ternary_weights(self) -> int:
        return self.layers * self.ternary_weights_per_layer()

    def embedding_params(self) -> int:
        return (1 if self.tied_embeddings else 2) * self.vocab * self.hidden

    def norm_params(self) -> int:
        # input and post-attention RMSNorm gains plus per-head q/k norms,
        # four tensors per layer, plus the final norm.
        per_layer = 2 * self.hidden + 2 * self.head_dim
        return self.layers * per_layer + self.hidden

    def total_params(self) -> int:
        return self.ternary_weights() + self.embedding_params() + self.norm_params()

    def kv_bytes_per_token_fp16(self) -> int:
        return self.layers * 2 * self.kv_heads * self.head_dim * 2


NEUTRINO_8B = ModelShape("8B", layers=36, hidden=4096, q_heads=32, kv_heads=8,
                         head_dim=128, ffn=12288, vocab=151936,
                         tied_embeddings=False)
NEUTRINO_06B = ModelShape("0.6B", layers=28, hidden=1024, q_heads=16, kv_heads=8,
                          head_dim=128, ffn=3072, vocab=151936,
                          tied_embeddings=True)

P0_DEFAULT = 0.626      # overall zero share, rounded (8B: 62.63 %)
P0_ATTENTION = 0.62     # flat attention band 61.84-63.51 %


def zero_fraction_8b(layer: int, proj: str) -> float:
    """Zero share used for the synthetic 8B stack (layers counted from 0).

    The pages number the FFN spike two ways (from 1 in the blog figure, from 0
    on the model page); read from 0: down 60.59 % at layer 0, gate and down
    near 71 % in layers 1-3, down 72.47 % at layer 2, gate 70.48 % at layer 3,
    everything else at the overall share.
    """
    if proj in ("q", "k", "v", "o"):
        return P0_ATTENTION
    if proj == "down" and layer == 0:
        return 0.6059
    if proj in ("gate", "down") and 1 <= layer <= 3:
        if proj == "down" and layer == 2:
            return 0.7247
        if proj == "gate" and layer == 3:
            return 0.7048
        return 0.71
    return P0_DEFAULT


def matrix_seed(base: int, layer: int, proj: str) -> int:
    return base + 1000 * layer + PROJ_ORDER.index(proj)


def ternary(M: int, K: int, p0: float, seed: int) -> np.ndarray:
    """int8 W[M, K] with P(0) = p0 and the two signs equally likely.

    One 16-bit draw per weight: values below p0 * 2^16 give 0, the rest take
    their sign from the draw's low bit.
    """
    rng = np.random.default_rng(seed)
    r = rng.integers(0, 1 << 16, size=(M, K), dtype=np.uint16)
    thr = np.uint16(min(int(round(p0 * 65536.0)), 65535))
    w = np.where(r & 1, np.int8(-1), np.int8(1)).astype(np.int8)
    w[r < thr] = 0
    return w


def scales(M: int, seed: int, lo: float = 0.005, hi: float = 0.05) -> np.ndarray:
    """fp32 per-row scale, U[lo, hi]."""
    rng = np.random.default_rng(seed + 7_000_003)
    return rng.uniform(lo, hi, size=M).astype(np.float32)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float data to bf16 (nearest, ties to even); returns uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(N: int, K: int, seed: int, outlier_frac: float = 0.0,
                outlier_gain: float = 20.0, unit_rms: bool = False) -> np.ndarray:
    """bf16 X[N, K] as uint16 bits: N(0,1), optionally with outlier channels.

    Outliers: round(outlier_frac * K) channel indices, drawn once per call and
    shared by all N tokens, multiplied by ``outlier_gain`` before rounding.
    ``unit_rms`` divides each token by its own RMS (fp64) before rounding.
    """
    rng = np.random.default_rng(seed + 9_000_011)
    x = rng.standard_normal(size=(N, K))
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * K))
        idx = rng.choice(K, size=n_out, replace=False)
        x[:, idx] *= outlier_gain
    if unit_rms and K > 0:
        rms = np.sqrt(np.mean(x * x, axis=1, keepdims=True))
        x = x / np.where(rms > 0, rms, 1.0)
    return to_bf16_bits(x.astype(np.float32))


def stack_layout(shape: ModelShape) -> list[tuple[int, str, int, int]]:
    """[(layer, proj, M, K)] in the stack's execution order."""
    shp = shape.linear_shapes()
    return [(l, p, *shp[p]) for l in range(shape.layers) for p in PROJ_ORDER]


def zero_fraction(shape: ModelShape, layer: int, proj: str) -> float:
    if shape is NEUTRINO_8B:
        return zero_fraction_8b(layer, proj)
    return P0_DEFAULT
