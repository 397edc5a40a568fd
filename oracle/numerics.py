"""Scalar building blocks of the oracle, fp64.  TEST INFRASTRUCTURE ONLY.

The pages fix none of these formulas (they name a transformer target and a
transformer drafter); each is the textbook definition, with the constants of
the stated readings: RMSNorm eps 1e-6 with unit gain, rotate-half RoPE,
softmax scale 1/sqrt(head_dim), SwiGLU feed-forward.
"""
from __future__ import annotations

import numpy as np


class Precision:
    """Where values are rounded to bfloat16.

    ``exact``   : fp64 everywhere (weights are used as stored).
    ``bf16emu`` : round-to-nearest-even to bf16 at every point where the GPU
                  path stores bf16: normalised GEMM inputs, Q/K/V, the
                  attention output, the SwiGLU product, the fused injection
                  feature F, and the hidden-state capture.  The residual
                  stream and all logits stay unrounded.
    """

    def __init__(self, mode: str = "exact"):
        if mode not in ("exact", "bf16emu"):
            raise ValueError(mode)
        self.mode = mode

    def store(self, x: np.ndarray) -> np.ndarray:
        return round_bf16(x) if self.mode == "bf16emu" else np.asarray(x, dtype=np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps the sign, the 8-bit exponent and 7 fraction bits.  In the
    fp64 encoding that means keeping the top 7 of the 52 fraction bits, so
    the low 45 bits are rounded away.  (Values below the bf16 normal range
    are not treated specially; they do not occur here.)
    """
    a = np.array(x, dtype=np.float64, copy=True)
    bits = a.view(np.uint64)
    drop = np.uint64(45)
    lsb = (bits >> drop) & np.uint64(1)
    half_minus_one = np.uint64((1 << 44) - 1)
    bits += half_minus_one + lsb
    bits &= ~np.uint64((1 << 45) - 1)
    return a


def rmsnorm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gain, dtype=np.float64)


def rope_angles(positions: np.ndarray, head_dim: int, theta: float):
    """cos/sin tables [n, head_dim/2]: angle(p, i) = p * theta^(-2i/head_dim)."""
    half = head_dim // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE on x[n, heads, head_dim]: the pair (i, i + hd/2) is
    rotated by the angle of frequency i at the row's position."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    cos, sin = rope_angles(positions, hd, theta)
    cos = cos[:, None, :]
    sin = sin[:, None, :]
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * cos - hi * sin, hi * cos + lo * sin], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = W x for every row x of ``x``; W is [out, in].

    One matrix-vector product per row, so a row's result never depends on
    how many rows are processed together (row independence: the verify pass
    and the one-token decode produce bitwise the same numbers for the same
    row).
    """
    w = np.asarray(w, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    return np.stack([w @ xi for xi in x]) if len(x) else np.zeros((0, w.shape[0]))


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Softmax attention of one query row over a list of keys.

    q [H, hd]; k, v [n, H_kv, hd].  Query head h reads KV head
    h // (H / H_kv) (grouped-query attention).  Scale 1/sqrt(hd).
    """
    n_heads, hd = q.shape
    group = n_heads // k.shape[1]
    out = np.empty((n_heads, hd), dtype=np.float64)
    scale = 1.0 / np.sqrt(hd)
    for h in range(n_heads):
        kh = k[:, h // group, :]
        vh = v[:, h // group, :]
        s = (kh @ q[h]) * scale
        s = s - np.max(s)
        p = np.exp(s)
        p = p / np.sum(p)
        out[h] = p @ vh
    return out


def argmax_lowest(logits: np.ndarray) -> int:
    """Index of the maximum; ties go to the lowest index."""
    return int(np.argmax(logits))


def top2_margin(logits: np.ndarray) -> float:
    """Gap between the largest and the second largest value."""
    if logits.shape[-1] < 2:
        return float("inf")
    part = np.partition(logits, -2)
    return float(part[-1] - part[-2])


def log_softmax(logits: np.ndarray) -> np.ndarray:
    l = np.asarray(logits, dtype=np.float64)
    m = np.max(l)
    return l - (m + np.log(np.sum(np.exp(l - m))))
