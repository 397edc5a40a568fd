"""Seeded synthetic workloads shared by the CPU oracle and the GPU harness.

This module holds only shapes and seeded random inputs: model shapes, the
five workloads, random weights, random prompts, random context lengths and
random attention operands.  It contains none of the method's arithmetic
(no norm, no attention, no projection, no acceptance rule), so both the
oracle and the GPU path may import it without sharing any computation.

Recipe (every value is reproducible from the seeds below):

* Weights.  A pool of 2**24 values is drawn i.i.d. N(0, std) from numpy's
  PCG64 seeded with ``seed`` and stored in the workload's storage type
  (float32, or bfloat16 by round-to-nearest-even).  Row ``r`` of a weight
  tensor of shape ``[R, K]`` is the circular window
  ``pool[(a*r + c) mod 2**24 : ... + K]`` where ``a`` (odd) and ``c`` come
  from PCG64 seeded with ``(seed, tensor index)``.  Distinct rows therefore
  start at distinct pool offsets.  RMSNorm gains are 1.
* Prompts.  Uniform token ids from PCG64 seeded with ``(prompt_seed, seq)``.
* Context lengths of the ragged batch.  Uniform integers from PCG64 seeded
  with ``(len_seed,)``.
* Attention operands.  Same pool construction with std 1 and seed 3.

Synthetic stand-ins: the pages measure on public benchmarks (GSM8K,
MATH-500, HumanEval, MT-Bench, Qasper) with trained models; none of those
datasets or weights is used or reproduced here.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np

POOL_LOG2 = 24
POOL_SIZE = 1 << POOL_LOG2


@dataclass(frozen=True)
class ModelShape:
    """Shape of a target model plus its block-diffusion drafter."""

    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_theta: float
    n_draft_layers: int
    inject_layers: Tuple[int, ...]
    rms_eps: float = 1e-6
    dtype: str = "bf16"  # storage type of weights, KV caches, capture: "f32" | "bf16"
    weight_std: float = 0.02

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def n_inject(self) -> int:
        return len(self.inject_layers)


def evenly_spaced_layers(n_layers: int, k: int) -> Tuple[int, ...]:
    """k target-layer indices spread from the first to the last layer,
    rounded half up: round(i * (L-1)/(k-1))."""
    if k == 1:
        return (n_layers - 1,)
    return tuple(int(np.floor(i * (n_layers - 1) / (k - 1) + 0.5)) for i in range(k))


TINY = ModelShape(
    name="tiny", n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64,
    ffn_dim=768, vocab=1024, rope_theta=1e4, n_draft_layers=1,
    inject_layers=(0, 1), dtype="f32")

QWEN3_8B = ModelShape(
    name="qwen3_8b", n_layers=36, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
    ffn_dim=12288, vocab=151936, rope_theta=1e6, n_draft_layers=5,
    inject_layers=(0, 9, 18, 26, 35), dtype="bf16")

LLAMA31_8B = ModelShape(
    name="llama31_8b", n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
    ffn_dim=14336, vocab=128256, rope_theta=5e5, n_draft_layers=5,
    inject_layers=(0, 8, 16, 23, 31), dtype="bf16")

# Small bf16 shapes with the production head geometry (GQA 4:1, hd 128).  They
# drive the bf16 kernels end to end at sizes the oracle finishes in seconds.
MINI_BF16 = ModelShape(
    name="mini_bf16", n_layers=3, d_model=1024, n_heads=8, n_kv_heads=2, head_dim=128,
    ffn_dim=2048, vocab=4096, rope_theta=1e6, n_draft_layers=2,
    inject_layers=(0, 2), dtype="bf16")

MINI_BF16_WIDE = ModelShape(
    name="mini_bf16_wide", n_layers=2, d_model=1024, n_heads=8, n_kv_heads=2, head_dim=128,
    ffn_dim=1536, vocab=5000, rope_theta=5e5, n_draft_layers=1,
    inject_layers=(1,), dtype="bf16")

# Two Qwen3-8B-shaped target layers and one draft layer: the same GEMM,
# attention and lm_head launch shapes as the full model at ~2 GB of weights
# (used to profile single kernels).
QWEN3_8B_SLICE = dataclasses.replace(QWEN3_8B, name="qwen3_8b_slice", n_layers=2,
                                     n_draft_layers=1, inject_layers=(0, 1))

SHAPES: Dict[str, ModelShape] = {s.name: s for s in (TINY, QWEN3_8B, LLAMA31_8B, MINI_BF16,
                                                     MINI_BF16_WIDE, QWEN3_8B_SLICE)}


@dataclass(frozen=True)
class Workload:
    """One benchmark or parity configuration."""

    name: str
    shape: ModelShape
    block_size: int
    batch: int
    prompt_len: Tuple[int, int]  # inclusive range; (P, P) for a fixed length
    new_tokens: int
    tree_budget: int = 0  # 0: linear block; N > 0: DDTree with N drafted nodes (+ root)
    topk: int = 0
    seed: int = 0
    prompt_seed: int = 1
    len_seed: int = 2


WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in (
        Workload("tiny_f32_e2e", TINY, 16, 1, (64, 64), 64),
        Workload("qwen3_8b_b1", QWEN3_8B, 16, 1, (2048, 2048), 256),
        Workload("qwen3_8b_b32", QWEN3_8B, 16, 32, (512, 4096), 128),
        Workload("llama31_8b_ddtree_b4", LLAMA31_8B, 16, 4, (4096, 4096), 64,
                 tree_budget=64, topk=8),
        Workload("mini_bf16_e2e", MINI_BF16, 16, 3, (40, 160), 48),
        Workload("mini_bf16_ddtree", MINI_BF16, 16, 2, (96, 130), 40, tree_budget=64, topk=8),
        Workload("qwen3_8b_slice_b1", QWEN3_8B_SLICE, 16, 1, (2048, 2048), 256),
        Workload("qwen3_8b_slice_b32", QWEN3_8B_SLICE, 16, 32, (512, 1024), 128),
    )
}

# Op-level block-draft attention grid (q-len 16, 32 q heads / 8 KV heads, hd 128).
ATTN_OP_CTX = (512, 2048, 8192, 16384)
ATTN_OP_BATCH = (1, 8, 32)
ATTN_OP_HEADS = (32, 8, 128)  # (q heads, kv heads, head dim)


# ----------------------------------------------------------------------------
# bf16 storage helpers (round-to-nearest-even of float32 values)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# value pools
# ----------------------------------------------------------------------------

_POOL_CACHE: Dict[Tuple[int, float, str], np.ndarray] = {}


def value_pool(seed: int, std: float, dtype: str) -> np.ndarray:
    """2**24 i.i.d. N(0, std) values as float32 (bf16-representable if dtype=='bf16')."""
    key = (seed, std, dtype)
    if key not in _POOL_CACHE:
        rng = np.random.Generator(np.random.PCG64(seed))
        p = (rng.standard_normal(POOL_SIZE) * std).astype(np.float32)
        if dtype == "bf16":
            p = bf16_bits_to_f32(f32_to_bf16_bits(p))
        _POOL_CACHE[key] = p
    return _POOL_CACHE[key]


def row_offsets(seed: int, index: int, n_rows: int) -> np.ndarray:
    """Pool start offsets of the rows of tensor number ``index``."""
    rng = np.random.Generator(np.random.PCG64([seed, index]))
    a = int(rng.integers(0, POOL_SIZE // 2)) * 2 + 1
    c = int(rng.integers(0, POOL_SIZE))
    r = np.arange(n_rows, dtype=np.int64)
    return (r * a + c) % POOL_SIZE


def pool_rows(pool: np.ndarray, offsets: np.ndarray, width: int) -> np.ndarray:
    """Rows ``pool[off : off+width]`` (circular), as a new float32 array."""
    ext = np.concatenate([pool, pool[:width]])
    win = np.lib.stride_tricks.sliding_window_view(ext, width)
    return np.ascontiguousarray(win[offsets])


# ----------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------

def layer_tensor_specs(prefix: str, s: ModelShape) -> List[Tuple[str, Tuple[int, ...]]]:
    d = s.d_model
    return [
        (f"{prefix}.attn_norm", (d,)),
        (f"{prefix}.wq", (s.q_dim, d)),
        (f"{prefix}.wk", (s.kv_dim, d)),
        (f"{prefix}.wv", (s.kv_dim, d)),
        (f"{prefix}.wo", (d, s.q_dim)),
        (f"{prefix}.ffn_norm", (d,)),
        (f"{prefix}.w_gate", (s.ffn_dim, d)),
        (f"{prefix}.w_up", (s.ffn_dim, d)),
        (f"{prefix}.w_down", (d, s.ffn_dim)),
    ]


def weight_specs(s: ModelShape) -> List[Tuple[str, Tuple[int, ...]]]:
    """Every named tensor of target + drafter, in a fixed order (the order
    fixes each tensor's generator index)."""
    specs: List[Tuple[str, Tuple[int, ...]]] = [("tok_emb", (s.vocab, s.d_model))]
    for l in range(s.n_layers):
        specs += layer_tensor_specs(f"layers.{l}", s)
    specs += [("final_norm", (s.d_model,)), ("lm_head", (s.vocab, s.d_model))]
    specs += [("draft.fuse", (s.d_model, s.n_inject * s.d_model)),
              ("draft.mask_emb", (s.d_model,))]
    for l in range(s.n_draft_layers):
        specs += layer_tensor_specs(f"draft.layers.{l}", s)
    specs += [("draft.final_norm", (s.d_model,))]
    return specs


def is_norm(name: str) -> bool:
    return name.endswith("norm")


class SyntheticWeights:
    """Lazily generated named weights of one model shape (float32 values)."""

    def __init__(self, shape: ModelShape, seed: int = 0):
        self.shape = shape
        self.seed = seed
        self.specs = dict(weight_specs(shape))
        self.index = {n: i for i, (n, _) in enumerate(weight_specs(shape))}
        self._cache: Dict[str, np.ndarray] = {}

    def names(self) -> List[str]:
        return list(self.specs)

    def pool(self) -> np.ndarray:
        return value_pool(self.seed, self.shape.weight_std, self.shape.dtype)

    def offsets(self, name: str) -> np.ndarray:
        shp = self.specs[name]
        rows = shp[0] if len(shp) == 2 else 1
        return row_offsets(self.seed, self.index[name], rows)

    def generate(self, name: str) -> np.ndarray:
        shp = self.specs[name]
        if is_norm(name):
            return np.ones(shp, dtype=np.float32)
        width = shp[-1]
        rows = pool_rows(self.pool(), self.offsets(name), width)
        return rows.reshape(shp)

    def __getitem__(self, name: str) -> np.ndarray:
        if name not in self._cache:
            self._cache[name] = self.generate(name)
        return self._cache[name]

    def drop(self, name: str) -> None:
        self._cache.pop(name, None)

    def with_override(self, overrides: Dict[str, np.ndarray]) -> "SyntheticWeights":
        w = SyntheticWeights(self.shape, self.seed)
        w._cache = dict(self._cache)
        w._cache.update({k: np.asarray(v, dtype=np.float32) for k, v in overrides.items()})
        return w


# ----------------------------------------------------------------------------
# prompts, lengths, attention operands
# ----------------------------------------------------------------------------

def prompt_lengths(w: Workload) -> List[int]:
    lo, hi = w.prompt_len
    if lo == hi:
        return [lo] * w.batch
    rng = np.random.Generator(np.random.PCG64([w.len_seed]))
    return [int(x) for x in rng.integers(lo, hi + 1, size=w.batch)]


def prompt_tokens(w: Workload, seq: int, length: Optional[int] = None) -> np.ndarray:
    if length is None:
        length = prompt_lengths(w)[seq]
    rng = np.random.Generator(np.random.PCG64([w.prompt_seed, seq]))
    return rng.integers(0, w.shape.vocab, size=length).astype(np.int32)


def prompts(w: Workload) -> List[np.ndarray]:
    return [prompt_tokens(w, s, n) for s, n in enumerate(prompt_lengths(w))]


ATTN_SEED = 3


def attn_operand_rows(which: str, n_rows: int, width: int = 128, seed: int = ATTN_SEED,
                      rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Rows of an N(0,1) bf16 attention operand ('q', 'k', 'v', 'kb', 'vb').

    ``rows`` selects a subset of row indices (for sampled checks); default all.
    """
    idx = {"q": 0, "k": 1, "v": 2, "kb": 3, "vb": 4}[which]
    off = row_offsets(seed, idx, n_rows)
    if rows is not None:
        off = off[np.asarray(rows, dtype=np.int64)]
    return pool_rows(value_pool(seed, 1.0, "bf16"), off, width)


SAMPLING_SEED = 4


def sampling_inputs(batch: int, block: int, vocab: int, seed: int = SAMPLING_SEED,
                    spread: float = 3.0, agreement: float = 0.8):
    """Seeded fp32 logits and uniforms for the temperature-1 acceptance op.

    A shared N(0, spread) score per (sequence, slot, token) plus independent
    noise for the drafter and the target (the target's row i is paired with
    the drafter's slot i + 1, the position both predict), so the two
    distributions agree to a tunable degree.  Returns (draft_logits,
    target_logits [batch, block, vocab] float32, u_draft, u_accept
    [batch, block], u_resample [batch]).
    """
    rng = np.random.Generator(np.random.PCG64([seed, batch, block, vocab]))
    base = rng.normal(0.0, spread, (batch, block + 1, vocab))
    noise = np.sqrt(max(0.0, 1.0 - agreement ** 2)) * spread
    draft = agreement * base[:, :block] + rng.normal(0.0, noise, (batch, block, vocab))
    target = agreement * base[:, 1:] + rng.normal(0.0, noise, (batch, block, vocab))
    u_draft = rng.random((batch, block))
    u_accept = rng.random((batch, block))
    u_res = rng.random(batch)
    return (draft.astype(np.float32), target.astype(np.float32), u_draft.astype(np.float32),
            u_accept.astype(np.float32), u_res.astype(np.float32))


def step_uniforms(step: int, batch: int, block: int, seed: int = SAMPLING_SEED):
    """Seeded uniforms of one temperature-1 step: (u_draft [batch, block-1],
    u_accept [batch, block], u_resample [batch]), float32 in [0, 1)."""
    rng = np.random.Generator(np.random.PCG64([seed, 7, step]))
    u_draft = rng.random((batch, max(block - 1, 0))).astype(np.float32)
    u_accept = rng.random((batch, block)).astype(np.float32)
    u_res = rng.random(batch).astype(np.float32)
    return u_draft, u_accept, u_res


def replace(w: Workload, **kw) -> Workload:
    return dataclasses.replace(w, **kw)
