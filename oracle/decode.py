"""Greedy AR decoding, the greedy accept rule and the DFlash loop, fp64.
TEST INFRASTRUCTURE ONLY.

* Greedy AR decoding (glossary "From autoregressive bottlenecks to
  speculative acceleration"; report "DFlash benchmark results" runs at
  temperature 0): x_P = argmax of the prefill logits at row P-1, then
  x_{t+1} = argmax logits(x_<=t).  Ties go to the lowest token id.
* The DFlash step (glossary "DFlash: architecture and workflow"): the anchor
  is the token at the decoding frontier; the drafter fills B-1 masked
  positions in one pass; the target computes its logits at every block
  position in one pass and a draft token passes when it equals the target's
  argmax; the longest contiguous accepted prefix is emitted, and the
  target's own argmax at the first mismatch is emitted after it (the page's
  fall-back to ordinary decoding, taken from the same verify pass); the
  cycle repeats from the new frontier.
* Speedup model (glossary "Mathematical view of acceptance and speedup"):
  S = C_AR / (C_DF / E[L]).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, List, Optional, Sequence

import numpy as np

from .models import KVCache, Weights, causal_visible, draft_block_logits, inject_kv, target_forward
from .numerics import Precision, argmax_lowest


def accept_longest_prefix(draft: Sequence[int], target_argmax: Sequence[int]):
    """Greedy acceptance of one block.

    ``draft`` = d_1..d_{B-1} (tokens proposed for block slots 1..B-1) and
    ``target_argmax`` = y_0..y_{B-1} (y_j = target argmax at slot j, i.e. its
    prediction for slot j+1).  Draft token d_i passes when d_i == y_{i-1};
    a = the length of the longest passing prefix; the bonus token is y_a.

    Returns (a, emitted) with emitted = [d_1..d_a, y_a] (a + 1 tokens).
    """
    a = 0
    while a < len(draft) and draft[a] == target_argmax[a]:
        a += 1
    emitted = [int(t) for t in draft[:a]] + [int(target_argmax[a])]
    return a, emitted


def speedup_model(c_ar: float, c_df: float, expected_len: float) -> float:
    """S = C_AR / (C_DF / E[L]): cost per accepted token vs one AR token."""
    return c_ar / (c_df / expected_len)


@dataclass
class StepRecord:
    ctx_len: int            # committed length P before the step (anchor at P)
    block: List[int]        # [anchor, d_1 .. d_{B-1}]
    target_argmax: List[int]
    accept_len: int         # a
    emitted: List[int]      # d_1..d_a, y_a
    draft_margins: List[float] = field(default_factory=list)
    target_margins: List[float] = field(default_factory=list)


class Sequence1:
    """State of one sequence: target cache, draft cache, committed length."""

    def __init__(self, w: Weights, shape, prec: Precision, max_len: int):
        s = shape
        self.w, self.shape, self.prec = w, shape, prec
        self.cache = KVCache(s.n_layers, max_len, s.n_kv_heads, s.head_dim)
        self.dcache = KVCache(s.n_draft_layers, max_len, s.n_kv_heads, s.head_dim)
        self.length = 0

    def prefill(self, prompt: Sequence[int], inject: bool = True):
        """Causal target pass over the prompt; returns (logits, capture)."""
        p = len(prompt)
        logits, cap = target_forward(self.w, self.shape, self.prec, self.cache, prompt,
                                     np.arange(p), np.arange(p), causal_visible(0, p))
        if inject:
            inject_kv(self.w, self.shape, self.prec, self.dcache, cap, np.arange(p))
        self.length = p
        return logits, cap

    def verify(self, block: Sequence[int]):
        """Target pass over a linear block at positions P..P+q-1 (causal over
        the cache and inside the block).  K/V are written tentatively."""
        q = len(block)
        pos = self.length + np.arange(q)
        return target_forward(self.w, self.shape, self.prec, self.cache, block, pos, pos,
                              causal_visible(self.length, q))

    def draft(self, anchor: int, block_size: int) -> np.ndarray:
        return draft_block_logits(self.w, self.shape, self.prec, self.dcache, anchor,
                                  self.length, block_size)

    def commit_linear(self, capture: np.ndarray, accept_len: int) -> None:
        """Keep the K/V of slots P..P+a (rollback of the rest is by length
        only) and inject the captured rows 0..a into the draft cache."""
        rows = accept_len + 1
        inject_kv(self.w, self.shape, self.prec, self.dcache, capture[:rows],
                  self.length + np.arange(rows))
        self.length += rows


def greedy_ar(w: Weights, shape, prec: Precision, prompt: Sequence[int], n_new: int,
              max_len: Optional[int] = None) -> List[int]:
    """Plain greedy autoregressive decoding of the target: n_new tokens."""
    seq = Sequence1(w, shape, prec, max_len or (len(prompt) + n_new + 1))
    logits, _ = seq.prefill(prompt, inject=False)
    out = [argmax_lowest(logits[-1])]
    while len(out) < n_new:
        logits, _ = seq.verify([out[-1]])
        seq.length += 1
        out.append(argmax_lowest(logits[0]))
    return out


DraftOverride = Callable[[int, int, List[int]], List[int]]


def dflash_generate(w: Weights, shape, prec: Precision, prompt: Sequence[int], n_new: int,
                    block_size: int, draft_override: Optional[DraftOverride] = None,
                    max_len: Optional[int] = None):
    """The DFlash loop for one sequence; returns (tokens, step records).

    ``draft_override(step, ctx_len, drafted)`` may replace the drafted
    tokens (teacher forcing / adversarial tests); the drafter still runs.
    Generation stops after n_new tokens; the last step's excess is cut.
    """
    b = block_size
    seq = Sequence1(w, shape, prec, max_len or (len(prompt) + n_new + 2 * b + 1))
    logits, _ = seq.prefill(prompt, inject=True)
    anchor = argmax_lowest(logits[-1])
    out = [anchor]
    steps: List[StepRecord] = []
    while len(out) < n_new:
        drafted: List[int] = []
        if b > 1:
            dlog = seq.draft(anchor, b)
            drafted = [argmax_lowest(r) for r in dlog]
        if draft_override is not None:
            drafted = list(draft_override(len(steps), seq.length, drafted))
        block = [anchor] + drafted
        vlog, cap = seq.verify(block)
        y = [argmax_lowest(r) for r in vlog]
        a, emitted = accept_longest_prefix(drafted, y)
        steps.append(StepRecord(seq.length, block, y, a, emitted))
        seq.commit_linear(cap, a)
        out.extend(emitted)
        anchor = emitted[-1]
    return out[:n_new], steps
