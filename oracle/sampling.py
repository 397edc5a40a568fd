"""Temperature-1 drafting and acceptance (speculative rejection sampling), fp64.
TEST INFRASTRUCTURE ONLY: nothing on the product path imports this module.

The pages run DFlash at temperature 1 as well as greedily (report "DFlash
benchmark results": an average 4.03x at temperature 1), say that the
drafter fills the masked block positions with *sampled* tokens and that a
draft token passes when it matches the target's argmax "or sits within an
acceptance criterion" (glossary "DFlash: architecture and workflow", stages
2 and 3), and call the result lossless.  They do not state the criterion.
The plainest reading that keeps the output distributed exactly as sampling
the target at temperature 1 is the standard speculative rejection rule:

* drafting: block slot j (1 <= j < B) draws d_j from p_j = softmax of the
  drafter's logits at slot j (the slots are drafted in one pass, so p_j does
  not depend on the other draft tokens);
* verification: q_i = softmax of the target's logits at block row i, the
  distribution of the token at position P + i + 1 given the prefix;
* for j = 1, 2, ...: d_j is accepted when u_j * p_j(d_j) < q_{j-1}(d_j)
  (accept with probability min(1, q/p)); at the first rejection the step
  emits one token drawn from the residual r = max(0, q_{j-1} - p_j),
  normalised, and stops; when all B - 1 are accepted, it emits one token
  drawn from q_{B-1} (the bonus);
* every draw is by inverse CDF over token ids in increasing order: the
  token is the smallest x with sum_{y <= x} w(y) > u * sum_y w(y).

Random numbers are inputs (one uniform per draft slot for drafting, one per
slot for the accept tests, one per step for the final draw), so a GPU path
given the same uniforms has exactly one correct answer wherever no
comparison is within rounding of a tie.
"""
from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np


def softmax(logits: np.ndarray) -> np.ndarray:
    """softmax(x) at temperature 1 along the last axis, fp64."""
    x = np.asarray(logits, dtype=np.float64)
    z = np.exp(x - x.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def inverse_cdf(weights: np.ndarray, u: float) -> int:
    """Smallest token x with sum_{y<=x} w(y) > u * sum(w), summed in id order.

    Weights are non-negative and not all zero; u is in [0, 1).
    """
    w = np.asarray(weights, dtype=np.float64)
    target = float(u) * w.sum()
    acc = 0.0
    for x, wx in enumerate(w):
        acc += wx
        if acc > target:
            return x
    # u * total rounds to total: the last token with positive weight
    return int(np.nonzero(w > 0)[0][-1])


def sample_row(logits: np.ndarray, u: float) -> int:
    """One draw from softmax(logits) by inverse CDF."""
    return inverse_cdf(softmax(logits), u)


def draft_tokens(draft_logits: np.ndarray, u_draft: Sequence[float]) -> np.ndarray:
    """d_j ~ p_j for slots 1..B-1 (slot 0 of the result is left 0)."""
    B = draft_logits.shape[0]
    out = np.zeros(B, dtype=np.int64)
    for j in range(1, B):
        out[j] = sample_row(draft_logits[j], u_draft[j])
    return out


def spec_accept(draft_logits: np.ndarray, target_logits: np.ndarray, tokens: Sequence[int],
                u_accept: Sequence[float], u_resample: float) -> Tuple[int, int]:
    """One step of the rule above for one sequence.

    draft_logits [B, V] (row j is slot j's drafter logits; row 0 unused),
    target_logits [B, V] (row i predicts position P + i + 1), tokens [B]
    (tokens[0] = the anchor, tokens[j] = d_j), u_accept [B] (entry j tests
    d_j; entry 0 unused), u_resample the uniform of the final draw.
    Returns (a, emitted): a accepted draft tokens, then the emitted token.
    """
    B = target_logits.shape[0]
    q = softmax(target_logits)
    p = softmax(draft_logits)
    for j in range(1, B):
        d = int(tokens[j])
        if not (u_accept[j] * p[j, d] < q[j - 1, d]):
            resid = np.maximum(q[j - 1] - p[j], 0.0)
            return j - 1, inverse_cdf(resid, u_resample)
    return B - 1, inverse_cdf(q[B - 1], u_resample)
