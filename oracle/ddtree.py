"""DDTree: draft tree from per-position distributions, best-first heap,
ancestor-only verification mask, tree accept walk.  TEST INFRASTRUCTURE ONLY.

Source: "LLMs hit ludicrous speed ..." (joindrip.ai), DDTree paragraph: a
draft tree holding several continuations is built from the drafter's
per-position distributions with a best-first heap, and all its nodes are
verified in one target pass under an attention mask that lets a node see
only its ancestors.

Readings (the paragraph gives no formulas):
* p_j = softmax of the draft logits at block slot j (temperature 1); the
  top k = 8 tokens per slot by logit, ties to the lower id; log p = logit -
  logsumexp.
* A node at depth j (1..B-1) takes rank r of slot j's top-k; its score is
  the fp32 sum of log p along its path, added in depth order.
* Heap order: score descending, then depth ascending, then the rank vector
  lexicographically ascending.  Popping a node pushes its first child
  (rank 0 one level deeper, while depth < B-1) and its next sibling
  (rank + 1 < k).  Scores never increase along either edge, so the popped
  set is the global top-N of all prefixes under that order.
* Budget N counts drafted nodes; the root (the anchor) is added, so the
  verify pass has N + 1 rows.
* Node n sits at position P + depth(n) and at tentative cache slot P + n; it
  sees the context 0..P-1, its ancestors and itself.  Its logits then equal
  those of a causal pass over its path, which keeps the tree lossless.
* Accept walk: from the root, step to the child whose token equals the
  current node's target argmax; stop when no child matches; the bonus is
  the argmax at the stop node.  The j-th accepted node's K/V move from slot
  P + s_j to slot P + j (all sources are read before any write).
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass
from typing import List, Sequence

import numpy as np

from .decode import Sequence1
from .models import inject_kv, target_forward
from .numerics import argmax_lowest, log_softmax


def topk_logprobs(logits: np.ndarray, k: int):
    """Top-k ids of one slot (logit descending, ties to the lower id) and
    their log-probabilities (fp32)."""
    l = np.asarray(logits, dtype=np.float64)
    ids = np.arange(l.shape[0])
    order = np.lexsort((ids, -l))[:k]
    lp = log_softmax(l)[order]
    return order.astype(np.int32), lp.astype(np.float32)


@dataclass
class DraftTree:
    tok: List[int]
    parent: List[int]
    depth: List[int]
    rank: List[int]
    score: List[float]
    ancestors: List[int]  # bitset (python int): bit m set when m is an ancestor-or-self

    @property
    def n_nodes(self) -> int:
        return len(self.tok)

    def children(self, n: int) -> List[int]:
        return [c for c in range(self.n_nodes) if self.parent[c] == n]


def order_key(score: np.float32, ranks: Sequence[int]):
    """Heap priority (smaller pops first): score desc, depth asc, ranks asc."""
    return (-float(score), len(ranks), tuple(ranks))


def build_tree(anchor: int, topk_ids: np.ndarray, topk_logp: np.ndarray, budget: int) -> DraftTree:
    """Best-first heap over prefixes; pops ``budget`` nodes after the root.

    topk_ids / topk_logp: [B-1, k]; row j-1 belongs to block slot j.
    """
    depth_max, k = topk_ids.shape
    lp = np.asarray(topk_logp, dtype=np.float32)
    tree = DraftTree([int(anchor)], [-1], [0], [0], [0.0], [1])
    index_of = {(): 0}
    score_of = {(): np.float32(0.0)}
    heap = []

    def push(ranks):
        parent_score = score_of[ranks[:-1]]
        sc = np.float32(parent_score + lp[len(ranks) - 1, ranks[-1]])
        heapq.heappush(heap, (order_key(sc, ranks), ranks, sc))

    if depth_max >= 1 and k >= 1 and budget > 0:
        push((0,))
    while heap and tree.n_nodes - 1 < budget:
        _, ranks, sc = heapq.heappop(heap)
        par = index_of[ranks[:-1]]
        n = tree.n_nodes
        index_of[ranks] = n
        score_of[ranks] = sc
        tree.tok.append(int(topk_ids[len(ranks) - 1, ranks[-1]]))
        tree.parent.append(par)
        tree.depth.append(len(ranks))
        tree.rank.append(ranks[-1])
        tree.score.append(float(sc))
        tree.ancestors.append(tree.ancestors[par] | (1 << n))
        if len(ranks) < depth_max:
            push(ranks + (0,))
        if ranks[-1] + 1 < k:
            push(ranks[:-1] + (ranks[-1] + 1,))
    return tree


def ancestor_slots(tree: DraftTree, n: int) -> List[int]:
    return [m for m in range(tree.n_nodes) if (tree.ancestors[n] >> m) & 1]


def tree_visible(tree: DraftTree, ctx_len: int) -> List[np.ndarray]:
    return [np.concatenate([np.arange(ctx_len), ctx_len + np.array(ancestor_slots(tree, n))])
            for n in range(tree.n_nodes)]


def tree_accept(tree: DraftTree, node_argmax: Sequence[int]):
    """Walk from the root along children whose token equals the argmax.

    Returns (a, path, emitted): path = accepted node ids starting at the
    root; emitted = tokens of path[1:] then the bonus argmax."""
    path = [0]
    cur = 0
    while True:
        nxt = [c for c in tree.children(cur) if tree.tok[c] == node_argmax[cur]]
        if not nxt:
            break
        cur = nxt[0]
        path.append(cur)
    emitted = [tree.tok[p] for p in path[1:]] + [int(node_argmax[cur])]
    return len(path) - 1, path, emitted


def tree_verify(seq: Sequence1, tree: DraftTree):
    """One target pass over every node of the tree."""
    n = tree.n_nodes
    pos = seq.length + np.asarray(tree.depth)
    slots = seq.length + np.arange(n)
    return target_forward(seq.w, seq.shape, seq.prec, seq.cache, tree.tok, pos, slots,
                          tree_visible(tree, seq.length))


def tree_commit(seq: Sequence1, capture: np.ndarray, path: List[int]) -> None:
    """Compact the accepted path's K/V (all target layers) to slots P..P+a,
    inject its captured rows, and advance the length."""
    p = seq.length
    src = p + np.asarray(path)
    dst = p + np.arange(len(path))
    k = seq.cache.k[:, src].copy()
    v = seq.cache.v[:, src].copy()
    seq.cache.k[:, dst] = k
    seq.cache.v[:, dst] = v
    inject_kv(seq.w, seq.shape, seq.prec, seq.dcache, capture[np.asarray(path)], dst)
    seq.length += len(path)


def ddtree_generate(w, shape, prec, prompt: Sequence[int], n_new: int, block_size: int,
                    topk: int, budget: int, max_len=None):
    """DDTree decoding of one sequence; returns (tokens, per-step (tree, a, emitted))."""
    b = block_size
    seq = Sequence1(w, shape, prec, max_len or (len(prompt) + n_new + budget + b + 2))
    logits, _ = seq.prefill(prompt, inject=True)
    anchor = argmax_lowest(logits[-1])
    out = [anchor]
    steps = []
    while len(out) < n_new:
        dlog = seq.draft(anchor, b)
        ids = np.zeros((b - 1, topk), dtype=np.int32)
        lps = np.zeros((b - 1, topk), dtype=np.float32)
        for j in range(b - 1):
            ids[j], lps[j] = topk_logprobs(dlog[j], topk)
        tree = build_tree(anchor, ids, lps, budget)
        vlog, cap = tree_verify(seq, tree)
        y = [argmax_lowest(r) for r in vlog]
        a, path, emitted = tree_accept(tree, y)
        steps.append((tree, a, emitted, y))
        tree_commit(seq, cap, path)
        out.extend(emitted)
        anchor = emitted[-1]
    return out[:n_new], steps
