"""Target transformer, block-diffusion drafter and KV injection, fp64.
TEST INFRASTRUCTURE ONLY.

What the pages fix, and the reading taken where they are silent:

* Target: an unchanged autoregressive LLM ("DFlash speculative decoding"
  glossary, "Practical meaning and deployment behaviour").  Read as a
  pre-RMSNorm decoder: per layer x += Wo·Attn(RoPE(Wq h), RoPE(Wk h), Wv h),
  h = RMSNorm(x); then x += Wdown·(SiLU(Wgate h) * Wup h), h = RMSNorm(x);
  final RMSNorm and an untied lm_head.
* Drafter conditioning on "hidden features from multiple layers of the
  target model" (ludicrous-speed story, DFlash paragraph): the residual
  stream after each selected target layer, concatenated in layer order.
* KV injection (Deep Research Report, "Key points"): the target features are
  fused by one linear projection F = W_fuse·h_cat and injected into the K/V
  projections of *every* draft layer (K = RoPE(Wk_l F), V = Wv_l F, each
  draft layer with its own Wk_l, Wv_l), stored in the draft KV cache at the
  context position of the row.
* Block draft (Deep Research Report, "Key points"; glossary "DFlash:
  architecture and workflow", stage 2): one forward pass over B positions,
  slot 0 = the anchor token's embedding, slots 1..B-1 = a mask embedding
  (the tutorial paragraph of the ludicrous-speed story appends a <MASK> id
  to the vocabulary; here its row is ``draft.mask_emb``).  Attention is
  bidirectional inside the block (report's MTP table; "Why DFlash beats
  EAGLE-3" item 3) and sees every injected context row.  Slot j >= 1
  predicts the token at position P + j through the shared target lm_head
  after the drafter's own final RMSNorm.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from .numerics import Precision, apply_rope, attend, linear, rmsnorm, silu


class KVCache:
    """Per-layer K/V rows indexed by cache slot: [layers, slots, H_kv, hd]."""

    def __init__(self, n_layers: int, n_slots: int, n_kv_heads: int, head_dim: int):
        self.k = np.zeros((n_layers, n_slots, n_kv_heads, head_dim), dtype=np.float64)
        self.v = np.zeros_like(self.k)

    def copy(self) -> "KVCache":
        c = KVCache.__new__(KVCache)
        c.k = self.k.copy()
        c.v = self.v.copy()
        return c


class Weights:
    """fp64 view of a name -> array mapping (converted on first use)."""

    def __init__(self, source):
        self.source = source
        self._cache: Dict[str, np.ndarray] = {}

    def __getitem__(self, name: str) -> np.ndarray:
        if name not in self._cache:
            self._cache[name] = np.asarray(self.source[name], dtype=np.float64)
        return self._cache[name]


def _layer(w: Weights, shape, prec: Precision, prefix: str, x: np.ndarray,
           positions: np.ndarray, attend_rows) -> np.ndarray:
    """One pre-RMSNorm decoder layer on rows x [M, d].

    ``attend_rows(q, k, v)`` receives this layer's roped Q [M,H,hd] and the
    rows' own roped K, V [M,H_kv,hd] and returns the attention output
    [M,H,hd]; it decides which keys each row sees.
    """
    m = x.shape[0]
    s = shape
    h = prec.store(rmsnorm(x, w[f"{prefix}.attn_norm"], s.rms_eps))
    q = linear(h, w[f"{prefix}.wq"]).reshape(m, s.n_heads, s.head_dim)
    k = linear(h, w[f"{prefix}.wk"]).reshape(m, s.n_kv_heads, s.head_dim)
    v = linear(h, w[f"{prefix}.wv"]).reshape(m, s.n_kv_heads, s.head_dim)
    q = prec.store(apply_rope(q, positions, s.rope_theta))
    k = prec.store(apply_rope(k, positions, s.rope_theta))
    v = prec.store(v)
    o = prec.store(attend_rows(q, k, v).reshape(m, s.q_dim))
    x = x + linear(o, w[f"{prefix}.wo"])
    h = prec.store(rmsnorm(x, w[f"{prefix}.ffn_norm"], s.rms_eps))
    act = prec.store(silu(linear(h, w[f"{prefix}.w_gate"])) * linear(h, w[f"{prefix}.w_up"]))
    return x + linear(act, w[f"{prefix}.w_down"])


def target_forward(w: Weights, shape, prec: Precision, cache: KVCache,
                   tokens: Sequence[int], positions: Sequence[int], slots: Sequence[int],
                   visible: List[np.ndarray], want_logits: bool = True):
    """Target pass over rows (one sequence).

    Row i holds token ``tokens[i]`` at position ``positions[i]``; its K/V are
    written to cache slot ``slots[i]`` of every layer before any row attends;
    it then attends to the cache slots ``visible[i]`` (which include its own).

    Returns (logits [M, V] or None, capture [M, n_inject, d]); the capture is
    the residual stream after each injected layer, in layer order.
    """
    s = shape
    tokens = np.asarray(tokens, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    slots = np.asarray(slots, dtype=np.int64)
    x = w["tok_emb"][tokens]
    caps = []
    for l in range(s.n_layers):
        def attend_rows(q, k, v, l=l):
            cache.k[l, slots] = k
            cache.v[l, slots] = v
            return np.stack([attend(q[i], cache.k[l, visible[i]], cache.v[l, visible[i]])
                             for i in range(len(tokens))])
        x = _layer(w, s, prec, f"layers.{l}", x, positions, attend_rows)
        if l in s.inject_layers:
            caps.append(prec.store(x))
    capture = np.stack(caps, axis=1)
    logits = None
    if want_logits:
        hn = prec.store(rmsnorm(x, w["final_norm"], s.rms_eps))
        logits = linear(hn, w["lm_head"])
    return logits, capture


def causal_visible(ctx_len: int, n_rows: int) -> List[np.ndarray]:
    """Row j (at slot ctx_len + j) sees slots 0 .. ctx_len + j."""
    return [np.arange(ctx_len + j + 1) for j in range(n_rows)]


def inject_kv(w: Weights, shape, prec: Precision, dcache: KVCache,
              capture_rows: np.ndarray, positions: Sequence[int]) -> None:
    """KV injection: F = W_fuse · concat(h_l1..h_lk); for every draft layer l,
    K = RoPE(Wk_l F) and V = Wv_l F are written to the draft cache at the
    rows' context positions."""
    s = shape
    positions = np.asarray(positions, dtype=np.int64)
    r = capture_rows.shape[0]
    if r == 0:
        return
    hcat = capture_rows.reshape(r, s.n_inject * s.d_model)
    f = prec.store(linear(hcat, w["draft.fuse"]))
    for l in range(s.n_draft_layers):
        k = linear(f, w[f"draft.layers.{l}.wk"]).reshape(r, s.n_kv_heads, s.head_dim)
        v = linear(f, w[f"draft.layers.{l}.wv"]).reshape(r, s.n_kv_heads, s.head_dim)
        dcache.k[l, positions] = prec.store(apply_rope(k, positions, s.rope_theta))
        dcache.v[l, positions] = prec.store(v)


def draft_block_logits(w: Weights, shape, prec: Precision, dcache: KVCache,
                       anchor: int, ctx_len: int, block_size: int,
                       pos0: Optional[int] = None) -> np.ndarray:
    """One block-diffusion draft pass; returns logits [B-1, V] of slots 1..B-1.

    Slot j sits at position ctx_len + j (the frontier: the anchor is the
    token at position P = ctx_len).  ``pos0`` overrides the position of
    slot 0 (the tests use it to move the block against its context).  Every
    slot attends to the injected context rows 0..ctx_len-1 and to all B
    in-block rows (no mask).  The in-block K/V are scratch and never enter
    the draft cache.
    """
    s = shape
    b = block_size
    positions = (ctx_len if pos0 is None else pos0) + np.arange(b)
    x = np.stack([w["tok_emb"][anchor]] + [w["draft.mask_emb"]] * (b - 1))
    for l in range(s.n_draft_layers):
        def attend_rows(q, k, v, l=l):
            kk = np.concatenate([dcache.k[l, :ctx_len], k])
            vv = np.concatenate([dcache.v[l, :ctx_len], v])
            return np.stack([attend(q[i], kk, vv) for i in range(b)])
        x = _layer(w, s, prec, f"draft.layers.{l}", x, positions, attend_rows)
    hn = prec.store(rmsnorm(x[1:], w["draft.final_norm"], s.rms_eps))
    return linear(hn, w["lm_head"])
