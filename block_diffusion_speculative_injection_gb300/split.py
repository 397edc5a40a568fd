"""Drafter and verifier in separate contexts, on separate devices.

The glossary "DFlash speculative decoding" (section "Practical meaning and
deployment behaviour") notes that the diffusion drafter and the verifier can
sit on distinct devices, so that drafting overlaps verification.  Here one
library context (the verifier side) runs the target passes and the commits,
another (the drafter side) the draft passes and the KV injection; per step
and sequence group:

  verifier  verify the group's block, commit it (greedy): accept lengths,
            next anchors, emitted tokens, and the committed rows' captured
            hidden states (dflash_injection_rows)
  drafter   inject those rows into its draft cache (dflash_inject_kv, the
            explicit-row form), move its committed lengths on by accept + 1
            (dflash_advance_lengths), draft the group's next block
  verifier  receives that block

Data crosses devices as device-to-device copies (NVLink peer copies within a
node; nothing goes through the host).  With the sequences in two groups the
host enqueues verify(A), hand-off(A), draft(A), verify(B), ...: on two
devices the drafter drafts A while the verifier verifies B.  Every step of
the path runs in the library's kernels; this module only routes buffers.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import capi
from .engine import DFlashEngine, device_view


@dataclass
class Handoff:
    """A commit's injection rows on the verifier's device (views of its
    context's buffers: valid until its next pass)."""
    hidden: torch.Tensor   # [rows][n_inject][d_model]
    row_seq: torch.Tensor  # [rows] int32, < 0: row not committed
    row_pos: torch.Tensor  # [rows] int32
    counts: torch.Tensor   # [batch] int32 tokens committed per sequence

    def detach_to(self, device) -> "Handoff":
        """The rows on `device`.  They are first copied on the verifier's own
        stream, so that its next pass (which rewrites the buffers viewed
        here) is ordered after the copy; the copy then crosses devices."""
        own = [self.hidden.clone(), self.row_seq.clone(), self.row_pos.clone(), self.counts.clone()]
        return Handoff(*[t.to(device=device, non_blocking=True) for t in own])


class VerifierSide:
    """The target passes and commits of one context."""

    def __init__(self, eng: DFlashEngine):
        self.eng = eng
        self.device = torch.device(eng.device)

    def _handoff(self, counts: torch.Tensor) -> Handoff:
        s = self.eng.shape
        h, rs, rp, n = capi.dflash_injection_rows(self.eng.ctx)
        tdt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
        hidden = device_view(h, (self.eng.max_rows, s.n_inject, s.d_model), tdt)[:n]
        return Handoff(hidden, device_view(rs, (self.eng.max_rows,), torch.int32)[:n],
                       device_view(rp, (self.eng.max_rows,), torch.int32)[:n], counts)

    def reset(self, seq: int) -> None:
        with torch.cuda.device(self.device):
            capi.dflash_reset_seq(self.eng.ctx, seq)

    def prefill_chunk(self, sid: torch.Tensor, toks: torch.Tensor):
        """One prompt chunk of one sequence: (next anchor [1], hand-off)."""
        e = self.eng
        with torch.cuda.device(self.device):
            q = toks.numel()
            capi.dflash_verify(e.ctx, 1, sid, toks, q, None, capi.DFLASH_VERIFY_LAST_ONLY, e.argmax)
            capi.dflash_accept_commit(e.ctx, 1, sid, None, e.argmax, None, capi.DFLASH_ACCEPT_ALL,
                                      e.accept_len, e.next_anchor, e.emitted)
            counts = torch.full((1,), q, dtype=torch.int32, device=self.device)
            return e.next_anchor[:1].clone(), self._handoff(counts)

    def verify_block(self, sid: torch.Tensor, block: torch.Tensor):
        """Verify [b][B] drafted blocks and commit greedily: (accept_len,
        next_anchor, emitted [b][B], argmax [b][B], hand-off)."""
        e = self.eng
        with torch.cuda.device(self.device):
            b, B = block.shape
            argmax = e.argmax[: b * B]
            capi.dflash_verify(e.ctx, b, sid, block, B, None, 0, argmax)
            acc, nxt, emitted = e.accept_len[:b], e.next_anchor[:b], e.emitted[: b * B]
            capi.dflash_accept_commit(e.ctx, b, sid, block, argmax, None, capi.DFLASH_ACCEPT_GREEDY,
                                      acc, nxt, emitted)
            counts = acc + 1
            return (acc.clone(), nxt.clone(), emitted.view(b, B).clone(), argmax.view(b, B).clone(),
                    self._handoff(counts))


    def verify_tree(self, sid: torch.Tensor, tree: dict):
        """Verify drafted trees (the dtree_buffers arrays, already on this
        device) with the ancestor-only mask and commit the accepted paths:
        (accept_len, next_anchor, emitted [b][n], argmax [b][n], hand-off)."""
        e = self.eng
        with torch.cuda.device(self.device):
            b, n, m = sid.numel(), e.max_tree_nodes, e.tree_mem
            w = e.tree.anc_words
            for k in ("tok", "parent", "depth"):
                m[k][: b * n].copy_(tree[k].reshape(-1))
            m["anc"][: b * n * w].copy_(tree["anc"].reshape(-1))
            m["n_nodes"][:b].copy_(tree["n_nodes"].reshape(-1))
            argmax = e.argmax[: b * n]
            capi.dtree_verify(e.ctx, b, sid, e.tree, argmax, e.margin[: b * n], None)
            acc, nxt, emitted = e.accept_len[:b], e.next_anchor[:b], e.emitted[: b * n]
            capi.dflash_accept_commit(e.ctx, b, sid, None, argmax, e.tree, capi.DFLASH_ACCEPT_GREEDY,
                                      acc, nxt, emitted)
            counts = acc + 1
            return (acc.clone(), nxt.clone(), emitted.view(b, n).clone(), argmax.view(b, n).clone(),
                    self._handoff(counts))


class DrafterSide:
    """The draft passes and the KV injection of one context."""

    def __init__(self, eng: DFlashEngine):
        self.eng = eng
        self.device = torch.device(eng.device)

    def reset(self, seq: int) -> None:
        with torch.cuda.device(self.device):
            capi.dflash_reset_seq(self.eng.ctx, seq)

    def absorb(self, sid: torch.Tensor, h: Handoff) -> None:
        """Inject a commit's rows (already on this device) and move the
        committed lengths on by its counts."""
        with torch.cuda.device(self.device):
            n = h.hidden.shape[0]
            if n:
                capi.dflash_inject_kv(self.eng.ctx, n, h.row_seq, h.row_pos, h.hidden)
            capi.dflash_advance_lengths(self.eng.ctx, sid.numel(), sid, h.counts)

    def draft(self, sid: torch.Tensor, anchors: torch.Tensor,
              want_logits: bool = False):
        """The block [b][B] drafted from the anchors (and the draft logits)."""
        e = self.eng
        with torch.cuda.device(self.device):
            b, B = sid.numel(), e.B
            block = torch.empty(b * B, dtype=torch.int32, device=self.device)
            dlog = None
            if want_logits:
                dlog = torch.empty(b * max(B - 1, 1) * e.shape.vocab, dtype=torch.float32,
                                   device=self.device)
            capi.dflash_draft_block(e.ctx, b, sid, anchors, block, 0, None, None, dlog)
            block = block.view(b, B)
            if want_logits:
                return block, dlog.view(b, max(B - 1, 1), -1)
            return block

    def draft_tree(self, sid: torch.Tensor, anchors: torch.Tensor, topk: int, budget: int) -> dict:
        """The draft pass with per-slot top-k, then the best-first tree
        (dtree_build): copies of the dtree_buffers arrays of the batch."""
        e = self.eng
        with torch.cuda.device(self.device):
            b, B, n, m = sid.numel(), e.B, e.max_tree_nodes, e.tree_mem
            ids = m["topk_ids"][: b * (B - 1) * topk]
            lps = m["topk_logp"][: b * (B - 1) * topk]
            capi.dflash_draft_block(e.ctx, b, sid, anchors, e.block[: b * B], topk, ids, lps, None)
            capi.dtree_build(e.ctx, b, anchors, ids, lps, topk, budget, e.tree)
            w = e.tree.anc_words
            return {"tok": m["tok"][: b * n].view(b, n).clone(),
                    "parent": m["parent"][: b * n].view(b, n).clone(),
                    "depth": m["depth"][: b * n].view(b, n).clone(),
                    "anc": m["anc"][: b * n * w].view(b, n, w).clone(),
                    "n_nodes": m["n_nodes"][:b].clone()}


@dataclass
class SplitStep:
    """One step of one sequence group, on the verifier's device."""
    block: torch.Tensor        # [b][B] drafted tokens (anchor first)
    argmax: torch.Tensor       # [b][B] target argmax
    accept_len: torch.Tensor   # [b]
    next_anchor: torch.Tensor  # [b]
    emitted: torch.Tensor      # [b][B], -1 past the emitted tokens


class SplitDFlash:
    """DFlash greedy decoding with the drafter on `draft_device` and the
    verifier on `target_device` (the same device is allowed: two contexts on
    one GPU, as the tests run it).  Both contexts hold the same seeded
    weights.  Sequence slot s is slot s in both contexts."""

    def __init__(self, shape, block_size: int, max_batch: int, max_ctx: int,
                 draft_device="cuda:0", target_device="cuda:0", max_rows: Optional[int] = None,
                 seed: int = 0, max_tree_nodes: int = 0):
        self.B = block_size
        mk = dict(max_rows=max_rows, seed=seed, max_tree_nodes=max_tree_nodes)
        self.verifier = VerifierSide(DFlashEngine(shape, block_size, max_batch, max_ctx,
                                                  device=str(target_device), **mk))
        self.drafter = DrafterSide(DFlashEngine(shape, block_size, max_batch, max_ctx,
                                                device=str(draft_device), **mk))
        self.vdev, self.ddev = self.verifier.device, self.drafter.device

    def close(self) -> None:
        self.verifier.eng.close()
        self.drafter.eng.close()

    def prefill(self, prompts: Sequence[np.ndarray]) -> torch.Tensor:
        """Target prefill of slots 0..len-1 on the verifier, every chunk's
        captured rows injected on the drafter; returns the first anchors
        (on the verifier's device)."""
        anchors = torch.empty(len(prompts), dtype=torch.int32, device=self.vdev)
        chunk = self.verifier.eng.max_rows
        for s, p in enumerate(prompts):
            self.verifier.reset(s)
            self.drafter.reset(s)
            sid_v = torch.tensor([s], dtype=torch.int32, device=self.vdev)
            sid_d = torch.tensor([s], dtype=torch.int32, device=self.ddev)
            toks = torch.from_numpy(np.asarray(p, dtype=np.int32)).to(self.vdev)
            for c0 in range(0, len(p), chunk):
                a, h = self.verifier.prefill_chunk(sid_v, toks[c0:c0 + chunk].contiguous())
                self.drafter.absorb(sid_d, h.detach_to(self.ddev))
                anchors[s:s + 1].copy_(a)
        return anchors

    def step(self, seq_ids: torch.Tensor, anchors: torch.Tensor,
             draft_override: Optional[torch.Tensor] = None) -> SplitStep:
        """One DFlash step of one group: draft (drafter), verify + commit
        (verifier), hand-off (drafter).  draft_override [b][B-1] (tests)
        replaces the drafted tokens before the verify pass."""
        sid_d = seq_ids.to(self.ddev)
        block = self.drafter.draft(sid_d, anchors.to(self.ddev))
        return self._verify(seq_ids, sid_d, block, draft_override)

    def _verify(self, seq_ids, sid_d, block, draft_override=None) -> SplitStep:
        block = block.to(self.vdev)
        if draft_override is not None:
            block[:, 1:].copy_(draft_override)
        acc, nxt, emitted, argmax, h = self.verifier.verify_block(seq_ids.to(self.vdev), block)
        self.drafter.absorb(sid_d, h.detach_to(self.ddev))
        return SplitStep(block, argmax, acc, nxt, emitted)

    def tree_step(self, seq_ids: torch.Tensor, anchors: torch.Tensor, topk: int, budget: int,
                  tree_override: Optional[dict] = None) -> SplitStep:
        """One DDTree step of one group: draft + tree build (drafter), the
        tree arrays to the verifier, ancestor-masked verify + commit of the
        accepted path (verifier), hand-off (drafter).  tree_override (tests)
        replaces the built tree's arrays before the verify pass.  The
        returned block is the tree's tokens [b][max_nodes]."""
        sid_d = seq_ids.to(self.ddev)
        tree = self.drafter.draft_tree(sid_d, anchors.to(self.ddev), topk, budget)
        tree = {k: (tree_override or tree)[k].to(self.vdev, non_blocking=True) for k in tree}
        acc, nxt, emitted, argmax, h = self.verifier.verify_tree(seq_ids.to(self.vdev), tree)
        self.drafter.absorb(sid_d, h.detach_to(self.ddev))
        return SplitStep(tree["tok"], argmax, acc, nxt, emitted)

    def generate(self, prompts: Sequence[np.ndarray], n_new: int, groups: int = 1) -> List[List[int]]:
        """Greedy generation of n_new tokens per prompt.  With groups > 1 the
        sequences go in that many groups and the host enqueues each group's
        verify right after the previous group's draft, so that on two devices
        the drafter works on one group while the verifier works on another."""
        b = len(prompts)
        anchors = self.prefill(prompts)
        out = [[int(x)] for x in anchors.tolist()]
        parts = [g for g in np.array_split(np.arange(b), groups) if len(g)]
        sids = [torch.tensor(g, dtype=torch.int32, device=self.vdev) for g in parts]
        sids_d = [s.to(self.ddev) for s in sids]
        # every group's first block, then verify(g) -> draft(g) in turn
        blocks = [self.drafter.draft(sd, anchors[s.long()].to(self.ddev))
                  for s, sd in zip(sids, sids_d)]
        while min(len(o) for o in out) < n_new:
            emitted = []
            for gi, (s, sd) in enumerate(zip(sids, sids_d)):
                r = self._verify(s, sd, blocks[gi])
                blocks[gi] = self.drafter.draft(sd, r.next_anchor.to(self.ddev))
                emitted.append(r.emitted)
            # one read-back per round, after every group's work is enqueued
            for gi, em in enumerate(emitted):
                for k, q in enumerate(parts[gi].tolist()):
                    out[q] += [t for t in em[k].tolist() if t >= 0]
        return [o[:n_new] for o in out]
