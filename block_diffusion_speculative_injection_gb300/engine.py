"""Host harness over the C ABI: seeded weights on the device, the step loops.

The harness only moves arguments: it uploads the seeded synthetic weights
(the generator's value pool, gathered on the device into each named tensor),
allocates the caller-side buffers, and calls the C functions in the order
the pages give for one step (anchor -> block draft -> one-pass verify ->
longest-prefix accept -> KV injection), or the DDTree order (draft top-k ->
heap tree -> tree verify -> accept walk -> injection).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

import workloads as wl

from . import capi
from .adaptive import AdaptiveBlock


def config_for(shape: wl.ModelShape, block_size: int, max_batch: int, max_ctx: int,
               max_rows: int, max_tree_nodes: int = 0, kv_pages: int = 0) -> capi.Config:
    c = capi.Config()
    c.d_model = shape.d_model
    c.n_heads = shape.n_heads
    c.n_kv_heads = shape.n_kv_heads
    c.head_dim = shape.head_dim
    c.ffn_dim = shape.ffn_dim
    c.vocab = shape.vocab
    c.n_target_layers = shape.n_layers
    c.n_draft_layers = shape.n_draft_layers
    c.n_inject = shape.n_inject
    for i, l in enumerate(shape.inject_layers):
        c.inject_layers[i] = l
    c.rope_theta = shape.rope_theta
    c.rms_eps = shape.rms_eps
    c.block_size = block_size
    c.max_batch = max_batch
    c.max_ctx = max_ctx
    c.max_rows = max_rows
    c.max_tree_nodes = max_tree_nodes
    c.dtype = capi.DFLASH_BF16 if shape.dtype == "bf16" else capi.DFLASH_F32
    c.kv_pages = kv_pages
    return c


def device_weights(shape: wl.ModelShape, seed: int = 0, device: str = "cuda"):
    """Named weight tensors on the device, bytes identical to the generator's."""
    sw = wl.SyntheticWeights(shape, seed)
    tdt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    pool = torch.from_numpy(sw.pool()).to(device).to(tdt)
    widest = max(s[-1] for _, s in sw.specs.items())
    ext = torch.cat([pool, pool[:widest]])
    out = {}
    for name, shp in sw.specs.items():
        if wl.is_norm(name):
            out[name] = torch.ones(shp, dtype=tdt, device=device)
            continue
        width = shp[-1]
        off = torch.from_numpy(sw.offsets(name)).to(device)
        t = ext.unfold(0, width, 1)[off]
        out[name] = t.reshape(shp).contiguous()
    return out


@dataclass
class StepOut:
    block: torch.Tensor        # [b][B] (linear) or tree tokens
    argmax: torch.Tensor       # [b][q]
    accept_len: torch.Tensor   # [b]
    next_anchor: torch.Tensor  # [b]
    emitted: torch.Tensor      # [b][q]


class DFlashEngine:
    """One library context plus its weights and step buffers."""

    def __init__(self, shape: wl.ModelShape, block_size: int, max_batch: int, max_ctx: int,
                 max_rows: Optional[int] = None, max_tree_nodes: int = 0, seed: int = 0,
                 weights=None, device: str = "cuda", kv_pages: int = 0):
        capi.load()
        self.shape = shape
        self.B = block_size
        self.B_max = block_size
        self.max_batch = max_batch
        self.max_tree_nodes = max_tree_nodes
        self.device = device
        self.max_rows = max_rows or max(max_batch * max(block_size, max_tree_nodes), 1)
        self.cfg = config_for(shape, block_size, max_batch, max_ctx, self.max_rows, max_tree_nodes,
                              kv_pages)
        # paged KV cache: pages are mapped on demand from a shared pool; the
        # engine keeps a host upper bound of every slot's length for that
        self.paged = kv_pages > 0
        self.len_ub = [0] * max_batch
        self.dtype_code = self.cfg.dtype
        # the context belongs to this engine's device: create it there
        with torch.cuda.device(torch.device(device)):
            self.ctx = capi.dflash_create(self.cfg)
            self.weights = weights if weights is not None else device_weights(shape, seed, device)
            for name, t in self.weights.items():
                capi.dflash_set_weight(self.ctx, name, t, self.dtype_code)
        i32 = dict(dtype=torch.int32, device=device)
        mb = max_batch
        q = max(block_size, max_tree_nodes, 1)
        self.argmax = torch.empty(self.max_rows, **i32)
        self.block = torch.empty(mb * block_size, **i32)
        self.accept_len = torch.empty(mb, **i32)
        self.next_anchor = torch.empty(mb, **i32)
        self.emitted = torch.empty(max(self.max_rows, mb * q), **i32)
        self.margin = torch.empty(self.max_rows, dtype=torch.float32, device=device)
        if max_tree_nodes:
            self.tree_mem = dict(
                tok=torch.empty(mb * max_tree_nodes, **i32),
                parent=torch.empty(mb * max_tree_nodes, **i32),
                depth=torch.empty(mb * max_tree_nodes, **i32),
                anc=torch.empty(mb * max_tree_nodes * ((max_tree_nodes + 63) // 64),
                                dtype=torch.int64, device=device),
                n_nodes=torch.empty(mb, **i32),
                topk_ids=torch.empty(mb * (block_size - 1) * 16, **i32),
                topk_logp=torch.empty(mb * (block_size - 1) * 16, dtype=torch.float32, device=device),
            )
            self.tree = self.make_tree(max_tree_nodes)

    def make_tree(self, max_nodes: int) -> capi.DTree:
        m = self.tree_mem
        t = capi.DTree()
        t.tok, t.parent, t.depth = m["tok"].data_ptr(), m["parent"].data_ptr(), m["depth"].data_ptr()
        t.anc, t.n_nodes = m["anc"].data_ptr(), m["n_nodes"].data_ptr()
        t.max_nodes = max_nodes
        t.anc_words = (max_nodes + 63) // 64
        return t

    def close(self) -> None:
        if getattr(self, "ctx", None):
            capi.dflash_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_block_size(self, block: int) -> None:
        """Block size of the following steps (1..the configured block size)."""
        capi.dflash_set_block_size(self.ctx, block)
        self.B = block

    # -- sequence setup ----------------------------------------------------
    def seq_ids(self, batch: int) -> torch.Tensor:
        return torch.arange(batch, dtype=torch.int32, device=self.device)

    def lengths(self, batch: int) -> List[int]:
        """Committed length of the first ``batch`` sequence slots (syncs)."""
        v = device_view(capi.dflash_seq_lengths(self.ctx), (self.max_batch,), torch.int32)
        torch.cuda.synchronize()
        return v[:batch].tolist()

    def gen_counts(self) -> torch.Tensor:
        """Live device view of the per-slot emitted-token counters."""
        return device_view(capi.dflash_debug_view(self.ctx, "gen_count")[0], (self.max_batch,),
                           torch.int32)

    def page_table(self) -> torch.Tensor:
        """Live device view of the page table [max_batch][pages per slot]."""
        ptr, nbytes = capi.dflash_debug_view(self.ctx, "page_table")
        return device_view(ptr, (self.max_batch, nbytes // 4 // self.max_batch), torch.int32)

    def debug_view(self, name: str, layer: int = 0) -> torch.Tensor:
        """A view of an internal buffer (see dflash_debug_view).  The caches
        come back as [max_batch][n_kv_heads][max_ctx][head_dim], gathered
        through the page table (a copy; slots of unmapped pages read as page
        0's); every other buffer is a zero-copy view."""
        ptr, nbytes = capi.dflash_debug_view(self.ctx, name, layer)
        es = 2 if self.shape.dtype == "bf16" else 4
        t = device_view(ptr, (nbytes // es,), torch.bfloat16 if es == 2 else torch.float32)
        s = self.shape
        if name == "capture":
            return t.view(self.max_rows, s.n_inject, s.d_model)
        if name == "fused":
            return t.view(self.max_rows, s.d_model)
        pool = t.view(-1, s.n_kv_heads, capi.PAGE_SLOTS, s.head_dim)
        g = pool[self.page_table().long().clamp(min=0)]  # [slot][page][kv][row][hd]
        g = g.permute(0, 2, 1, 3, 4).reshape(self.max_batch, s.n_kv_heads, -1, s.head_dim)
        return g[:, :, : self.cfg.max_ctx]

    # -- paged KV cache ------------------------------------------------------
    def reserve(self, seq: int, n_slots: int) -> None:
        """Maps pages so that slot `seq` covers cache slots 0..n_slots-1."""
        capi.dflash_kv_reserve(self.ctx, seq, n_slots)

    def release(self, seq: int) -> None:
        """Returns slot `seq`'s pages to the pool (after its last pass)."""
        capi.dflash_kv_release(self.ctx, seq)
        self.len_ub[seq] = 0

    def free_pages(self) -> int:
        return capi.dflash_kv_free_pages(self.ctx)

    def reserve_ahead(self, seq_ids, steps: int, rows: int) -> None:
        """Paged mode: pages for `steps` more steps of at most self.B committed
        tokens each, plus one pass of `rows` rows (e.g. before capturing a
        step graph, whose replays map nothing)."""
        if not self.paged:
            return
        for s in _host_ids(seq_ids):
            self.reserve(s, min(self.len_ub[s] + steps * self.B_max + rows, self.cfg.max_ctx))

    def _pages_for_pass(self, seq_ids, rows: int, advance: int):
        """Paged mode: maps the pages a pass of `rows` rows per sequence touches
        and moves the length bound on by `advance` (the most a step commits)."""
        if not self.paged or torch.cuda.is_current_stream_capturing():
            return  # a captured step maps nothing: reserve_ahead before capturing
        for s in _host_ids(seq_ids):
            self.reserve(s, min(self.len_ub[s] + rows, self.cfg.max_ctx))
            self.len_ub[s] += advance

    def prefill(self, prompts: Sequence[np.ndarray], chunk: Optional[int] = None) -> torch.Tensor:
        """Target prefill of each sequence (slot = its index); returns the
        first generated token of every sequence (the first anchors)."""
        b = len(prompts)
        anchors = torch.empty(b, dtype=torch.int32, device=self.device)
        chunk = chunk or self.max_rows
        for s, p in enumerate(prompts):
            capi.dflash_reset_seq(self.ctx, s)
            if self.paged:
                self.reserve(s, len(p))
                self.len_ub[s] = len(p)
            sid = torch.tensor([s], dtype=torch.int32, device=self.device)
            toks = torch.from_numpy(np.asarray(p, dtype=np.int32)).to(self.device)
            for c0 in range(0, len(p), chunk):
                part = toks[c0:c0 + chunk].contiguous()
                q = part.numel()
                capi.dflash_verify(self.ctx, 1, sid, part, q, None, capi.DFLASH_VERIFY_LAST_ONLY,
                                   self.argmax)
                capi.dflash_accept_commit(self.ctx, 1, sid, None, self.argmax, None,
                                          capi.DFLASH_ACCEPT_ALL, self.accept_len, self.next_anchor,
                                          self.emitted)
                capi.dflash_inject_kv(self.ctx)
            anchors[s:s + 1].copy_(self.next_anchor[:1])
        return anchors

    # -- one DFlash step -----------------------------------------------------
    def step(self, seq_ids: torch.Tensor, anchors: torch.Tensor, want_logits: bool = False,
             draft_override: Optional[torch.Tensor] = None):
        b = seq_ids.numel()
        B = self.B
        self._pages_for_pass(seq_ids, B, B)
        block = self.block[: b * B]
        dlog = vlog = None
        if want_logits:
            dlog = torch.empty(b * max(B - 1, 1) * self.shape.vocab, dtype=torch.float32,
                               device=self.device)
            vlog = torch.empty(b * B * self.shape.vocab, dtype=torch.float32, device=self.device)
        capi.dflash_draft_block(self.ctx, b, seq_ids, anchors, block, 0, None, None, dlog)
        if draft_override is not None:
            block.view(b, B)[:, 1:].copy_(draft_override)
        argmax = self.argmax[: b * B]
        margin = self.margin[: b * B]
        capi.dflash_verify(self.ctx, b, seq_ids, block, B, None, 0, argmax, margin, vlog)
        emitted = self.emitted[: b * B]
        capi.dflash_accept_commit(self.ctx, b, seq_ids, block, argmax, None,
                                  capi.DFLASH_ACCEPT_GREEDY, self.accept_len[:b],
                                  self.next_anchor[:b], emitted)
        capi.dflash_inject_kv(self.ctx)
        out = StepOut(block.view(b, B), argmax.view(b, B), self.accept_len[:b],
                      self.next_anchor[:b], emitted.view(b, B))
        if want_logits:
            return out, dlog.view(b, max(B - 1, 1), -1), vlog.view(b, B, -1), margin.view(b, B)
        return out

    # -- one temperature-1 DFlash step -----------------------------------------
    def sample_step(self, seq_ids: torch.Tensor, anchors: torch.Tensor, u_draft: torch.Tensor,
                    u_accept: torch.Tensor, u_resample: torch.Tensor):
        """Draft block -> draft tokens drawn from the drafter's softmax (u_draft
        [b][B-1]) -> verify -> speculative rejection test (u_accept [b][B],
        u_resample [b]) -> commit the accepted prefix and the drawn token ->
        injection.  Every step runs in the library's kernels; this method only
        moves device buffers between the calls."""
        b = seq_ids.numel()
        B = self.B
        V = self.shape.vocab
        self._pages_for_pass(seq_ids, B, B)
        if not hasattr(self, "_samp"):
            rows = self.max_batch * max(self.B_max - 1, 1)
            self._samp = {
                "dlog": torch.empty(rows * V, dtype=torch.float32, device=self.device),
                "vlog": torch.empty(self.max_batch * self.B_max * V, dtype=torch.float32,
                                    device=self.device),
                "draws": torch.empty(rows, dtype=torch.int32, device=self.device),
                "ws_draw": torch.empty(max(capi.dflash_sample_workspace(rows, V), 256), dtype=torch.uint8,
                                       device=self.device),
                "ws_acc": torch.empty(capi.dflash_spec_accept_workspace(self.max_batch, self.B_max, V),
                                      dtype=torch.uint8, device=self.device),
            }
        m = self._samp
        block = self.block[: b * B]
        dlog = m["dlog"][: b * max(B - 1, 1) * V]
        capi.dflash_draft_block(self.ctx, b, seq_ids, anchors, block, 0, None, None, dlog)
        if B > 1:
            draws = m["draws"][: b * (B - 1)]
            capi.dflash_sample_rows(b * (B - 1), V, dlog, u_draft.contiguous(), draws, m["ws_draw"])
            block.view(b, B)[:, 1:].copy_(draws.view(b, B - 1))
        vlog = m["vlog"][: b * B * V]
        argmax = self.argmax[: b * B]
        capi.dflash_verify(self.ctx, b, seq_ids, block, B, None, 0, argmax, None, vlog)
        acc, nxt = self.accept_len[:b], self.next_anchor[:b]
        capi.dflash_spec_accept_sampled(b, B, V, dlog, vlog, block, u_accept.contiguous(),
                                        u_resample.contiguous(), acc, nxt, m["ws_acc"])
        emitted = self.emitted[: b * B]
        capi.dflash_accept_commit(self.ctx, b, seq_ids, block, block, None, capi.DFLASH_ACCEPT_GIVEN,
                                  acc, nxt, emitted)
        capi.dflash_inject_kv(self.ctx)
        return StepOut(block.view(b, B), argmax.view(b, B), acc, nxt, emitted.view(b, B))

    def ar_step(self, seq_ids: torch.Tensor, anchors: torch.Tensor):
        """Plain greedy decoding step: verify the anchor alone, commit it."""
        b = seq_ids.numel()
        self._pages_for_pass(seq_ids, 1, 1)
        toks = anchors.contiguous()
        argmax = self.argmax[:b]
        capi.dflash_verify(self.ctx, b, seq_ids, toks, 1, None, 0, argmax)
        capi.dflash_accept_commit(self.ctx, b, seq_ids, toks, argmax, None,
                                  capi.DFLASH_ACCEPT_GREEDY, self.accept_len[:b],
                                  self.next_anchor[:b], self.emitted[:b])
        capi.dflash_inject_kv(self.ctx)
        return self.next_anchor[:b]

    # -- one DDTree step -----------------------------------------------------
    def tree_step(self, seq_ids: torch.Tensor, anchors: torch.Tensor, topk: int, budget: int,
                  want_logits: bool = False, tree_override: Optional[dict] = None,
                  want_draft_logits: bool = False, before_commit=None):
        """One DDTree step.  tree_override (tests: teacher forcing) replaces the
        built tree with the caller's arrays before the verify pass: device
        tensors tok, parent, depth [b][max_nodes] int32, anc [b][max_nodes]
        [anc_words] int64 and n_nodes [b] int32, in the layout of
        dtree_buffers; the drafter and the heap builder still run.
        before_commit, if given, is called between the verify pass and the
        accept call (tests snapshot the caches there)."""
        b = seq_ids.numel()
        B = self.B
        m = self.tree_mem
        n = self.max_tree_nodes
        self._pages_for_pass(seq_ids, max(B, n), B)
        ids = m["topk_ids"][: b * (B - 1) * topk]
        lps = m["topk_logp"][: b * (B - 1) * topk]
        block = self.block[: b * B]
        dlog = None
        if want_draft_logits:
            dlog = torch.empty(b * (B - 1) * self.shape.vocab, dtype=torch.float32,
                               device=self.device)
        capi.dflash_draft_block(self.ctx, b, seq_ids, anchors, block, topk, ids, lps, dlog)
        capi.dtree_build(self.ctx, b, anchors, ids, lps, topk, budget, self.tree)
        if tree_override is not None:
            w = self.tree.anc_words
            m["tok"][: b * n].copy_(tree_override["tok"].reshape(-1))
            m["parent"][: b * n].copy_(tree_override["parent"].reshape(-1))
            m["depth"][: b * n].copy_(tree_override["depth"].reshape(-1))
            m["anc"][: b * n * w].copy_(tree_override["anc"].reshape(-1))
            m["n_nodes"][:b].copy_(tree_override["n_nodes"].reshape(-1))
        argmax = self.argmax[: b * n]
        margin = self.margin[: b * n]
        vlog = None
        if want_logits:
            vlog = torch.empty(b * n * self.shape.vocab, dtype=torch.float32, device=self.device)
        capi.dtree_verify(self.ctx, b, seq_ids, self.tree, argmax, margin, vlog)
        if before_commit is not None:
            before_commit()
        emitted = self.emitted[: b * n]
        capi.dflash_accept_commit(self.ctx, b, seq_ids, None, argmax, self.tree,
                                  capi.DFLASH_ACCEPT_GREEDY, self.accept_len[:b],
                                  self.next_anchor[:b], emitted)
        capi.dflash_inject_kv(self.ctx)
        res = dict(ids=ids.view(b, B - 1, topk), logp=lps.view(b, B - 1, topk),
                   tok=m["tok"][: b * n].view(b, n), parent=m["parent"][: b * n].view(b, n),
                   depth=m["depth"][: b * n].view(b, n), n_nodes=m["n_nodes"][:b],
                   anc=m["anc"][: b * n * self.tree.anc_words].view(b, n, -1),
                   argmax=argmax.view(b, n), margin=margin.view(b, n),
                   accept_len=self.accept_len[:b], next_anchor=self.next_anchor[:b],
                   emitted=emitted.view(b, n))
        if want_logits:
            res["logits"] = vlog.view(b, n, -1)
        if want_draft_logits:
            res["draft_logits"] = dlog.view(b, B - 1, -1)
        return res

    # -- whole generations ---------------------------------------------------
    def generate(self, prompts: Sequence[np.ndarray], n_new: int, mode: str = "dflash",
                 topk: int = 8, budget: int = 64, block_schedule=None) -> List[List[int]]:
        """Greedy generation.  mode "dflash" / "ddtree" / "ar"; "adaptive" is
        "dflash" with the block size of every step chosen by AdaptiveBlock
        from the previous steps' accepted lengths.  block_schedule (a list
        of block sizes, cycled) fixes the block size of each dflash step
        instead."""
        b = len(prompts)
        sid = self.seq_ids(b)
        anchors = self.prefill(prompts)
        outs = [[int(t)] for t in anchors.tolist()]
        policy = AdaptiveBlock(self.B_max) if mode == "adaptive" else None
        b_entry = self.B
        n_step = 0
        while min(len(o) for o in outs) < n_new:
            if mode in ("dflash", "adaptive") and (policy is not None or block_schedule is not None):
                nb = policy.next_block() if policy is not None else \
                    block_schedule[n_step % len(block_schedule)]
                if nb != self.B:
                    self.set_block_size(nb)
            n_step += 1
            if mode == "ar":
                anchors = self.ar_step(sid, anchors).clone()
                for s, t in enumerate(anchors.tolist()):
                    outs[s].append(int(t))
                continue
            if mode == "ddtree":
                r = self.tree_step(sid, anchors, topk, budget)
                em = r["emitted"]
            else:
                em = self.step(sid, anchors).emitted
                if policy is not None:
                    policy.update(self.accept_len[:b].tolist())
            anchors = self.next_anchor[:b].clone()
            for s, row in enumerate(em.tolist()):
                outs[s].extend(int(t) for t in row if t >= 0)
        if self.B != b_entry:
            self.set_block_size(b_entry)
        return [o[:n_new] for o in outs]


class _CudaArray:
    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 2, "strides": None}


def _host_ids(seq_ids) -> List[int]:
    return seq_ids.tolist() if isinstance(seq_ids, torch.Tensor) else list(seq_ids)


def device_view(ptr: int, shape, dtype: torch.dtype) -> torch.Tensor:
    """Zero-copy torch view of device memory owned by the library."""
    if dtype == torch.bfloat16:
        return torch.as_tensor(_CudaArray(ptr, shape, "<i2"), device="cuda").view(torch.bfloat16)
    code = {torch.int32: "<i4", torch.float32: "<f4", torch.int64: "<i8"}[dtype]
    return torch.as_tensor(_CudaArray(ptr, shape, code), device="cuda")


def device_operand(which: str, n_rows: int, width: int = 128, device: str = "cuda") -> torch.Tensor:
    """Seeded N(0,1) bf16 attention operand rows built on the device (same
    bytes as workloads.attn_operand_rows)."""
    pool = torch.from_numpy(wl.value_pool(wl.ATTN_SEED, 1.0, "bf16")).to(device).to(torch.bfloat16)
    ext = torch.cat([pool, pool[:width]])
    idx = {"q": 0, "k": 1, "v": 2, "kb": 3, "vb": 4}[which]
    off = torch.from_numpy(wl.row_offsets(wl.ATTN_SEED, idx, n_rows)).to(device)
    return ext.unfold(0, width, 1)[off].contiguous()


def capture_step_graph(eng: "DFlashEngine", seq_ids: torch.Tensor, tree: bool = False,
                       topk: int = 8, budget: int = 64) -> torch.cuda.CUDAGraph:
    """Captures one whole step (the C calls of draft, verify, accept and
    injection) into a CUDA graph.  The step reads its anchors from the
    library's next-anchor buffer, so successive replays continue decoding.
    Every buffer and launch shape is fixed at capture; per-sequence lengths
    live on the device, so the graph stays valid as the sequences grow."""
    b = seq_ids.numel()
    anchors = eng.next_anchor[:b]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        if tree:
            eng.tree_step(seq_ids, anchors, topk, budget)
        else:
            eng.step(seq_ids, anchors)
    return g
