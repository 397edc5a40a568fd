"""Step-by-step comparison of the GPU library with the CPU oracle (replay).

The oracle follows the GPU's committed tokens: at every step it recomputes
the draft and verify logits for the GPU's block, checks the GPU's logits
within the tolerance, checks every GPU argmax where the oracle's top-1/top-2
margin exceeds 1e-2 (near-ties may legitimately flip), checks the accept
decision against the stated rule, then commits the GPU's accepted rows.
"""
import numpy as np
import torch

import workloads as wl

from oracle import numerics as nm
from oracle.decode import Sequence1, accept_longest_prefix
from oracle.ddtree import DraftTree, build_tree, tree_accept, tree_commit, tree_verify

MARGIN = 1e-2


def check_close(gpu, ref, atol, rtol, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref) - (atol + rtol * np.abs(ref))
    if np.any(err > 0):
        i = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(f"{what}: |gpu-oracle| exceeds tol at {i}: gpu={gpu[i]} oracle={ref[i]} "
                             f"max abs diff={np.abs(gpu - ref).max():.3e}")


def check_argmax(gpu_ids, logits, what, atol=2e-2, rtol=1e-2):
    """Exact where the oracle margin exceeds 1e-2; at exempt (near-tie)
    positions the GPU's pick must still be a near-maximal logit: within
    twice the logit tolerance of the oracle's maximum."""
    n_checked = 0
    for j, (g, row) in enumerate(zip(gpu_ids, logits)):
        if nm.top2_margin(row) > MARGIN:
            assert int(g) == nm.argmax_lowest(row), f"{what} row {j}: gpu {g} oracle {nm.argmax_lowest(row)}"
            n_checked += 1
        else:
            top = float(np.max(row))
            assert row[int(g)] >= top - 2 * (atol + rtol * abs(top)), \
                f"{what} row {j}: near-tie but gpu {g} (logit {row[int(g)]}) far from max {top}"
    return n_checked


def replay_prefill(eng, W, shape, prec, prompts, max_len, atol, rtol):
    anchors = eng.prefill(prompts)
    torch.cuda.synchronize()
    seqs = []
    for s, p in enumerate(prompts):
        seq = Sequence1(W, shape, prec, max_len)
        lg, _ = seq.prefill(p, inject=True)
        check_argmax([anchors[s].item()], lg[-1:], f"prefill seq {s}")
        seqs.append(seq)
    assert eng.lengths(len(prompts)) == [len(p) for p in prompts]
    return anchors, seqs


def replay_linear(eng, W, shape, prec, prompts, n_steps, atol, rtol, max_len):
    b = len(prompts)
    B = eng.B
    sid = eng.seq_ids(b)
    anchors, seqs = replay_prefill(eng, W, shape, prec, prompts, max_len, atol, rtol)
    stats = dict(checked=0, steps=0, accepted=0)
    for step in range(n_steps):
        out, dlog, vlog, _ = eng.step(sid, anchors, want_logits=True)
        torch.cuda.synchronize()
        blocks = out.block.cpu().numpy()
        ys = out.argmax.cpu().numpy()
        acc = out.accept_len.cpu().numpy()
        em = out.emitted.cpu().numpy()
        dl = dlog.cpu().numpy()
        vl = vlog.cpu().numpy()
        for s in range(b):
            blk = [int(t) for t in blocks[s]]
            if B > 1:
                odl = seqs[s].draft(blk[0], B)
                check_close(dl[s], odl, atol, rtol, f"step {step} seq {s} draft logits")
                stats["checked"] += check_argmax(blk[1:], odl, f"step {step} seq {s} draft")
            ovl, cap = seqs[s].verify(blk)
            check_close(vl[s], ovl, atol, rtol, f"step {step} seq {s} verify logits")
            stats["checked"] += check_argmax(ys[s], ovl, f"step {step} seq {s} verify")
            a, emitted = accept_longest_prefix(blk[1:], [int(v) for v in ys[s]])
            assert a == int(acc[s]), (step, s, a, acc[s])
            assert emitted == [int(t) for t in em[s] if t >= 0]
            seqs[s].commit_linear(cap, a)
            stats["accepted"] += a
        anchors = out.next_anchor.clone()
        stats["steps"] += 1
    assert eng.lengths(b) == [sq.length for sq in seqs]
    return seqs, stats


def replay_tree(eng, W, shape, prec, prompts, n_steps, topk, budget, atol, rtol, max_len):
    b = len(prompts)
    B = eng.B
    sid = eng.seq_ids(b)
    anchors, seqs = replay_prefill(eng, W, shape, prec, prompts, max_len, atol, rtol)
    for step in range(n_steps):
        r = eng.tree_step(sid, anchors, topk, budget, want_logits=True)
        torch.cuda.synchronize()
        h = {k: v.cpu().numpy() for k, v in r.items()}
        for s in range(b):
            anchor = int(anchors[s].item())
            # the drafter's top-k lists against the oracle's draft logits
            odl = seqs[s].draft(anchor, B)
            for j in range(B - 1):
                lp = nm.log_softmax(odl[j])
                check_close(h["logp"][s, j], lp[h["ids"][s, j]], atol, rtol, f"step {step} topk logp")
                if nm.top2_margin(odl[j]) > MARGIN:
                    assert h["ids"][s, j, 0] == nm.argmax_lowest(odl[j])
            # the heap on the GPU's own top-k input: bit-exact node order
            t = build_tree(anchor, h["ids"][s], h["logp"][s], budget)
            n = t.n_nodes
            assert int(h["n_nodes"][s]) == n
            assert list(h["tok"][s, :n]) == t.tok
            assert list(h["parent"][s, :n]) == t.parent
            assert list(h["depth"][s, :n]) == t.depth
            for i in range(n):
                words = [int(x) & ((1 << 64) - 1) for x in h["anc"][s, i]]
                assert sum(w << (64 * k) for k, w in enumerate(words)) == t.ancestors[i]
            ovl, cap = tree_verify(seqs[s], t)
            check_close(h["logits"][s, :n], ovl, atol, rtol, f"step {step} seq {s} tree logits")
            check_argmax(h["argmax"][s, :n], ovl, f"step {step} seq {s} tree verify")
            a, path, emitted = tree_accept(t, [int(v) for v in h["argmax"][s, :n]])
            assert a == int(h["accept_len"][s])
            assert emitted == [int(v) for v in h["emitted"][s] if v >= 0]
            tree_commit(seqs[s], cap, path)
        anchors = r["next_anchor"].clone()
    assert eng.lengths(b) == [sq.length for sq in seqs]
    return seqs


# ---------------------------------------------------------------------------
# teacher-forced draft trees (DDTree accept walk and KV compaction)
# ---------------------------------------------------------------------------

def forced_tree(anchor, path_tokens, next_token, n_nodes, vocab, depth_max):
    """A draft tree whose greedy walk follows ``path_tokens`` (the target's
    greedy continuation after ``anchor``) at slots s_j > j.

    Node 0 is the anchor.  A decoy sibling (a token other than the path
    token) takes the slot before path nodes 1 and 3, so the path sits at
    s = 0, 2, 3, 5, 6, 7, ...: compaction then writes slots that are
    themselves sources of earlier path rows (the overlapping case of the
    two-phase gather).  The last path node gets a decoy child whose token
    differs from ``next_token``, so the walk stops there.  The rest of the
    budget is filled by decoy children of node 1, off the path."""
    tok, parent, depth = [int(anchor)], [-1], [0]

    def add(t, p):
        tok.append(int(t) % vocab)
        parent.append(p)
        depth.append(depth[p] + 1)
        return len(tok) - 1

    cur = 0
    for j, t in enumerate(path_tokens, start=1):
        if j in (1, 3):
            add(int(t) + 1, cur)
        cur = add(t, cur)
    assert depth[cur] <= depth_max
    if depth[cur] < depth_max and len(tok) < n_nodes:
        add(int(next_token) + 1, cur)
    k = 2
    while len(tok) < n_nodes:
        add(int(path_tokens[0]) + k, 1)
        k += 1
    anc = []
    for i, p in enumerate(parent):
        anc.append((anc[p] if p >= 0 else 0) | (1 << i))
    n = len(tok)
    return DraftTree(tok, parent, depth, [0] * n, [0.0] * n, anc)


def tree_arrays(trees, max_nodes, device="cuda"):
    """The dtree_buffers arrays of oracle trees (one per sequence), on the
    device, in the layout dtree_build writes."""
    b, words = len(trees), (max_nodes + 63) // 64
    tok = np.full((b, max_nodes), -1, np.int32)
    parent = np.full((b, max_nodes), -1, np.int32)
    depth = np.zeros((b, max_nodes), np.int32)
    anc = np.zeros((b, max_nodes, words), np.int64)
    for s, t in enumerate(trees):
        n = t.n_nodes
        tok[s, :n], parent[s, :n], depth[s, :n] = t.tok, t.parent, t.depth
        for i in range(n):
            for w in range(words):
                v = (t.ancestors[i] >> (64 * w)) & ((1 << 64) - 1)
                anc[s, i, w] = v - (1 << 64) if v >= (1 << 63) else v
    n_nodes = np.array([t.n_nodes for t in trees], np.int32)
    arr = dict(tok=tok, parent=parent, depth=depth, anc=anc, n_nodes=n_nodes)
    return {k: torch.from_numpy(v).to(device) for k, v in arr.items()}


def cache_band(eng, names_layers, b, lo, hi):
    """Host copies of cache slots [lo, hi) of the first b sequences:
    {(name, layer): array [b][H_kv][hi-lo][hd] float32}."""
    return {(nm_, l): eng.debug_view(nm_, l)[:b, :, lo:hi].float().cpu().numpy()
            for nm_, l in names_layers}


# ---------------------------------------------------------------------------
# full-size spot checks (the oracle computes sampled rows and layers only)
# ---------------------------------------------------------------------------

def lm_logits(shape, seed, h_final, gain_name="final_norm"):
    """Oracle lm_head logits [n, V] of fp32 residual rows h_final [n, d]
    after the final RMSNorm (norm gains are 1 in the synthetic weights; the
    gain name only documents which norm it is), streaming the lm_head rows in
    chunks so that the whole table is never held in fp64."""
    assert gain_name in ("final_norm", "draft.final_norm")
    sw = wl.SyntheticWeights(shape, seed)
    h = np.atleast_2d(np.asarray(h_final, dtype=np.float64))
    hn = nm.round_bf16(nm.rmsnorm(h, np.ones(shape.d_model), shape.rms_eps))
    offs = sw.offsets("lm_head")
    out = np.empty((h.shape[0], shape.vocab))
    for c0 in range(0, shape.vocab, 16384):
        rows = wl.pool_rows(sw.pool(), offs[c0: c0 + 16384], shape.d_model).astype(np.float64)
        out[:, c0: c0 + len(rows)] = hn @ rows.T
    return out


def draft_inputs(shape, seed, anchor, block):
    """Residual rows entering the first draft layer: the anchor's embedding,
    then the mask embedding in every other slot."""
    sw = wl.SyntheticWeights(shape, seed)
    emb = wl.pool_rows(sw.pool(), sw.offsets("tok_emb")[[int(anchor)]], shape.d_model)[0]
    return np.stack([emb] + [sw["draft.mask_emb"]] * (block - 1)).astype(np.float64)


def check_draft_layer(W, shape, l, x, ctx_len, ctx_k, ctx_v, q_gpu, attn_gpu, out_gpu, what,
                      atol=2e-2, rtol=1e-2):
    """Teacher-forced check of draft layer l over all B block rows, in three
    well-conditioned stages (each gets the exact inputs the GPU consumed):
      1. the roped queries: the oracle's, from the block rows x [B, d] at
         positions ctx_len .., against the GPU's q_gpu [B, H*hd];
      2. the attention: the GPU's queries over the context rows ctx_k / ctx_v
         [ctx_len, H_kv, hd] (the GPU's draft cache) and the block's own K/V
         (no mask), against the GPU's attention output attn_gpu [B, H*hd];
      3. the rest of the layer (O projection, residual, FFN) from the GPU's
         attention output, against the GPU's residual after the layer.
    The injected context keys of a random-init drafter are large, so its
    softmax is close to a hard maximum: one bf16 rounding of a query element
    that lands on the other side of a rounding boundary can move weight
    between two near-tied keys.  Stage 2 therefore uses the GPU's queries."""
    from oracle.models import _layer
    B = x.shape[0]
    rec = {}
    G = shape.n_heads // shape.n_kv_heads
    qg = np.asarray(q_gpu, dtype=np.float64).reshape(B, shape.n_heads, shape.head_dim)

    def attend_rows(q, k, v):
        rec["q"] = q
        kk = np.concatenate([ctx_k, k])
        vv = np.concatenate([ctx_v, v])
        rec["attn"] = np.stack([nm.attend(qg[i], kk, vv) for i in range(B)])
        assert kk.shape[1] * G == shape.n_heads
        return np.asarray(attn_gpu, dtype=np.float64).reshape(B, shape.n_heads, shape.head_dim)

    y = _layer(W, shape, nm.Precision("bf16emu"), f"draft.layers.{l}", x,
               ctx_len + np.arange(B), attend_rows)
    check_close(q_gpu, rec["q"].reshape(B, -1), atol, rtol, f"{what}: roped queries")
    check_close(attn_gpu, rec["attn"].reshape(B, -1), atol, rtol, f"{what}: attention output")
    check_close(out_gpu, y, atol, rtol, f"{what}: layer output")


def check_injection(W, shape, hcat, fused_gpu, positions, k_gpu, v_gpu, what, atol=2e-2,
                    rtol=1e-2):
    """KV injection of rows hcat [n, n_inject, d] at ``positions``, in two
    stages: F = bf16(W_fuse h_cat) against the GPU's F (fused_gpu [n, d]), then
    every draft layer's K = RoPE(W_k F) and V = W_v F from the GPU's F against
    the GPU's cache rows k_gpu[l] / v_gpu[l] [n, H_kv, hd].  (F of a deep
    random target is large, so one bf16 rounding of F that differs between
    the two sides would show up in K beyond the element-wise tolerance of
    near-zero elements; each stage on its own is well conditioned.)"""
    n = hcat.shape[0]
    prec = nm.Precision("bf16emu")
    f = prec.store(nm.linear(np.asarray(hcat, dtype=np.float64).reshape(n, -1), W["draft.fuse"]))
    check_close(fused_gpu, f, atol, rtol, f"{what}: fused feature F")
    fg = np.asarray(fused_gpu, dtype=np.float64)
    pos = np.asarray(positions)
    for l in range(shape.n_draft_layers):
        k = nm.linear(fg, W[f"draft.layers.{l}.wk"]).reshape(n, shape.n_kv_heads, shape.head_dim)
        k = prec.store(nm.apply_rope(k, pos, shape.rope_theta))
        v = prec.store(nm.linear(fg, W[f"draft.layers.{l}.wv"]).reshape(n, shape.n_kv_heads,
                                                                         shape.head_dim))
        check_close(k_gpu[l], k, atol, rtol, f"{what}: draft layer {l} K")
        check_close(v_gpu[l], v, atol, rtol, f"{what}: draft layer {l} V")
