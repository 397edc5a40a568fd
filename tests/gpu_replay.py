"""Step-by-step comparison of the GPU library with the CPU oracle (replay).

The oracle follows the GPU's committed tokens: at every step it recomputes
the draft and verify logits for the GPU's block, checks the GPU's logits
within the tolerance, checks every GPU argmax where the oracle's top-1/top-2
margin exceeds 1e-2 (near-ties may legitimately flip), checks the accept
decision against the stated rule, then commits the GPU's accepted rows.
"""
import numpy as np
import torch

from oracle import numerics as nm
from oracle.decode import Sequence1, accept_longest_prefix
from oracle.ddtree import build_tree, tree_accept, tree_commit, tree_verify

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
