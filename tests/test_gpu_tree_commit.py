"""The commit half of a DDTree step on the GPU, with a teacher-forced tree.

"LLMs hit ludicrous speed ..." (joindrip.ai), DDTree paragraph: the target
verifies every node of the draft tree in one pass and the path it accepts is
kept.  With random weights the drafter's own trees are never accepted, so
these tests force the tree: its path carries the target's greedy
continuation (taken from the GPU's plain AR decoding) at cache slots
s_j > j, with decoys before path nodes 1 and 3, so that compaction moves rows
onto slots that are themselves sources of earlier path rows (the two-phase
gather of the compaction reading).  Checked against the oracle:
  * verify logits and argmax of every node (ancestor-only mask);
  * the accept walk (a >= 3), the emitted tokens and the new length;
  * every target layer's K/V after the commit: row P + j is, bit for bit,
    the pre-commit row P + s_j;
  * the draft cache rows P .. P + a of every draft layer: the oracle's
    injection of the captured rows of the path nodes at positions P + j;
  * the next step's draft logits against the oracle after its own
    tree commit.
Also: dflash_inject_kv with explicit hidden rows (not the commit queue).

Tolerances: max-abs 2e-2, relative 1e-2 (bf16 path); argmax exact where the
oracle's top-1/top-2 margin exceeds 1e-2; compaction bit-exact.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import numerics as nm
from oracle.ddtree import tree_accept, tree_commit, tree_verify
from oracle.decode import Sequence1
from oracle.models import KVCache, Weights, inject_kv

from gpu_replay import cache_band, check_argmax, check_close, forced_tree, tree_arrays

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-2, 1e-2
PATH_LEN = 6


@pytest.fixture(scope="module")
def forced_mini():
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["mini_bf16_ddtree"]
    s, b, B = w.shape, w.batch, w.block_size
    prompts = wl.prompts(w)
    lens = [len(p) for p in prompts]
    nmax = w.tree_budget + 1
    eng = DFlashEngine(s, B, b, 512, max_rows=256, max_tree_nodes=nmax)
    ar = eng.generate(prompts, PATH_LEN + 3, mode="ar")
    sid = eng.seq_ids(b)
    anchors = eng.prefill(prompts)
    torch.cuda.synchronize()
    assert anchors.tolist() == [a[0] for a in ar]
    trees = [forced_tree(ar[q][0], ar[q][1:1 + PATH_LEN], ar[q][1 + PATH_LEN], nmax, s.vocab,
                         B - 1) for q in range(b)]
    lo, hi = min(lens) - 2, max(lens) + nmax
    tl = [(n, l) for l in range(s.n_layers) for n in ("k_cache", "v_cache")]
    dl = [(n, l) for l in range(s.n_draft_layers) for n in ("dk_cache", "dv_cache")]
    snap = {}
    r = eng.tree_step(sid, anchors, w.topk, w.tree_budget, want_logits=True,
                      tree_override=tree_arrays(trees, nmax),
                      before_commit=lambda: snap.update(cache_band(eng, tl, b, lo, hi)))
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in r.items()}
    post = cache_band(eng, tl, b, lo, hi)
    dpost = cache_band(eng, dl, b, lo, hi)
    capture = eng.debug_view("capture")[: b * nmax].float().cpu().numpy()
    lengths = eng.lengths(b)
    anchors2 = r["next_anchor"][:b].clone()
    dlog = torch.empty(b * (B - 1) * s.vocab, dtype=torch.float32, device="cuda")
    capi.dflash_draft_block(eng.ctx, b, sid, anchors2, eng.block[: b * B], 0, None, None, dlog)
    torch.cuda.synchronize()
    res = dict(w=w, prompts=prompts, lens=lens, lo=lo, nmax=nmax, trees=trees, out=out, snap=snap,
               post=post, dpost=dpost, capture=capture, lengths=lengths,
               anchors2=anchors2.cpu().numpy(), dlog=dlog.view(b, B - 1, -1).cpu().numpy(),
               dblock=eng.block[: b * B].view(b, B).cpu().numpy())
    eng.close()
    res["W"] = Weights(wl.SyntheticWeights(s))
    return res


def test_forced_tree_verify_and_walk(forced_mini):
    r = forced_mini
    w, out = r["w"], r["out"]
    prec = nm.Precision("bf16emu")
    best = 0
    for q in range(w.batch):
        t = r["trees"][q]
        n = t.n_nodes
        assert list(out["tok"][q, :n]) == t.tok and list(out["parent"][q, :n]) == t.parent
        seq = Sequence1(r["W"], w.shape, prec, 512)
        seq.prefill(r["prompts"][q], inject=True)
        ovl, _ = tree_verify(seq, t)
        check_close(out["logits"][q, :n], ovl, ATOL, RTOL, f"seq {q} tree logits")
        check_argmax(out["argmax"][q, :n], ovl, f"seq {q} tree argmax")
        a, path, emitted = tree_accept(t, [int(v) for v in out["argmax"][q, :n]])
        assert a == int(out["accept_len"][q])
        assert emitted == [int(v) for v in out["emitted"][q] if v >= 0]
        assert r["lengths"][q] == r["lens"][q] + a + 1
        assert path[:4] == [0, 2, 3, 5][: a + 1]  # the designed slots s_j > j
        best = max(best, a)
    assert best >= 3, "no forced path was accepted (greedy continuation lost to a near-tie?)"


def _path(r, q):
    t = r["trees"][q]
    return tree_accept(t, [int(v) for v in r["out"]["argmax"][q, : t.n_nodes]])[1]


def test_forced_tree_compaction_is_bit_exact(forced_mini):
    r = forced_mini
    s = r["w"].shape
    for q in range(r["w"].batch):
        path = _path(r, q)
        P, lo = r["lens"][q], r["lo"]
        for l in range(s.n_layers):
            for n in ("k_cache", "v_cache"):
                pre, post = r["snap"][(n, l)][q], r["post"][(n, l)][q]
                for j, node in enumerate(path):
                    np.testing.assert_array_equal(post[:, P + j - lo], pre[:, P + node - lo],
                                                  err_msg=f"seq {q} layer {l} {n} row {j}")
                # context rows and the rows past the accepted path are untouched
                np.testing.assert_array_equal(post[:, : P - lo], pre[:, : P - lo])
                np.testing.assert_array_equal(post[:, P + len(path) - lo:],
                                              pre[:, P + len(path) - lo:])


def test_forced_tree_path_injected_into_draft_cache(forced_mini):
    r = forced_mini
    w, s = r["w"], r["w"].shape
    prec = nm.Precision("bf16emu")
    for q in range(w.batch):
        path = _path(r, q)
        P, lo = r["lens"][q], r["lo"]
        rows = r["capture"][q * r["nmax"] + np.array(path)].astype(np.float64)
        dc = KVCache(s.n_draft_layers, P + len(path), s.n_kv_heads, s.head_dim)
        pos = P + np.arange(len(path))
        inject_kv(r["W"], s, prec, dc, rows, pos)
        for l in range(s.n_draft_layers):
            gk = r["dpost"][("dk_cache", l)][q][:, pos - lo].transpose(1, 0, 2)
            gv = r["dpost"][("dv_cache", l)][q][:, pos - lo].transpose(1, 0, 2)
            check_close(gk, dc.k[l, pos], ATOL, RTOL, f"seq {q} draft layer {l} K")
            check_close(gv, dc.v[l, pos], ATOL, RTOL, f"seq {q} draft layer {l} V")


def test_next_draft_after_tree_commit_matches_oracle(forced_mini):
    r = forced_mini
    w = r["w"]
    prec = nm.Precision("bf16emu")
    for q in range(w.batch):
        t = r["trees"][q]
        seq = Sequence1(r["W"], w.shape, prec, 512)
        seq.prefill(r["prompts"][q], inject=True)
        _, cap = tree_verify(seq, t)
        tree_commit(seq, cap, _path(r, q))
        assert seq.length == r["lengths"][q]
        odl = seq.draft(int(r["anchors2"][q]), w.block_size)
        check_close(r["dlog"][q], odl, ATOL, RTOL, f"seq {q} next draft logits")
        check_argmax(r["dblock"][q, 1:], odl, f"seq {q} next draft argmax")


def test_inject_kv_with_explicit_hidden_rows():
    """dflash_inject_kv with caller rows: F = W_fuse h, K = RoPE(W_k F),
    V = W_v F into the given (slot, position) of every draft layer; a row
    with position -1 is skipped."""
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    s = wl.MINI_BF16
    eng = DFlashEngine(s, 16, 2, 256, max_rows=64)
    rng = np.random.default_rng(31)
    n = 7
    hid = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(
        (rng.standard_normal((n, s.n_inject, s.d_model)) * 0.5).astype(np.float32)))
    seqs = np.array([0, 1, 1, 0, 1, 0, 1], np.int32)
    pos = np.array([3, 100, 101, 200, -1, 17, 5], np.int32)
    dk0 = [eng.debug_view("dk_cache", l).float().cpu().numpy() for l in range(s.n_draft_layers)]
    capi.dflash_inject_kv(eng.ctx, n, torch.from_numpy(seqs).cuda(), torch.from_numpy(pos).cuda(),
                          torch.from_numpy(hid).cuda().to(torch.bfloat16))
    capi.dflash_check(eng.ctx)
    W = Weights(wl.SyntheticWeights(s))
    live = np.nonzero(pos >= 0)[0]
    oc = KVCache(s.n_draft_layers, 256, s.n_kv_heads, s.head_dim)  # positions are distinct
    inject_kv(W, s, nm.Precision("bf16emu"), oc, hid[live].astype(np.float64), pos[live])
    for l in range(s.n_draft_layers):
        gk = eng.debug_view("dk_cache", l).float().cpu().numpy()
        gv = eng.debug_view("dv_cache", l).float().cpu().numpy()
        for i in live:
            check_close(gk[seqs[i], :, pos[i]], oc.k[l, pos[i]], ATOL, RTOL, f"row {i} layer {l} K")
            check_close(gv[seqs[i], :, pos[i]], oc.v[l, pos[i]], ATOL, RTOL, f"row {i} layer {l} V")
        # nothing else was written: only the live rows' slots changed
        changed = np.argwhere(np.any(gk != dk0[l], axis=(1, 3)))
        assert {(int(a), int(p)) for a, p in changed} <= {(int(seqs[i]), int(pos[i])) for i in live}
    eng.close()
