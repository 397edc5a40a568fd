"""Full-size parity of the batched and draft-tree workloads.

* Qwen3-8B-shaped target + 5-layer drafter, batch 32, prompt lengths drawn
  uniform in [512, 4096] (ragged caches), one DFlash step: accept rule and
  lengths of every sequence; layer-0 cache rows; sampled layers of sampled
  rows teacher-forced on the GPU's fp32 residual and caches; final logits.
* Llama-3.1-8B-shaped target + 5-layer drafter, batch 4, prompt 4096, one
  DDTree step (top-8 per slot, 64 drafted nodes + root): the heap tree is
  rebuilt by the oracle from the GPU's top-k lists and must match bit for
  bit; sampled nodes' layers are teacher-forced under the ancestor-only mask
  at position P + depth; the accept walk follows the stated rule; the
  accepted path's K/V rows are moved to consecutive slots in every layer
  (bit-exact against the pre-commit cache).

Tolerance: max-abs 2e-2, relative 1e-2; argmax exact where the oracle's
top-1/top-2 margin exceeds 1e-2; integer results bit-exact.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import numerics as nm
from oracle.ddtree import build_tree, tree_accept
from oracle.decode import accept_longest_prefix
from oracle.models import Weights, _layer

from gpu_replay import (cache_band, check_argmax, check_close, check_draft_layer, check_injection,
                        draft_inputs, forced_tree, lm_logits, tree_arrays)

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-2, 1e-2


def _row_layer(W, shape, l, x, pos, kc, vc, visible_slots, own_slot_last=True):
    """Oracle layer l for one row: keys = cache rows `visible_slots` (GPU
    values) followed by the row's own K/V."""
    def attend_rows(q, k, v):
        kk = np.concatenate([kc[visible_slots], k])
        vv = np.concatenate([vc[visible_slots], v])
        return np.stack([nm.attend(q[0], kk, vv)])
    return _layer(W, shape, nm.Precision("bf16emu"), f"layers.{l}", x, np.array([pos]), attend_rows)


def _lm_logits(shape, seed, h_final):
    sw = wl.SyntheticWeights(shape, seed)
    hn = nm.round_bf16(nm.rmsnorm(h_final[None, :], np.ones(shape.d_model), shape.rms_eps))[0]
    offs = sw.offsets("lm_head")
    out = np.empty(shape.vocab)
    for c0 in range(0, shape.vocab, 16384):
        rows = wl.pool_rows(sw.pool(), offs[c0: c0 + 16384], shape.d_model).astype(np.float64)
        out[c0: c0 + len(rows)] = rows @ hn
    return out


# ---------------------------------------------------------------------------
# batch 32, ragged
# ---------------------------------------------------------------------------
B32_LAYERS = (1, 18, 35)
B32_DRAFT_LAYERS = (0, 4)


@pytest.fixture(scope="module")
def b32():
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["qwen3_8b_b32"]
    prompts = wl.prompts(w)
    lens = [len(p) for p in prompts]
    eng = DFlashEngine(w.shape, 16, w.batch, max(lens) + 64, max_rows=max(lens))
    sid = eng.seq_ids(w.batch)
    anchors = eng.prefill(prompts)
    trace = torch.zeros(w.shape.n_layers, eng.max_rows, w.shape.d_model, dtype=torch.float32,
                        device="cuda")
    dtrace = torch.zeros(w.shape.n_draft_layers, eng.max_rows, w.shape.d_model,
                         dtype=torch.float32, device="cuda")
    qa = [torch.zeros(w.shape.n_draft_layers, eng.max_rows, w.shape.q_dim, dtype=torch.bfloat16,
                      device="cuda") for _ in range(2)]
    capi.dflash_debug_trace(eng.ctx, trace)
    capi.dflash_debug_trace_draft(eng.ctx, dtrace)
    capi.dflash_debug_trace_draft_attn(eng.ctx, *qa)
    out, dlog, vlog, _ = eng.step(sid, anchors, want_logits=True)
    torch.cuda.synchronize()
    capi.dflash_debug_trace(eng.ctx, None)
    capi.dflash_debug_trace_draft(eng.ctx, None)
    capi.dflash_debug_trace_draft_attn(eng.ctx, None, None)
    picks = [(3, 0), (17, 9)]  # (sequence, block row)
    r = dict(w=w, prompts=prompts, lens=lens, picks=picks,
             block=out.block.cpu().numpy(), argmax=out.argmax.cpu().numpy(),
             accept=out.accept_len.cpu().numpy(), emitted=out.emitted.cpu().numpy(),
             length=eng.lengths(w.batch),
             vlog={(s, j): vlog[s, j].cpu().numpy() for s, j in picks},
             trace={(s, j): trace[:, s * 16 + j].cpu().numpy() for s, j in picks},
             cache={},
             dtrace={s: dtrace[:, s * 16:(s + 1) * 16].cpu().numpy() for s, _ in picks},
             dq={s: qa[0][:, s * 16:(s + 1) * 16].float().cpu().numpy() for s, _ in picks},
             dao={s: qa[1][:, s * 16:(s + 1) * 16].float().cpu().numpy() for s, _ in picks},
             dlog={s: dlog[s].cpu().numpy() for s, _ in picks},
             dctx={(s, l): (eng.debug_view("dk_cache", l)[s, :, :lens[s]].float().cpu().numpy()
                            .transpose(1, 0, 2),
                            eng.debug_view("dv_cache", l)[s, :, :lens[s]].float().cpu().numpy()
                            .transpose(1, 0, 2))
                   for s, _ in picks for l in B32_DRAFT_LAYERS})
    for s, j in picks:
        n = lens[s] + 16
        for l in (0,) + B32_LAYERS:
            r["cache"][(s, l)] = (eng.debug_view("k_cache", l)[s, :, :n].float().cpu().numpy().transpose(1, 0, 2),
                                  eng.debug_view("v_cache", l)[s, :, :n].float().cpu().numpy().transpose(1, 0, 2))
    eng.close()
    del eng, trace, dtrace, qa, vlog, dlog
    torch.cuda.empty_cache()
    r["W"] = Weights(wl.SyntheticWeights(w.shape, w.seed))
    return r


def test_b32_accept_and_lengths(b32):
    for s in range(b32["w"].batch):
        a, em = accept_longest_prefix([int(t) for t in b32["block"][s, 1:]],
                                      [int(y) for y in b32["argmax"][s]])
        assert a == int(b32["accept"][s])
        assert em == [int(t) for t in b32["emitted"][s] if t >= 0]
        assert b32["length"][s] == b32["lens"][s] + a + 1


def test_b32_layer0_cache_rows(b32):
    s_ = b32["w"].shape
    W = b32["W"]
    prec = nm.Precision("bf16emu")
    for s, _ in b32["picks"]:
        P = b32["lens"][s]
        toks = np.concatenate([b32["prompts"][s], b32["block"][s]]).astype(np.int64)
        slots = [0, P // 2, P - 1, P, P + 15]
        h = prec.store(nm.rmsnorm(W["tok_emb"][toks[slots]], W["layers.0.attn_norm"], s_.rms_eps))
        k = nm.linear(h, W["layers.0.wk"]).reshape(len(slots), s_.n_kv_heads, s_.head_dim)
        k = prec.store(nm.apply_rope(k, np.array(slots), s_.rope_theta))
        check_close(b32["cache"][(s, 0)][0][slots], k, ATOL, RTOL, f"seq {s} layer-0 K rows")


def test_b32_sampled_layers_teacher_forced(b32):
    s_ = b32["w"].shape
    for s, j in b32["picks"]:
        P = b32["lens"][s]
        for l in B32_LAYERS:
            kc, vc = b32["cache"][(s, l)]
            x = b32["trace"][(s, j)][l - 1][None, :].astype(np.float64)
            y = _row_layer(b32["W"], s_, l, x, P + j, kc, vc, np.arange(P + j))
            b32["W"]._cache.clear()
            check_close(b32["trace"][(s, j)][l], y[0], ATOL, RTOL, f"seq {s} row {j} layer {l}")


def test_b32_final_logits(b32):
    w = b32["w"]
    for s, j in b32["picks"]:
        lg = _lm_logits(w.shape, w.seed, b32["trace"][(s, j)][-1].astype(np.float64))
        check_close(b32["vlog"][(s, j)], lg, ATOL, RTOL, f"seq {s} row {j} logits")
        check_argmax([b32["argmax"][s, j]], lg[None, :], f"seq {s} row {j} argmax")


@pytest.mark.parametrize("l", B32_DRAFT_LAYERS)
def test_b32_draft_layers_teacher_forced(b32, l):
    """Draft layer l of two sequences' blocks (16 rows each, ragged contexts),
    teacher-forced on the GPU's draft traces and draft cache (three stages:
    queries, attention on the GPU's queries, the rest of the layer)."""
    w = b32["w"]
    for s, _ in b32["picks"]:
        P = b32["lens"][s]
        x = (draft_inputs(w.shape, w.seed, b32["block"][s, 0], 16) if l == 0
             else b32["dtrace"][s][l - 1].astype(np.float64))
        check_draft_layer(b32["W"], w.shape, l, x, P, *b32["dctx"][(s, l)], b32["dq"][s][l],
                          b32["dao"][s][l], b32["dtrace"][s][l], f"seq {s} draft layer {l}")
        b32["W"]._cache.clear()


def test_b32_draft_logits_and_argmax(b32):
    w = b32["w"]
    for s, _ in b32["picks"]:
        lg = lm_logits(w.shape, w.seed, b32["dtrace"][s][-1][1:], "draft.final_norm")
        check_close(b32["dlog"][s], lg, ATOL, RTOL, f"seq {s} draft logits")
        check_argmax(b32["block"][s, 1:], lg, f"seq {s} drafted tokens")


# ---------------------------------------------------------------------------
# DDTree, Llama shape, batch 4, context 4096
# ---------------------------------------------------------------------------
TREE_LAYERS = (1, 16, 31)


@pytest.fixture(scope="module")
def tree():
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["llama31_8b_ddtree_b4"]
    prompts = wl.prompts(w)
    P = len(prompts[0])
    nmax = w.tree_budget + 1
    eng = DFlashEngine(w.shape, 16, w.batch, P + nmax + 64, max_rows=P, max_tree_nodes=nmax)
    sid = eng.seq_ids(w.batch)
    anchors = eng.prefill(prompts)
    b, B, k = w.batch, 16, w.topk
    m = eng.tree_mem
    ids = m["topk_ids"][: b * (B - 1) * k]
    lps = m["topk_logp"][: b * (B - 1) * k]
    block = eng.block[: b * B]
    capi.dflash_draft_block(eng.ctx, b, sid, anchors, block, k, ids, lps, None)
    capi.dtree_build(eng.ctx, b, anchors, ids, lps, k, w.tree_budget, eng.tree)
    trace = torch.zeros(w.shape.n_layers, eng.max_rows, w.shape.d_model, dtype=torch.float32,
                        device="cuda")
    capi.dflash_debug_trace(eng.ctx, trace)
    argmax = eng.argmax[: b * nmax]
    vlog = torch.empty(b * nmax * w.shape.vocab, dtype=torch.float32, device="cuda")
    capi.dtree_verify(eng.ctx, b, sid, eng.tree, argmax, None, vlog)
    torch.cuda.synchronize()
    capi.dflash_debug_trace(eng.ctx, None)
    pre = {l: (eng.debug_view("k_cache", l)[:, :, : P + nmax].float().cpu().numpy(),
               eng.debug_view("v_cache", l)[:, :, : P + nmax].float().cpu().numpy())
           for l in (0,) + TREE_LAYERS}
    emitted = eng.emitted[: b * nmax]
    capi.dflash_accept_commit(eng.ctx, b, sid, None, argmax, eng.tree, capi.DFLASH_ACCEPT_GREEDY,
                              eng.accept_len[:b], eng.next_anchor[:b], emitted)
    capi.dflash_inject_kv(eng.ctx)
    torch.cuda.synchronize()
    post = {l: (eng.debug_view("k_cache", l)[:, :, : P + nmax].float().cpu().numpy(),
                eng.debug_view("v_cache", l)[:, :, : P + nmax].float().cpu().numpy())
            for l in (0,) + TREE_LAYERS}
    picks = [(0, 1), (2, 40)]  # (sequence, node)
    r = dict(w=w, P=P, nmax=nmax, picks=picks,
             anchors=anchors.cpu().numpy(),
             ids=ids.view(b, B - 1, k).cpu().numpy(), logp=lps.view(b, B - 1, k).cpu().numpy(),
             tok=m["tok"][: b * nmax].view(b, nmax).cpu().numpy(),
             parent=m["parent"][: b * nmax].view(b, nmax).cpu().numpy(),
             depth=m["depth"][: b * nmax].view(b, nmax).cpu().numpy(),
             anc=m["anc"][: b * nmax * 2].view(b, nmax, 2).cpu().numpy(),
             n_nodes=m["n_nodes"][:b].cpu().numpy(),
             argmax=argmax.view(b, nmax).cpu().numpy(),
             accept=eng.accept_len[:b].cpu().numpy(),
             emitted=emitted.view(b, nmax).cpu().numpy(), length=eng.lengths(b),
             vlog={(s, n): vlog.view(b, nmax, -1)[s, n].cpu().numpy() for s, n in picks},
             trace={(s, n): trace[:, s * nmax + n].cpu().numpy() for s, n in picks},
             pre=pre, post=post)
    eng.close()
    del eng, trace, vlog
    torch.cuda.empty_cache()
    r["W"] = Weights(wl.SyntheticWeights(w.shape, w.seed))
    return r


def _oracle_tree(r, s):
    return build_tree(int(r["anchors"][s]), r["ids"][s], r["logp"][s], r["w"].tree_budget)


def test_tree_topk_lists_are_sorted_distributions(tree):
    ids, lp = tree["ids"], tree["logp"]
    assert np.all(lp <= 1e-6)
    assert np.all(np.diff(lp, axis=-1) <= 0)
    for s in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            assert len(set(ids[s, j].tolist())) == ids.shape[2]


def test_tree_build_bit_exact(tree):
    for s in range(tree["w"].batch):
        t = _oracle_tree(tree, s)
        n = t.n_nodes
        assert int(tree["n_nodes"][s]) == n == tree["w"].tree_budget + 1
        assert list(tree["tok"][s, :n]) == t.tok
        assert list(tree["parent"][s, :n]) == t.parent
        assert list(tree["depth"][s, :n]) == t.depth
        for i in range(n):
            words = [int(x) & ((1 << 64) - 1) for x in tree["anc"][s, i]]
            assert words[0] | (words[1] << 64) == t.ancestors[i]


def test_tree_nodes_teacher_forced_under_ancestor_mask(tree):
    s_ = tree["w"].shape
    P = tree["P"]
    for s, n in tree["picks"]:
        t = _oracle_tree(tree, s)
        anc = [m for m in range(t.n_nodes) if (t.ancestors[n] >> m) & 1 and m != n]
        visible = np.concatenate([np.arange(P), P + np.array(anc, dtype=np.int64)]).astype(np.int64)
        pos = P + t.depth[n]
        for l in TREE_LAYERS:
            kc = tree["pre"][l][0][s].transpose(1, 0, 2)
            vc = tree["pre"][l][1][s].transpose(1, 0, 2)
            x = tree["trace"][(s, n)][l - 1][None, :].astype(np.float64)
            y = _row_layer(tree["W"], s_, l, x, pos, kc, vc, visible)
            tree["W"]._cache.clear()
            check_close(tree["trace"][(s, n)][l], y[0], ATOL, RTOL, f"seq {s} node {n} layer {l}")


def test_tree_final_logits(tree):
    w = tree["w"]
    for s, n in tree["picks"]:
        lg = _lm_logits(w.shape, w.seed, tree["trace"][(s, n)][-1].astype(np.float64))
        check_close(tree["vlog"][(s, n)], lg, ATOL, RTOL, f"seq {s} node {n} logits")
        check_argmax([tree["argmax"][s, n]], lg[None, :], f"seq {s} node {n} argmax")


def test_tree_accept_walk_and_compaction(tree):
    P = tree["P"]
    for s in range(tree["w"].batch):
        t = _oracle_tree(tree, s)
        a, path, emitted = tree_accept(t, [int(v) for v in tree["argmax"][s, : t.n_nodes]])
        assert a == int(tree["accept"][s])
        assert emitted == [int(v) for v in tree["emitted"][s] if v >= 0]
        assert tree["length"][s] == P + a + 1
        for l in (0,) + TREE_LAYERS:
            for j, node in enumerate(path):
                for which in (0, 1):
                    np.testing.assert_array_equal(tree["post"][l][which][s, :, P + j],
                                                  tree["pre"][l][which][s, :, P + node])
            np.testing.assert_array_equal(tree["post"][l][0][s, :, :P], tree["pre"][l][0][s, :, :P])


# ---------------------------------------------------------------------------
# DDTree commit at full size: a teacher-forced tree (the drafter's own trees
# are never accepted with random weights).  The path carries the target's
# greedy continuation (GPU AR decoding) at slots s = 0, 2, 3, 5, 6, ... (decoy
# siblings before path nodes 1 and 3), so compaction writes rows that are
# sources of earlier path rows.
# ---------------------------------------------------------------------------
FORCED_PATH = 5
FORCED_DRAFT_LAYERS = (0, 4)


@pytest.fixture(scope="module")
def forced():
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["llama31_8b_ddtree_b4"]
    s, b = w.shape, w.batch
    prompts = wl.prompts(w)
    P = len(prompts[0])
    nmax = w.tree_budget + 1
    eng = DFlashEngine(s, 16, b, P + nmax + 64, max_rows=P, max_tree_nodes=nmax)
    ar = eng.generate(prompts, FORCED_PATH + 3, mode="ar")
    sid = eng.seq_ids(b)
    anchors = eng.prefill(prompts)
    torch.cuda.synchronize()
    assert anchors.tolist() == [a[0] for a in ar]
    trees = [forced_tree(ar[q][0], ar[q][1:1 + FORCED_PATH], ar[q][1 + FORCED_PATH], nmax,
                         s.vocab, 15) for q in range(b)]
    tl = [(n, l) for l in range(s.n_layers) for n in ("k_cache", "v_cache")]
    lo, hi = P - 2, P + nmax
    snap = {}
    r = eng.tree_step(sid, anchors, w.topk, w.tree_budget, tree_override=tree_arrays(trees, nmax),
                      before_commit=lambda: snap.update(cache_band(eng, tl, b, lo, hi)))
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in r.items()}
    post = cache_band(eng, tl, b, lo, hi)
    dl = [(n, l) for l in range(s.n_draft_layers) for n in ("dk_cache", "dv_cache")]
    dpost = cache_band(eng, dl, b, P, P + FORCED_PATH + 1)
    capture = eng.debug_view("capture")[: b * nmax].float().cpu().numpy()
    fused = eng.debug_view("fused")[: b * nmax].float().cpu().numpy()
    lengths = eng.lengths(b)
    # the next draft pass, over the committed and injected path
    dtrace = torch.zeros(s.n_draft_layers, eng.max_rows, s.d_model, dtype=torch.float32,
                         device="cuda")
    qa = [torch.zeros(s.n_draft_layers, eng.max_rows, s.q_dim, dtype=torch.bfloat16,
                      device="cuda") for _ in range(2)]
    capi.dflash_debug_trace_draft(eng.ctx, dtrace)
    capi.dflash_debug_trace_draft_attn(eng.ctx, *qa)
    anchors2 = r["next_anchor"][:b].clone()
    dlog = torch.empty(b * 15 * s.vocab, dtype=torch.float32, device="cuda")
    capi.dflash_draft_block(eng.ctx, b, sid, anchors2, eng.block[: b * 16], 0, None, None, dlog)
    torch.cuda.synchronize()
    capi.dflash_debug_trace_draft(eng.ctx, None)
    capi.dflash_debug_trace_draft_attn(eng.ctx, None, None)
    q0 = int(np.argmax(out["accept_len"][:b]))  # the longest accepted path
    P2 = lengths[q0]
    res = dict(w=w, P=P, lo=lo, nmax=nmax, trees=trees, out=out, snap=snap, post=post,
               dpost=dpost, capture=capture, fused=fused, lengths=lengths, q0=q0, P2=P2,
               dq=qa[0][:, q0 * 16:(q0 + 1) * 16].float().cpu().numpy(),
               dao=qa[1][:, q0 * 16:(q0 + 1) * 16].float().cpu().numpy(),
               anchor2=int(anchors2[q0].item()),
               dtrace=dtrace[:, q0 * 16:(q0 + 1) * 16].cpu().numpy(),
               dlog=dlog.view(b, 15, -1)[q0].cpu().numpy(),
               dblock=eng.block[q0 * 16:(q0 + 1) * 16].cpu().numpy(),
               dctx={l: (eng.debug_view("dk_cache", l)[q0, :, :P2].float().cpu().numpy()
                         .transpose(1, 0, 2),
                         eng.debug_view("dv_cache", l)[q0, :, :P2].float().cpu().numpy()
                         .transpose(1, 0, 2)) for l in FORCED_DRAFT_LAYERS})
    eng.close()
    del eng, dtrace, qa, dlog
    torch.cuda.empty_cache()
    res["W"] = Weights(wl.SyntheticWeights(s, w.seed))
    return res


def _forced_path(r, q):
    t = r["trees"][q]
    return tree_accept(t, [int(v) for v in r["out"]["argmax"][q, : t.n_nodes]])


def test_forced_tree_walk_full_size(forced):
    best = 0
    for q in range(forced["w"].batch):
        t = forced["trees"][q]
        n = t.n_nodes
        assert list(forced["out"]["tok"][q, :n]) == t.tok
        a, path, emitted = _forced_path(forced, q)
        assert a == int(forced["out"]["accept_len"][q])
        assert emitted == [int(v) for v in forced["out"]["emitted"][q] if v >= 0]
        assert forced["lengths"][q] == forced["P"] + a + 1
        assert path[:4] == [0, 2, 3, 5][: a + 1]
        best = max(best, a)
    assert best >= 3, "no forced path was accepted"


def test_forced_tree_compaction_full_size(forced):
    """Every target layer: committed row P + j is the pre-commit row P + s_j,
    bit for bit; rows before P and past the path are untouched."""
    P, lo = forced["P"], forced["lo"]
    for q in range(forced["w"].batch):
        _, path, _ = _forced_path(forced, q)
        for (name, l), pre in forced["snap"].items():
            post = forced["post"][(name, l)][q]
            for j, node in enumerate(path):
                np.testing.assert_array_equal(post[:, P + j - lo], pre[q][:, P + node - lo],
                                              err_msg=f"seq {q} {name} {l} row {j}")
            np.testing.assert_array_equal(post[:, : P - lo], pre[q][:, : P - lo])
            np.testing.assert_array_equal(post[:, P + len(path) - lo:],
                                          pre[q][:, P + len(path) - lo:])


def test_forced_tree_injection_full_size(forced):
    """Draft cache rows P .. P + a of every draft layer hold the injection of
    the captured rows of the accepted nodes s_j at positions P + j (checked
    as F, then K / V from the GPU's F)."""
    w, P = forced["w"], forced["P"]
    s = w.shape
    for q in range(w.batch):
        a, path, _ = _forced_path(forced, q)
        rows = q * forced["nmax"] + np.array(path)
        kg = [forced["dpost"][("dk_cache", l)][q][:, : a + 1].transpose(1, 0, 2)
              for l in range(s.n_draft_layers)]
        vg = [forced["dpost"][("dv_cache", l)][q][:, : a + 1].transpose(1, 0, 2)
              for l in range(s.n_draft_layers)]
        check_injection(forced["W"], s, forced["capture"][rows], forced["fused"][rows],
                        P + np.arange(a + 1), kg, vg, f"seq {q}")
    forced["W"]._cache.clear()


@pytest.mark.parametrize("l", FORCED_DRAFT_LAYERS)
def test_next_draft_layers_after_tree_commit(forced, l):
    w = forced["w"]
    x = (draft_inputs(w.shape, w.seed, forced["anchor2"], 16) if l == 0
         else forced["dtrace"][l - 1].astype(np.float64))
    check_draft_layer(forced["W"], w.shape, l, x, forced["P2"], *forced["dctx"][l],
                      forced["dq"][l], forced["dao"][l], forced["dtrace"][l], f"next draft layer {l}")
    forced["W"]._cache.clear()


def test_next_draft_logits_after_tree_commit(forced):
    w = forced["w"]
    lg = lm_logits(w.shape, w.seed, forced["dtrace"][-1][1:], "draft.final_norm")
    check_close(forced["dlog"], lg, ATOL, RTOL, "next draft logits")
    check_argmax(forced["dblock"][1:], lg, "next drafted tokens")
