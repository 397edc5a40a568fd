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
from oracle.ddtree import DraftTree, build_tree, tree_accept
from oracle.decode import accept_longest_prefix
from oracle.models import Weights, _layer

from gpu_replay import check_argmax, check_close

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
    capi.dflash_debug_trace(eng.ctx, trace)
    out, dlog, vlog, _ = eng.step(sid, anchors, want_logits=True)
    torch.cuda.synchronize()
    capi.dflash_debug_trace(eng.ctx, None)
    picks = [(3, 0), (17, 9)]  # (sequence, block row)
    r = dict(w=w, prompts=prompts, lens=lens, picks=picks,
             block=out.block.cpu().numpy(), argmax=out.argmax.cpu().numpy(),
             accept=out.accept_len.cpu().numpy(), emitted=out.emitted.cpu().numpy(),
             length=eng.lengths(w.batch),
             vlog={(s, j): vlog[s, j].cpu().numpy() for s, j in picks},
             trace={(s, j): trace[:, s * 16 + j].cpu().numpy() for s, j in picks},
             cache={})
    for s, j in picks:
        n = lens[s] + 16
        for l in (0,) + B32_LAYERS:
            r["cache"][(s, l)] = (eng.debug_view("k_cache", l)[s, :, :n].float().cpu().numpy().transpose(1, 0, 2),
                                  eng.debug_view("v_cache", l)[s, :, :n].float().cpu().numpy().transpose(1, 0, 2))
    eng.close()
    del eng, trace, vlog
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
