"""The paged KV cache on the GPU.

The same generation runs twice on the bf16 mini model: once with every
sequence slot owning its own cache region (kv_pages = 0), once with all
pages drawn from one shared pool in scattered order (the slots reserve
128-slot pages round-robin, last slot first, so every sequence's pages are
non-contiguous and out of order, and key tiles straddle nothing but page
boundaries).  Only the addressing differs, so every result must be bit for
bit the same: the teacher-forced DDTree step (ancestor-masked verify, an
accepted path of 6 nodes, compaction that moves rows across pages, path
injection), the DFlash steps after it (draft and verify logits, argmax,
accept lengths, emitted tokens, lengths) and every target and draft layer's
cache, gathered through the page table.

Also: a pass over a sequence whose pages are not mapped is refused on the
device (DFLASH_E_CAPACITY from dflash_check) without touching other
sequences, and the context stays usable; the free-page count follows
reserve and release.
"""
import numpy as np
import pytest
import torch

import workloads as wl

from gpu_replay import forced_tree, tree_arrays

pytestmark = pytest.mark.gpu
PATH_LEN = 6
LENS = [300, 129, 250, 40]  # ragged: tiles cross page boundaries at different offsets
STEPS = 2


def _prompts(vocab):
    rng = np.random.default_rng(7)
    return [rng.integers(0, vocab, size=n).astype(np.int32) for n in LENS]


def _run(kv_pages, ar=None):
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["mini_bf16_ddtree"]
    s, B = w.shape, w.block_size
    b, nmax = len(LENS), w.tree_budget + 1
    prompts = _prompts(s.vocab)
    max_ctx = 640
    eng = DFlashEngine(s, B, b, max_ctx, max_rows=max(max(LENS), b * nmax), max_tree_nodes=nmax,
                       kv_pages=kv_pages)
    if ar is None:
        ar = eng.generate(prompts, PATH_LEN + 3, mode="ar")
    need = [n + (STEPS + 2) * B + nmax for n in LENS]
    if kv_pages:
        # scattered pages: one page per slot per round, last slot first
        for r in range(-(-max(need) // capi.PAGE_SLOTS)):
            for q in reversed(range(b)):
                eng.reserve(q, min(need[q], (r + 1) * capi.PAGE_SLOTS))
        tab = eng.page_table().cpu().numpy()
        assert any(np.any(np.diff(row[row >= 0]) != 1) for row in tab)
    sid = eng.seq_ids(b)
    anchors = eng.prefill(prompts)
    trees = [forced_tree(ar[q][0], ar[q][1:1 + PATH_LEN], ar[q][1 + PATH_LEN], nmax, s.vocab,
                         B - 1) for q in range(b)]
    r = eng.tree_step(sid, anchors, w.topk, w.tree_budget, want_logits=True,
                      tree_override=tree_arrays(trees, nmax))
    out = {f"tree_{k}": v.cpu().numpy() for k, v in r.items()}
    anchors = r["next_anchor"][:b].clone()
    for i in range(STEPS):
        o, dlog, vlog, margin = eng.step(sid, anchors, want_logits=True)
        out.update({f"s{i}_dlog": dlog.cpu().numpy(), f"s{i}_vlog": vlog.cpu().numpy(),
                    f"s{i}_argmax": o.argmax.cpu().numpy(), f"s{i}_acc": o.accept_len.cpu().numpy(),
                    f"s{i}_emit": o.emitted.cpu().numpy(), f"s{i}_margin": margin.cpu().numpy()})
        anchors = o.next_anchor.clone()
    torch.cuda.synchronize()
    lens = eng.lengths(b)
    out["lengths"] = np.array(lens)
    for l in range(s.n_layers):
        for nm_ in ("k_cache", "v_cache"):
            v = eng.debug_view(nm_, l)
            out[f"{nm_}{l}"] = [v[q, :, :lens[q]].float().cpu().numpy() for q in range(b)]
    for l in range(s.n_draft_layers):
        for nm_ in ("dk_cache", "dv_cache"):
            v = eng.debug_view(nm_, l)
            out[f"{nm_}{l}"] = [v[q, :, :lens[q]].float().cpu().numpy() for q in range(b)]
    free = eng.free_pages()
    eng.close()
    return out, ar, free


@pytest.fixture(scope="module")
def runs():
    w = wl.WORKLOADS["mini_bf16_ddtree"]
    B, nmax = w.block_size, w.tree_budget + 1
    flat, ar, _ = _run(0)
    pages = sum(-(-(n + (STEPS + 2) * B + nmax) // 128) for n in LENS)
    paged, _, free = _run(pages + 3, ar)
    return flat, paged, free, ar


def test_paged_run_is_bit_identical_to_fixed_regions(runs):
    flat, paged, free, _ = runs
    assert free == 3
    assert flat.keys() == paged.keys()
    for k in flat:
        a, b = flat[k], paged[k]
        if isinstance(a, list):  # caches: one [H_kv][length][hd] array per sequence
            assert len(a) == len(b) and all(np.array_equal(x, y) for x, y in zip(a, b)), k
        else:
            assert np.array_equal(a, b, equal_nan=True), k


def test_forced_tree_commit_moved_rows(runs):
    flat, _, _, ar = runs
    acc = flat["tree_accept_len"]
    assert np.all(acc >= 3), acc
    for q in range(len(LENS)):
        emitted = flat["tree_emitted"][q][: acc[q] + 1].tolist()
        assert emitted == ar[q][1:2 + acc[q]]


def test_unmapped_sequence_is_refused_on_the_device():
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["mini_bf16_e2e"]
    s, B = w.shape, w.block_size
    eng = DFlashEngine(s, B, 2, 1024, max_rows=256, kv_pages=4)
    assert eng.free_pages() == 4
    with pytest.raises(capi.DFlashError) as e:
        eng.reserve(0, 5 * capi.PAGE_SLOTS)  # more than the pool
    assert e.value.status == 2 and eng.free_pages() == 4
    prompt = _prompts(s.vocab)[1][:100]
    eng.prefill([prompt])  # slot 0: one page
    assert eng.free_pages() == 3
    # slot 1 was never given pages: its pass is skipped and flagged
    capi.dflash_reset_seq(eng.ctx, 1)
    sid = torch.tensor([1], dtype=torch.int32, device="cuda")
    toks = torch.from_numpy(prompt[:16].copy()).cuda()
    capi.dflash_verify(eng.ctx, 1, sid, toks, 16, None, capi.DFLASH_VERIFY_LAST_ONLY, eng.argmax)
    with pytest.raises(capi.DFlashError) as e:
        capi.dflash_check(eng.ctx)
    assert e.value.status == 2
    # the context goes on: map pages, run the same pass, nothing flagged
    eng.reserve(1, 16)
    capi.dflash_verify(eng.ctx, 1, sid, toks, 16, None, capi.DFLASH_VERIFY_LAST_ONLY, eng.argmax)
    capi.dflash_check(eng.ctx)
    assert eng.free_pages() == 2
    eng.release(0)
    eng.release(1)
    assert eng.free_pages() == 4
    assert (eng.page_table().cpu().numpy() == -1).all()
    eng.close()
