"""Drafter and verifier in separate contexts (glossary "DFlash speculative
decoding", section "Practical meaning and deployment behaviour").

Every run here has one GPU, so both contexts sit on it; the hand-off is the
same device-to-device path a two-GPU run takes, minus the peer link.  The
split run must reproduce the single-context run bit for bit, because the
same kernels see the same inputs: the draft cache is filled from the
verifier's captured rows by explicit-row injection instead of the commit
queue, and the drafter's lengths move by dflash_advance_lengths instead of
a commit.  Checked per step: drafted blocks, target argmax, accept lengths,
next anchors, emitted tokens, and both sides' committed lengths.  One step
is teacher-forced to accept the whole block (the target's own greedy
continuation as the draft), so that 16 rows per sequence cross over and the
next draft reads all of them.  Grouped generation (two groups, the schedule
that overlaps drafting and verification on two GPUs) gives the greedy AR
tokens (lossless).
"""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu
LENS = [150, 37, 260]


def _prompts(vocab):
    rng = np.random.default_rng(11)
    return [rng.integers(0, vocab, size=n).astype(np.int32) for n in LENS]


@pytest.fixture(scope="module")
def setup():
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["mini_bf16_e2e"]
    prompts = _prompts(w.shape.vocab)
    eng = DFlashEngine(w.shape, w.block_size, len(LENS), 512, max_rows=max(LENS))
    ar = eng.generate(prompts, 3 * w.block_size + 4, mode="ar")
    return w, prompts, eng, ar


def _lengths(eng, b):
    return eng.lengths(b)


def test_split_steps_match_one_context(setup):
    from block_diffusion_speculative_injection_gb300.split import SplitDFlash
    w, prompts, eng, ar = setup
    b, B = len(LENS), w.block_size
    sid = eng.seq_ids(b)
    sp = SplitDFlash(w.shape, B, b, 512, max_rows=max(LENS))
    a1 = eng.prefill(prompts)
    a2 = sp.prefill(prompts)
    assert torch.equal(a1, a2)
    # the first step is forced to accept the whole block: its draft is the
    # target's own greedy continuation after the first anchor (ar[q][0])
    force = torch.tensor([ar[q][1:B] for q in range(b)], dtype=torch.int32, device="cuda")
    for k in range(4):
        ov = force if k == 0 else None
        o1 = eng.step(sid, a1, draft_override=ov)
        o2 = sp.step(sid, a2, draft_override=ov)
        for name in ("block", "argmax", "accept_len", "next_anchor", "emitted"):
            x, y = getattr(o1, name), getattr(o2, name)
            assert torch.equal(x.view(y.shape), y), (k, name)
        if k == 0:
            assert (o2.accept_len == B - 1).all()
        a1, a2 = o1.next_anchor.clone(), o2.next_anchor.clone()
        torch.cuda.synchronize()
        lv = sp.verifier.eng.lengths(b)
        ld = sp.drafter.eng.lengths(b)
        assert lv == ld == _lengths(eng, b), k
    sp.close()


def test_grouped_generation_is_lossless(setup):
    from block_diffusion_speculative_injection_gb300.split import SplitDFlash
    w, prompts, _, ar = setup
    n = 2 * w.block_size + 3
    sp = SplitDFlash(w.shape, w.block_size, len(LENS), 512, max_rows=max(LENS))
    assert sp.generate(prompts, n, groups=2) == [a[:n] for a in ar]
    assert sp.generate(prompts, n, groups=1) == [a[:n] for a in ar]
    sp.close()


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs a second GPU")
def test_calls_with_another_device_current_are_refused(setup):
    from block_diffusion_speculative_injection_gb300 import capi
    w, _, eng, _ = setup
    with torch.cuda.device(1):
        with pytest.raises(capi.DFlashError) as e:
            capi.dflash_reset_seq(eng.ctx, 0)
    assert e.value.status == 8


def test_split_tree_steps_match_one_context():
    """The DDTree step split the same way: the drafter drafts top-k and
    builds the tree, the tree arrays cross to the verifier, which runs the
    ancestor-masked verify and commits the accepted path (compaction of the
    target K/V in its own caches); the path rows' hidden states cross back
    for injection.  The first step is teacher-forced onto a tree whose path
    is the target's greedy continuation at slots s_j > j (accept length 6)."""
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    from block_diffusion_speculative_injection_gb300.split import SplitDFlash
    from gpu_replay import forced_tree, tree_arrays
    w = wl.WORKLOADS["mini_bf16_ddtree"]
    s, B = w.shape, w.block_size
    b, nmax = len(LENS), w.tree_budget + 1
    prompts = _prompts(s.vocab)
    mr = max(max(LENS), b * nmax)
    eng = DFlashEngine(s, B, b, 640, max_rows=mr, max_tree_nodes=nmax)
    ar = eng.generate(prompts, 9, mode="ar")
    sp = SplitDFlash(s, B, b, 640, max_rows=mr, max_tree_nodes=nmax)
    sid = eng.seq_ids(b)
    a1, a2 = eng.prefill(prompts), sp.prefill(prompts)
    assert torch.equal(a1, a2)
    forced = tree_arrays([forced_tree(ar[q][0], ar[q][1:7], ar[q][7], nmax, s.vocab, B - 1)
                          for q in range(b)], nmax)
    for k in range(3):
        ov = forced if k == 0 else None
        r1 = eng.tree_step(sid, a1, w.topk, w.tree_budget, tree_override=ov)
        r2 = sp.tree_step(sid, a2, w.topk, w.tree_budget, tree_override=ov)
        for n1, n2 in (("tok", "block"), ("argmax", "argmax"), ("accept_len", "accept_len"),
                       ("next_anchor", "next_anchor"), ("emitted", "emitted")):
            assert torch.equal(r1[n1].view(getattr(r2, n2).shape), getattr(r2, n2)), (k, n1)
        if k == 0:
            assert (r2.accept_len == 6).all()
        a1, a2 = r1["next_anchor"].clone(), r2.next_anchor.clone()
        torch.cuda.synchronize()
        assert sp.verifier.eng.lengths(b) == sp.drafter.eng.lengths(b) == eng.lengths(b), k
    sp.close()
    eng.close()
