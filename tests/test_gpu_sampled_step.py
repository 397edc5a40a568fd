"""The temperature-1 DFlash step end to end (DFlashEngine.sample_step: draft
pass, draws from the drafter's softmax, verify pass, speculative rejection
test, commit of the accepted prefix and the drawn token, injection) replayed
against the oracle on the fp32 model, step by step.

Each step checks the drafter's and the target's logits (1e-4), every draft
draw and the accept decision against oracle.sampling on the oracle's own
logits and the same uniforms, then commits the GPU's decision on both sides.
A decision within 1e-3 (relative) of a tie may go either way; the GPU's
choice must then still be valid for the oracle's distributions.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle.models import Weights
from oracle.numerics import Precision
from oracle.sampling import sample_row, softmax, spec_accept

from gpu_replay import check_close, replay_prefill

pytestmark = pytest.mark.gpu

BAND = 1e-3


def _draw_ok(w, u, got, want):
    if got == want:
        return True
    if not 0 <= got < len(w) or w[got] <= 0:
        return False
    c = np.cumsum(w)
    t = float(u) * c[-1]
    lo = c[got - 1] if got > 0 else 0.0
    return lo - BAND * c[-1] <= t <= c[got] + BAND * c[-1]


def test_tiny_f32_sampled_step_replay():
    from block_diffusion_speculative_injection_gb300 import engine
    w = wl.WORKLOADS["tiny_f32_e2e"]
    prompts = wl.prompts(w)
    B = w.block_size
    eng = engine.DFlashEngine(w.shape, B, 1, 256, max_rows=128)
    W = Weights(wl.SyntheticWeights(w.shape))
    prec = Precision("exact")
    sid = eng.seq_ids(1)
    anchors, seqs = replay_prefill(eng, W, w.shape, prec, prompts[:1], 256, 1e-4, 1e-4)
    exact = accepted = 0
    for step in range(8):
        ud, ua, ur = wl.step_uniforms(step, 1, B)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        out = eng.sample_step(sid, anchors, t(ud), t(ua), t(ur))
        torch.cuda.synchronize()
        V = w.shape.vocab
        blk = [int(x) for x in out.block.cpu().numpy()[0]]
        dl = eng._samp["dlog"][: (B - 1) * V].view(B - 1, V).cpu().numpy()
        vl = eng._samp["vlog"][: B * V].view(B, V).cpu().numpy()
        a_gpu, tok_gpu = int(out.accept_len[0]), int(out.next_anchor[0])
        em = [int(x) for x in out.emitted.cpu().numpy()[0] if x >= 0]
        sq = seqs[0]
        odl = sq.draft(blk[0], B)
        check_close(dl, odl, 1e-4, 1e-4, f"step {step} draft logits")
        for j in range(1, B):
            want = sample_row(odl[j - 1], float(ud[0, j - 1]))
            assert _draw_ok(softmax(odl[j - 1]), ud[0, j - 1], blk[j], want), (step, j, blk[j], want)
        ovl, cap = sq.verify(blk)
        check_close(vl, ovl, 1e-4, 1e-4, f"step {step} verify logits")
        dpad = np.vstack([np.zeros((1, V)), odl])
        a_or, tok_or = spec_accept(dpad, ovl, blk, ua[0], float(ur[0]))
        p, q = softmax(dpad), softmax(ovl)
        for j in range(1, B):  # every test before a_gpu passed, the one at a_gpu failed (or a tie)
            lhs, rhs = float(ua[0, j]) * p[j, blk[j]], q[j - 1, blk[j]]
            tie = abs(lhs - rhs) <= BAND * max(lhs, rhs)
            if j <= a_gpu:
                assert lhs < rhs or tie, (step, j)
            elif j == a_gpu + 1:
                assert not (lhs < rhs) or tie, (step, j)
        if a_gpu == a_or:
            wdraw = np.maximum(q[a_gpu] - p[a_gpu + 1], 0.0) if a_gpu < B - 1 else q[B - 1]
            assert _draw_ok(wdraw if wdraw.sum() > 0 else q[a_gpu], ur[0], tok_gpu, tok_or)
            exact += 1
        # the commit: emitted = accepted drafts + the drawn token; lengths agree
        assert em == blk[1: a_gpu + 1] + [tok_gpu]
        sq.commit_linear(cap, a_gpu)
        accepted += a_gpu
        anchors = out.next_anchor.clone()
        assert eng.lengths(1) == [sq.length]
    assert exact >= 7
    eng.close()
