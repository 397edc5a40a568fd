"""The paged KV cache at the Qwen3-8B shape (36 + 5 layers, 8 KV heads).

Two sequences with ragged prompts (700 and 1290 tokens) run prefill and
three DFlash steps twice, on one set of weights: once with fixed per-slot
regions, once with the pages of both sequences drawn from a shared pool in
scattered order (one page per sequence per round, last sequence first).  The
first step is teacher-forced to accept the whole block (the target's own
greedy continuation as the draft), so the injection writes 16 rows per
sequence across page boundaries.  Only the addressing differs, so every
result is required bit for bit: drafted blocks, target argmax and margins,
accept lengths, emitted tokens, lengths, and the K/V rows of sampled target
and draft layers up to each sequence's length.

The attention planner sizes its key split for the longest context a pass
can see (max_ctx with fixed regions, the slots of the largest mapping when
paged), and the split sets the summation order; the longer sequence is
therefore mapped up to max_ctx, so both runs plan the same splits.
"""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu
LENS = (700, 1290)
B = 16
MAX_CTX = 1536


def _need():
    # slots each sequence maps: three steps' growth, the longest up to max_ctx
    need = [n + 4 * B + 16 for n in LENS]
    need[LENS.index(max(LENS))] = MAX_CTX
    return need


def _run(w, weights, kv_pages, force):
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    b = len(LENS)
    eng = DFlashEngine(w.shape, B, b, MAX_CTX, max_rows=max(LENS), seed=w.seed, weights=weights,
                       kv_pages=kv_pages)
    if kv_pages:
        need = _need()
        for r in range(-(-max(need) // capi.PAGE_SLOTS)):
            for q in reversed(range(b)):
                eng.reserve(q, min(need[q], (r + 1) * capi.PAGE_SLOTS))
    prompts = [wl.prompt_tokens(w, q, n) for q, n in enumerate(LENS)]
    sid = eng.seq_ids(b)
    anchors = eng.prefill(prompts)
    out = {"anchors0": anchors.cpu().numpy()}
    for k in range(3):
        o, _, vlog, margin = eng.step(sid, anchors, want_logits=True,
                                      draft_override=force if k == 0 else None)
        out.update({f"s{k}_block": o.block.cpu().numpy(), f"s{k}_argmax": o.argmax.cpu().numpy(),
                    f"s{k}_margin": margin.cpu().numpy(), f"s{k}_acc": o.accept_len.cpu().numpy(),
                    f"s{k}_emit": o.emitted.cpu().numpy()})
        anchors = o.next_anchor.clone()
    torch.cuda.synchronize()
    lens = eng.lengths(b)
    out["lengths"] = np.array(lens)
    caches = {}
    for nm_, layers in (("k_cache", (0, 17, 35)), ("v_cache", (0, 35)), ("dk_cache", (0, 4)),
                        ("dv_cache", (4,))):
        for l in layers:
            v = eng.debug_view(nm_, l)
            caches[(nm_, l)] = [v[q, :, :lens[q]].cpu() for q in range(b)]
    free = eng.free_pages()
    eng.close()
    return out, caches, free


def test_full_size_paged_steps_are_bit_identical():
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["qwen3_8b_b1"]
    b = len(LENS)
    ref = DFlashEngine(w.shape, B, b, MAX_CTX, max_rows=max(LENS), seed=w.seed)
    prompts = [wl.prompt_tokens(w, q, n) for q, n in enumerate(LENS)]
    ar = ref.generate(prompts, B + 2, mode="ar")
    weights = ref.weights
    ref.close()
    force = torch.tensor([a[1:B] for a in ar], dtype=torch.int32, device="cuda")
    pages = sum(-(-n // 128) for n in _need())
    flat, cflat, _ = _run(w, weights, 0, force)
    paged, cpaged, free = _run(w, weights, pages + 5, force)
    assert free == 5
    assert (flat["s0_acc"] == B - 1).all()
    for k in flat:
        assert np.array_equal(flat[k], paged[k], equal_nan=True), k
    for key in cflat:
        for q in range(b):
            assert torch.equal(cflat[key][q], cpaged[key][q]), (key, q)
