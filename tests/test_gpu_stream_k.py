"""The persistent GEMM's stream-K remainder is deterministic.

Qwen3-8B-shaped slice (two target layers, one draft layer), 32 sequences
with prompts of 512..1024 tokens: the prefill's QKV passes over more than 768
rows (192 tiles on 152 SMs) and the step's gate/up projection at 512 rows
(384 tiles) cut their last tiles along K over all CTAs, which trade fp32
partial sums through global memory.  CTAs take their work index from a
ticket, so the SM that runs a given range changes from launch to launch while
the ranges and the order of the sums do not: two runs on the same weights
and prompts must agree bit for bit in everything they produce (first
anchors, drafted block, target argmax and logits, draft logits, accept
lengths, and the K/V rows of every target and draft layer).  Parity with
the oracle on the same launch shapes is the full-size batch test's job.
"""
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def _run(w, weights):
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    prompts = wl.prompts(w)
    lens = [len(p) for p in prompts]
    eng = DFlashEngine(w.shape, w.block_size, w.batch, max(lens) + 64, max_rows=max(lens),
                       seed=w.seed, weights=weights)
    sid = eng.seq_ids(w.batch)
    anchors = eng.prefill(prompts)
    a0 = anchors.clone()
    out, dlog, vlog, _ = eng.step(sid, anchors, want_logits=True)
    torch.cuda.synchronize()
    r = {"anchors": a0, "block": out.block.clone(), "argmax": out.argmax.clone(),
         "accept": out.accept_len.clone(), "emitted": out.emitted.clone(),
         "vlog": vlog.clone(), "dlog": dlog.clone(),
         "lengths": torch.tensor(eng.lengths(w.batch))}
    for l in range(w.shape.n_layers):
        r[f"k{l}"] = eng.debug_view("k_cache", l).clone()
        r[f"v{l}"] = eng.debug_view("v_cache", l).clone()
    for l in range(w.shape.n_draft_layers):
        r[f"dk{l}"] = eng.debug_view("dk_cache", l).clone()
        r[f"dv{l}"] = eng.debug_view("dv_cache", l).clone()
    keep = eng.weights
    eng.close()
    return r, keep


def test_stream_k_launches_are_deterministic():
    w = wl.WORKLOADS["qwen3_8b_slice_b32"]
    first, weights = _run(w, None)
    second, _ = _run(w, weights)
    assert first.keys() == second.keys()
    for k in first:
        assert torch.equal(first[k], second[k]), k
