"""GPU parity of whole DFlash / DDTree steps through the C ABI against the
CPU oracle, at sizes the oracle finishes in seconds (several GEMM tiles,
ragged prompt lengths, a vocabulary that is not a multiple of the tile).

Tolerances: fp32 model -- logits within 1e-4 (abs and rel); bf16 models --
within max-abs 2e-2 and relative 1e-2 of the oracle's bf16-emulation mode.
Token ids and accept lengths must match wherever the oracle's top-1/top-2
margin exceeds 1e-2; accept decisions must follow the rule exactly.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle.models import Weights
from oracle.numerics import Precision

from gpu_replay import replay_linear, replay_tree

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def engine_mod():
    from block_diffusion_speculative_injection_gb300 import engine
    return engine


def test_tiny_f32_dflash_replay(engine_mod):
    w = wl.WORKLOADS["tiny_f32_e2e"]
    prompts = wl.prompts(w)
    eng = engine_mod.DFlashEngine(w.shape, w.block_size, 1, 256, max_rows=128)
    W = Weights(wl.SyntheticWeights(w.shape))
    seqs, st = replay_linear(eng, W, w.shape, Precision("exact"), prompts, 6, 1e-4, 1e-4, 256)
    assert st["checked"] > 100
    eng.close()


def test_tiny_f32_generate_equals_oracle_ar(engine_mod):
    from oracle.decode import greedy_ar
    w = wl.WORKLOADS["tiny_f32_e2e"]
    prompt = wl.prompts(w)[0]
    eng = engine_mod.DFlashEngine(w.shape, w.block_size, 1, 256, max_rows=128)
    got = eng.generate([prompt], w.new_tokens)[0]
    ar_gpu = eng.generate([prompt], w.new_tokens, mode="ar")[0]
    W = Weights(wl.SyntheticWeights(w.shape))
    ref = greedy_ar(W, w.shape, Precision("exact"), prompt, w.new_tokens)
    # lossless: speculative output = GPU AR output = oracle AR output
    assert got == ar_gpu == ref
    eng.close()


def test_mini_bf16_dflash_replay_ragged_batch(engine_mod):
    w = wl.WORKLOADS["mini_bf16_e2e"]
    prompts = wl.prompts(w)
    assert len(set(len(p) for p in prompts)) > 1
    eng = engine_mod.DFlashEngine(w.shape, w.block_size, w.batch, 512, max_rows=256)
    W = Weights(wl.SyntheticWeights(w.shape))
    seqs, st = replay_linear(eng, W, w.shape, Precision("bf16emu"), prompts, 4, 2e-2, 1e-2, 512)
    assert st["checked"] > 200
    eng.close()


def test_mini_bf16_wide_vocab_and_single_inject(engine_mod):
    s = wl.MINI_BF16_WIDE
    w = wl.Workload("mini_wide", s, 16, 2, (33, 77), 16)
    prompts = wl.prompts(w)
    eng = engine_mod.DFlashEngine(s, 16, 2, 256, max_rows=128)
    W = Weights(wl.SyntheticWeights(s))
    replay_linear(eng, W, s, Precision("bf16emu"), prompts, 3, 2e-2, 1e-2, 256)
    eng.close()


def test_mini_bf16_teacher_forced_full_acceptance(engine_mod):
    """A draft equal to the target's greedy continuation is accepted whole:
    tau = B every step (the full-acceptance reading of the acceptance rule)."""
    w = wl.WORKLOADS["mini_bf16_e2e"]
    prompt = wl.prompts(w)[0]
    eng = engine_mod.DFlashEngine(w.shape, 16, 1, 512, max_rows=256)
    ar = eng.generate([prompt], 3 * 16 + 2, mode="ar")[0]
    sid = eng.seq_ids(1)
    anchors = eng.prefill([prompt])
    pos = 0
    for _ in range(3):
        forced = torch.tensor([ar[pos + 1: pos + 16]], dtype=torch.int32, device="cuda")
        out = eng.step(sid, anchors, draft_override=forced)
        torch.cuda.synchronize()
        assert int(out.accept_len[0]) == 15
        assert out.emitted[0].tolist() == ar[pos + 1: pos + 17]
        anchors = out.next_anchor.clone()
        pos += 16
    eng.close()


def test_mini_bf16_ddtree_replay(engine_mod):
    w = wl.WORKLOADS["mini_bf16_ddtree"]
    prompts = wl.prompts(w)
    eng = engine_mod.DFlashEngine(w.shape, w.block_size, w.batch, 512, max_rows=256,
                                  max_tree_nodes=w.tree_budget + 1)
    W = Weights(wl.SyntheticWeights(w.shape))
    replay_tree(eng, W, w.shape, Precision("bf16emu"), prompts, 2, w.topk, w.tree_budget,
                2e-2, 1e-2, 512)
    eng.close()


def test_block_size_one_is_ar(engine_mod):
    w = wl.WORKLOADS["mini_bf16_e2e"]
    prompt = wl.prompts(w)[1]
    eng1 = engine_mod.DFlashEngine(w.shape, 1, 1, 512, max_rows=256)
    a = eng1.generate([prompt], 12)[0]
    b = eng1.generate([prompt], 12, mode="ar")[0]
    assert a == b
    eng1.close()


def test_capacity_overflow_sets_device_status(engine_mod):
    """A sequence that would pass max_ctx is skipped on the device and the
    sticky status reports it (no fault, no out-of-bounds write)."""
    from block_diffusion_speculative_injection_gb300 import capi
    w = wl.WORKLOADS["tiny_f32_e2e"]
    eng = engine_mod.DFlashEngine(w.shape, 16, 1, 80, max_rows=128)
    eng.prefill([wl.prompts(w)[0]])  # 64 tokens
    capi.dflash_check(eng.ctx)
    sid = eng.seq_ids(1)
    toks = torch.zeros(32, dtype=torch.int32, device="cuda")
    capi.dflash_verify(eng.ctx, 1, sid, toks, 32, None, 0, eng.argmax)
    with pytest.raises(capi.DFlashError) as e:
        capi.dflash_check(eng.ctx)
    assert e.value.status == 2
    assert eng.argmax[:32].cpu().tolist() == [-1] * 32
    eng.close()


def test_expired_device_wait_is_reported_and_context_survives(engine_mod):
    """A bounded device wait that runs out (a barrier nothing completes)
    records DFLASH_E_TIMEOUT in the sticky status; the context then runs a
    normal step and checks clean."""
    from block_diffusion_speculative_injection_gb300 import capi
    w = wl.WORKLOADS["tiny_f32_e2e"]
    eng = engine_mod.DFlashEngine(w.shape, w.block_size, 1, 256, max_rows=128)
    anchors = eng.prefill([wl.prompts(w)[0]])
    capi.dflash_check(eng.ctx)
    capi.dflash_debug_wait_timeout(eng.ctx)
    with pytest.raises(capi.DFlashError) as e:
        capi.dflash_check(eng.ctx)
    assert e.value.status == 6  # DFLASH_E_TIMEOUT
    out = eng.step(eng.seq_ids(1), anchors)
    capi.dflash_check(eng.ctx)
    assert int(out.accept_len[0]) >= 0
    eng.close()


def test_block_size_per_step_is_lossless(engine_mod):
    """Greedy output does not depend on the block size of each step: a fixed
    schedule of block sizes and the adaptive policy both emit the oracle's
    greedy AR tokens."""
    from oracle.decode import greedy_ar
    w = wl.WORKLOADS["tiny_f32_e2e"]
    prompt = wl.prompts(w)[0]
    eng = engine_mod.DFlashEngine(w.shape, w.block_size, 1, 256, max_rows=128)
    sched = [w.block_size, 5, 1, 9, 2, w.block_size, 3]
    got = eng.generate([prompt], w.new_tokens, block_schedule=sched)[0]
    assert eng.B == w.block_size  # restored after the run
    adaptive = eng.generate([prompt], w.new_tokens, mode="adaptive")[0]
    W = Weights(wl.SyntheticWeights(w.shape))
    ref = greedy_ar(W, w.shape, Precision("exact"), prompt, w.new_tokens)
    assert got == ref
    assert adaptive == ref
    eng.close()


def test_set_block_size_bounds(engine_mod):
    from block_diffusion_speculative_injection_gb300 import capi
    w = wl.WORKLOADS["tiny_f32_e2e"]
    eng = engine_mod.DFlashEngine(w.shape, w.block_size, 1, 256, max_rows=128)
    for bad in (0, -1, w.block_size + 1):
        with pytest.raises(capi.DFlashError) as e:
            capi.dflash_set_block_size(eng.ctx, bad)
        assert e.value.status == 1
    capi.dflash_set_block_size(eng.ctx, 1)
    capi.dflash_set_block_size(eng.ctx, w.block_size)
    eng.close()
