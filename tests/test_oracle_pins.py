"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks one oracle function against what the pages or the
mathematics fix: hand-derived cases of the stated rules (tests/golden),
closed forms, library routines for textbook special cases, invariants, and
brute force on tiny inputs.  Chosen so that a plausible mistake (a dropped
term, a sign, an index, a transposed operand) fails at least one of them.
"""
import dataclasses
import itertools
import os

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import numerics as nm
from oracle.ddtree import (build_tree, ddtree_generate, tree_accept, tree_verify,
                           tree_commit, topk_logprobs)
from oracle.decode import (Sequence1, accept_longest_prefix, dflash_generate, greedy_ar,
                           speedup_model)
from oracle.models import (KVCache, Weights, causal_visible, draft_block_logits, inject_kv,
                           target_forward)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = wl.WORKLOADS["tiny_f32_e2e"]


@pytest.fixture(scope="module")
def tiny_w():
    return Weights(wl.SyntheticWeights(TINY.shape))


@pytest.fixture(scope="module")
def tiny_prompt():
    return wl.prompts(TINY)[0]


# --------------------------------------------------------------------------
# numerics: library routines and closed forms
# --------------------------------------------------------------------------

def test_round_bf16_matches_torch_bfloat16():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 8, 20000),
                        # exact halfway points between bf16 neighbours: ties to even
                        (np.arange(1, 513, dtype=np.float64) * 2 + 1) * 2.0 ** -9])
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(nm.round_bf16(x32.astype(np.float64)), ref)


def test_rmsnorm_against_torch_and_closed_form():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 37))
    g = rng.standard_normal(37)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (37,), torch.from_numpy(g),
                                       eps=1e-6).numpy()
    np.testing.assert_allclose(nm.rmsnorm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-12)
    # constant vector c*1: output = c / sqrt(c^2 + eps) per element
    c = 0.37
    y = nm.rmsnorm(np.full((1, 8), c), np.ones(8), 1e-6)
    np.testing.assert_allclose(y, c / np.sqrt(c * c + 1e-6), rtol=1e-14)


def test_rope_is_complex_rotation():
    """Rotate-half RoPE = multiplying z_i = x_i + 1j*x_{i+hd/2} by
    exp(1j * pos * theta^(-2i/hd)) (complex-number formulation)."""
    rng = np.random.default_rng(2)
    hd, theta = 16, 1e4
    x = rng.standard_normal((6, 3, hd))
    pos = np.array([0, 1, 2, 17, 511, 4095])
    y = nm.apply_rope(x, pos, theta)
    z = x[..., : hd // 2] + 1j * x[..., hd // 2:]
    freq = theta ** (-np.arange(hd // 2) * 2.0 / hd)
    z = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    np.testing.assert_allclose(y, np.concatenate([z.real, z.imag], -1), atol=1e-12)
    np.testing.assert_array_equal(nm.apply_rope(x[:1], np.array([0]), theta), x[:1])


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    s = [float(np.sum(nm.apply_rope(q, np.array([m + c]), 1e6) *
                      nm.apply_rope(k, np.array([n + c]), 1e6)))
         for (m, n) in [(10, 3), (5, 9)] for c in (0, 1000)]
    assert abs(s[0] - s[1]) < 1e-9 and abs(s[2] - s[3]) < 1e-9
    assert abs(s[0] - s[2]) > 1e-3


def test_silu_against_scipy():
    from scipy.special import expit
    x = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(nm.silu(x), x * expit(x), rtol=1e-13, atol=1e-300)


def test_linear_convention_is_w_times_x():
    w = np.zeros((3, 4))
    w[2, 1] = 5.0  # output feature 2 reads input feature 1
    y = nm.linear(np.array([[0.0, 1.0, 0.0, 0.0]]), w)
    np.testing.assert_array_equal(y, [[0.0, 0.0, 5.0]])


@pytest.mark.parametrize("n_heads,n_kv", [(4, 4), (8, 2), (32, 8)])
def test_attend_against_torch_sdpa(n_heads, n_kv):
    rng = np.random.default_rng(4)
    hd, n = 32, 23
    q = rng.standard_normal((n_heads, hd))
    k = rng.standard_normal((n, n_kv, hd))
    v = rng.standard_normal((n, n_kv, hd))
    out = nm.attend(q, k, v)
    rep = n_heads // n_kv
    tq = torch.from_numpy(q)[:, None, :]                       # [H, 1, hd]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(rep, 0)  # [H, n, hd]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(rep, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[:, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_attend_special_cases():
    rng = np.random.default_rng(5)
    k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 8))
    # a single key: output is its value row
    np.testing.assert_allclose(nm.attend(rng.standard_normal((4, 8)), k, v),
                               np.repeat(v[0], 2, axis=0), atol=1e-15)
    # zero query: uniform weights, output is the mean value
    k5, v5 = rng.standard_normal((5, 1, 8)), rng.standard_normal((5, 1, 8))
    np.testing.assert_allclose(nm.attend(np.zeros((1, 8)), k5, v5)[0], v5[:, 0].mean(0),
                               atol=1e-14)


def test_argmax_ties_and_margin():
    assert nm.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert nm.top2_margin(np.array([1.0, 3.0, 2.5])) == 0.5
    lp = nm.log_softmax(np.array([0.0, np.log(3.0)]))
    np.testing.assert_allclose(np.exp(lp), [0.25, 0.75], rtol=1e-14)


def test_topk_ties_go_to_lower_id():
    ids, lp = topk_logprobs(np.array([0.0, 2.0, 1.0, 2.0, -1.0]), 3)
    assert list(ids) == [1, 3, 2]
    np.testing.assert_allclose(np.exp(lp.astype(np.float64)).sum(),
                               (2 * np.exp(2) + np.exp(1)) / (np.exp(0) + 2 * np.exp(2) + np.exp(1) + np.exp(-1)),
                               rtol=1e-6)


# --------------------------------------------------------------------------
# workload readings
# --------------------------------------------------------------------------

def test_injected_layers_evenly_spaced():
    assert wl.evenly_spaced_layers(36, 5) == wl.QWEN3_8B.inject_layers == (0, 9, 18, 26, 35)
    assert wl.evenly_spaced_layers(32, 5) == wl.LLAMA31_8B.inject_layers == (0, 8, 16, 23, 31)


def test_generator_rows_are_distinct_pool_windows():
    w = wl.SyntheticWeights(wl.TINY)
    a = w["lm_head"]
    assert a.shape == (1024, 256) and a.dtype == np.float32
    assert len({r.tobytes() for r in a}) == a.shape[0]
    assert abs(float(a.std()) - 0.02) < 0.002
    np.testing.assert_array_equal(w["final_norm"], 1.0)


# --------------------------------------------------------------------------
# transformer invariants
# --------------------------------------------------------------------------

def _prefill_logits(w, shape, prompt, positions=None):
    p = len(prompt)
    cache = KVCache(shape.n_layers, p, shape.n_kv_heads, shape.head_dim)
    pos = np.arange(p) if positions is None else positions
    logits, cap = target_forward(w, shape, nm.Precision("exact"), cache, prompt, pos,
                                 np.arange(p), causal_visible(0, p))
    return logits, cap, cache


def test_zero_branch_weights_leave_residual_unchanged(tiny_w, tiny_prompt):
    s = TINY.shape
    over = {}
    for l in range(s.n_layers):
        over[f"layers.{l}.wo"] = np.zeros((s.d_model, s.q_dim), np.float32)
        over[f"layers.{l}.w_down"] = np.zeros((s.d_model, s.ffn_dim), np.float32)
    w = Weights(wl.SyntheticWeights(s).with_override(over))
    logits, cap, _ = _prefill_logits(w, s, tiny_prompt[:5])
    emb = w["tok_emb"][tiny_prompt[:5]]
    np.testing.assert_allclose(cap[:, 0], emb, atol=0)
    ref = nm.linear(nm.rmsnorm(emb, np.ones(s.d_model), s.rms_eps), w["lm_head"])
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name", ["tiny_f32_e2e", "mini_bf16_e2e"])  # MHA, and GQA 8 / 2
def test_attention_branch_with_zero_scores_is_a_causal_mean(name):
    """W_q = W_k = 0 makes every score 0, so each query head takes the plain
    mean of the V rows it may see (rows 0..i); with the FFN switched off
    (W_down = 0) layer 0 must give x + W_o . mean(V), V = W_v . RMSNorm(x),
    query head h reading KV head h // (H / H_kv).  Pins the pre-norm, the GQA
    mapping, the output projection and the residual add of the attention
    branch against a formula without softmax or RoPE."""
    s = wl.WORKLOADS[name].shape
    prompt = wl.prompts(wl.WORKLOADS[name])[0]
    over = {"layers.0.wq": np.zeros((s.q_dim, s.d_model), np.float32),
            "layers.0.wk": np.zeros((s.n_kv_heads * s.head_dim, s.d_model), np.float32),
            "layers.0.w_down": np.zeros((s.d_model, s.ffn_dim), np.float32)}
    w = Weights(wl.SyntheticWeights(s).with_override(over))
    t = 6
    _, cap, _ = _prefill_logits(w, s, prompt[:t])
    x = w["tok_emb"][prompt[:t]]
    h = nm.rmsnorm(x, np.ones(s.d_model), s.rms_eps)
    v = (h @ w["layers.0.wv"].T).reshape(t, s.n_kv_heads, s.head_dim)
    mean = np.cumsum(v, axis=0) / np.arange(1, t + 1)[:, None, None]
    group = s.n_heads // s.n_kv_heads
    o = np.repeat(mean, group, axis=1).reshape(t, s.q_dim)
    want = x + o @ w["layers.0.wo"].T
    np.testing.assert_allclose(cap[:, 0], want, rtol=1e-10, atol=1e-12)


def test_ffn_branch_alone_is_swiglu_of_the_normed_residual(tiny_w, tiny_prompt):
    """W_o = 0 switches the attention branch off: layer 0 must give
    x + W_down . (SiLU(W_gate . n) * (W_up . n)), n = RMSNorm(x), with SiLU
    from scipy.  Pins the FFN's norm placement, the SwiGLU order (SiLU on the
    gate, not the up projection) and the residual add."""
    from scipy.special import expit
    s = TINY.shape
    w = Weights(wl.SyntheticWeights(s).with_override(
        {"layers.0.wo": np.zeros((s.d_model, s.q_dim), np.float32)}))
    t = 5
    _, cap, _ = _prefill_logits(w, s, tiny_prompt[:t])
    x = w["tok_emb"][tiny_prompt[:t]]
    n = nm.rmsnorm(x, np.ones(s.d_model), s.rms_eps)
    g = n @ w["layers.0.w_gate"].T
    u = n @ w["layers.0.w_up"].T
    want = x + ((g * expit(g)) * u) @ w["layers.0.w_down"].T
    np.testing.assert_allclose(cap[:, 0], want, rtol=1e-10, atol=1e-12)


def test_causal_prefix_unchanged_by_later_tokens(tiny_w, tiny_prompt):
    s = TINY.shape
    p = tiny_prompt[:12].copy()
    l1, _, _ = _prefill_logits(tiny_w, s, p)
    p[9] = (p[9] + 1) % s.vocab
    l2, _, _ = _prefill_logits(tiny_w, s, p)
    np.testing.assert_array_equal(l1[:9], l2[:9])
    assert np.abs(l1[9:] - l2[9:]).max() > 1e-6


def test_logits_invariant_to_global_position_shift(tiny_w, tiny_prompt):
    s = TINY.shape
    p = tiny_prompt[:10]
    l1, _, _ = _prefill_logits(tiny_w, s, p)
    l2, _, _ = _prefill_logits(tiny_w, s, p, positions=np.arange(10) + 777)
    np.testing.assert_allclose(l1, l2, rtol=1e-9, atol=1e-9)


def test_prefill_rows_equal_incremental_decode_bitwise(tiny_w, tiny_prompt):
    """Row independence: the verify pass over a block gives bitwise the same
    logits as one-token steps over the same tokens."""
    s = TINY.shape
    p = list(tiny_prompt[:20])
    full, _, _ = _prefill_logits(tiny_w, s, p)
    seq = Sequence1(tiny_w, s, nm.Precision("exact"), 32)
    seq.prefill(p[:8], inject=False)
    rows = []
    for t in p[8:]:
        lg, _ = seq.verify([t])
        seq.length += 1
        rows.append(lg[0])
    np.testing.assert_array_equal(np.stack(rows), full[8:])


def test_injection_selects_layers_in_concat_order(tiny_w):
    """With W_fuse = [0 | I] only the second injected layer's feature reaches
    the draft K/V, and K is the roped Wk projection of that feature."""
    s = TINY.shape
    d = s.d_model
    fuse = np.concatenate([np.zeros((d, d)), np.eye(d)], axis=1).astype(np.float32)
    w = Weights(wl.SyntheticWeights(s).with_override({"draft.fuse": fuse}))
    rng = np.random.default_rng(6)
    cap = rng.standard_normal((3, 2, d)) * 0.1
    dc = KVCache(s.n_draft_layers, 8, s.n_kv_heads, s.head_dim)
    inject_kv(w, s, nm.Precision("exact"), dc, cap, np.array([2, 3, 5]))
    wk = w["draft.layers.0.wk"]
    wv = w["draft.layers.0.wv"]
    h = cap[:, 1]
    k = nm.apply_rope((h @ wk.T).reshape(3, s.n_kv_heads, s.head_dim), np.array([2, 3, 5]),
                      s.rope_theta)
    np.testing.assert_allclose(dc.k[0, [2, 3, 5]], k, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dc.v[0, [2, 3, 5]],
                               (h @ wv.T).reshape(3, s.n_kv_heads, s.head_dim), atol=1e-14)
    assert np.all(dc.k[0, [0, 1, 4]] == 0)


def test_draft_block_is_bidirectional(tiny_w, tiny_prompt):
    """Bidirectional block attention: slot 1's logits change when later mask
    slots are added to the block (under a causal mask they could not)."""
    from oracle.models import draft_block_logits
    s = TINY.shape
    prec = nm.Precision("exact")
    seq = Sequence1(tiny_w, s, prec, 64)
    seq.prefill(tiny_prompt[:16], inject=True)
    a = draft_block_logits(tiny_w, s, prec, seq.dcache, 5, 16, 4)
    b = draft_block_logits(tiny_w, s, prec, seq.dcache, 5, 16, 3)
    assert a.shape == (3, s.vocab) and b.shape == (2, s.vocab)
    assert np.abs(a[0] - b[0]).max() > 1e-6
    # the injected context matters: an empty context gives other logits
    c = draft_block_logits(tiny_w, s, prec, seq.dcache, 5, 0, 4)
    assert np.abs(a - c).max() > 1e-6


# --------------------------------------------------------------------------
# the draft pass: closed-form special cases (Deep Research Report, "Key
# points": B masked positions drafted in one pass over the injected context;
# "Why DFlash beats EAGLE-3" item 3 and the MTP table: bidirectional block)
# --------------------------------------------------------------------------

def _one_layer_draft_shape(base):
    return dataclasses.replace(base, name=base.name + "_d1", n_draft_layers=1, dtype="f32")


def _draft_context(w, s, P, seed):
    """Draft cache holding P injected context rows built from seeded capture
    rows (the injection itself is pinned above)."""
    rng = np.random.default_rng(seed)
    hcat = rng.standard_normal((P, s.n_inject, s.d_model)) * 0.1
    dc = KVCache(s.n_draft_layers, P + 64, s.n_kv_heads, s.head_dim)
    inject_kv(w, s, nm.Precision("exact"), dc, hcat, np.arange(P))
    return hcat, dc


@pytest.mark.parametrize("base", [TINY.shape, wl.MINI_BF16], ids=["mha", "gqa4"])
@pytest.mark.parametrize("zero", ["wq", "wk"])
def test_draft_layer_with_zero_scores_is_a_mean_over_context_and_block(base, zero):
    """W_q = 0 (or W_k = 0, which also zeroes the injected context keys) makes
    every score 0, so every block slot takes the plain mean of all P injected
    V rows and all B block V rows: no mask in the block or on the context.
    With W_down = 0 the one draft layer gives x + W_o . mean(V) with
    x = [E[anchor]; e_mask x (B-1)], block V = W_v . RMSNorm_g(x) (the draft
    layer's own W_v and norm), context V = W_v . W_fuse . h_cat, query head h
    reading KV head h // (H / H_kv); the logits of slots 1..B-1 are the shared
    lm_head over the drafter's own final norm.  Non-unit norm gains make the
    choice of gain visible."""
    s = _one_layer_draft_shape(base)
    d = s.d_model
    rng = np.random.default_rng(21)
    g_attn = (0.5 + rng.random(d)).astype(np.float32)
    g_fin = (0.5 + rng.random(d)).astype(np.float32)
    wshape = (s.q_dim, d) if zero == "wq" else (s.kv_dim, d)
    over = {f"draft.layers.0.{zero}": np.zeros(wshape, np.float32),
            "draft.layers.0.w_down": np.zeros((d, s.ffn_dim), np.float32),
            "draft.layers.0.attn_norm": g_attn, "draft.final_norm": g_fin}
    w = Weights(wl.SyntheticWeights(s).with_override(over))
    P, B, anchor = 11, 6, 7
    hcat, dc = _draft_context(w, s, P, 22)
    got = draft_block_logits(w, s, nm.Precision("exact"), dc, anchor, P, B)
    x = np.stack([w["tok_emb"][anchor]] + [w["draft.mask_emb"]] * (B - 1))
    wv = w["draft.layers.0.wv"]
    vb = (nm.rmsnorm(x, g_attn, s.rms_eps) @ wv.T).reshape(B, s.n_kv_heads, s.head_dim)
    f = hcat.reshape(P, -1) @ w["draft.fuse"].T
    vc = (f @ wv.T).reshape(P, s.n_kv_heads, s.head_dim)
    mean = (vc.sum(0) + vb.sum(0)) / (P + B)
    o = np.repeat(mean, s.n_heads // s.n_kv_heads, axis=0).reshape(s.q_dim)
    x_out = x + o @ w["draft.layers.0.wo"].T
    want = nm.rmsnorm(x_out[1:], g_fin, s.rms_eps) @ w["lm_head"].T
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-11)


def test_draft_logits_depend_on_relative_positions_only(tiny_w):
    """RoPE makes every score a function of query position minus key
    position.  Moving the injected context AND the block by the same offset
    leaves the draft logits unchanged; moving the block alone changes them.
    So the block sits at positions P + j against a context roped at 0..P-1."""
    s = TINY.shape
    P, B, anchor, off = 13, 5, 9, 500
    prec = nm.Precision("exact")
    hcat, c0 = _draft_context(tiny_w, s, P, 23)
    ref = draft_block_logits(tiny_w, s, prec, c0, anchor, P, B)
    big = KVCache(s.n_draft_layers, off + P, s.n_kv_heads, s.head_dim)
    inject_kv(tiny_w, s, prec, big, hcat, off + np.arange(P))
    c1 = KVCache(s.n_draft_layers, P, s.n_kv_heads, s.head_dim)
    c1.k[:] = big.k[:, off:]
    c1.v[:] = big.v[:, off:]
    shifted = draft_block_logits(tiny_w, s, prec, c1, anchor, P, B, pos0=off + P)
    np.testing.assert_allclose(shifted, ref, rtol=1e-9, atol=1e-9)
    moved = draft_block_logits(tiny_w, s, prec, c0, anchor, P, B, pos0=P + 37)
    assert np.abs(moved - ref).max() > 1e-4


def test_draft_mask_slots_are_interchangeable():
    """With a zero mask embedding, RMSNorm of slots 1..B-1 is 0, so their
    queries, keys and values are 0; with W_q = 0 every slot averages the same
    key set.  Slots 1..B-1 then enter and leave the layer identically, so
    their logits are equal -- unless a mask (causal or otherwise) gives the
    block slots different key sets."""
    s = _one_layer_draft_shape(TINY.shape)
    over = {"draft.mask_emb": np.zeros(s.d_model, np.float32),
            "draft.layers.0.wq": np.zeros((s.q_dim, s.d_model), np.float32)}
    w = Weights(wl.SyntheticWeights(s).with_override(over))
    P, B = 9, 7
    _, dc = _draft_context(w, s, P, 24)
    got = draft_block_logits(w, s, nm.Precision("exact"), dc, 3, P, B)
    for j in range(1, B - 1):
        np.testing.assert_allclose(got[j], got[0], rtol=1e-12, atol=1e-12)
    assert np.abs(got[0]).max() > 1e-3


# --------------------------------------------------------------------------
# accept rule (T2), losslessness (T1), B = 1 (T3), forced drafts (T4)
# --------------------------------------------------------------------------

def _read_accept_cases():
    cases = []
    with open(os.path.join(GOLDEN, "accept_cases.txt")) as f:
        for line in f:
            if not line.strip() or line.lstrip().startswith("#"):
                continue
            d, y, a, e = [c.split() for c in line.split("|")]
            cases.append(([int(t) for t in d], [int(t) for t in y], int(a[0]), [int(t) for t in e]))
    return cases


def test_accept_rule_golden_cases():
    cases = _read_accept_cases()
    assert len(cases) >= 7
    for d, y, a, e in cases:
        assert accept_longest_prefix(d, y) == (a, e)


def test_dflash_is_lossless_vs_greedy_ar(tiny_w, tiny_prompt):
    ar = greedy_ar(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, 40)
    df, steps = dflash_generate(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, 40, 16)
    assert df == ar
    assert all(1 <= s.accept_len + 1 <= 16 for s in steps)


def test_block_size_one_is_ar_step_for_step(tiny_w, tiny_prompt):
    ar = greedy_ar(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, 12)
    df, steps = dflash_generate(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, 12, 1)
    assert df == ar
    assert [s.ctx_len for s in steps] == list(range(64, 64 + 11))
    assert all(s.accept_len == 0 and len(s.block) == 1 for s in steps)


def test_teacher_forced_draft_accepts_full_blocks(tiny_w, tiny_prompt):
    n = 50
    ar = greedy_ar(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, n + 16)
    p0 = len(tiny_prompt)

    def forced(step, ctx_len, drafted):
        j = ctx_len - p0  # index of the anchor in the AR stream
        return ar[j + 1: j + 16]

    df, steps = dflash_generate(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, n, 16,
                                draft_override=forced)
    assert df == ar[:n]
    assert all(s.accept_len == 15 for s in steps)
    assert len(steps) == int(np.ceil((n - 1) / 16))


def test_adversarial_draft_accepts_nothing(tiny_w, tiny_prompt):
    n = 10
    ar = greedy_ar(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, n + 16)
    p0 = len(tiny_prompt)

    def adversarial(step, ctx_len, drafted):
        j = ctx_len - p0
        return [(t + 1) % TINY.shape.vocab for t in ar[j + 1: j + 16]]

    df, steps = dflash_generate(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, n, 16,
                                draft_override=adversarial)
    assert df == ar[:n]
    assert all(s.accept_len == 0 for s in steps) and len(steps) == n - 1


def test_speedup_model():
    # S = C_AR / (C_DF / E[L]); e.g. an AR token of 2 ms, a block of 3 ms and
    # 7.5 accepted tokens per block give 5x.
    assert speedup_model(2.0, 3.0, 7.5) == pytest.approx(5.0)
    assert speedup_model(1.0, 1.0, 1.0) == 1.0


# --------------------------------------------------------------------------
# DDTree (T5)
# --------------------------------------------------------------------------

def _read_tree_cases():
    recs, cur = [], {}
    with open(os.path.join(GOLDEN, "ddtree_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("#"):
                continue
            if not line:
                if cur:
                    recs.append(cur)
                cur = {}
                continue
            key, rest = line.split(None, 1)
            cur[key] = rest
    if cur:
        recs.append(cur)
    return recs


def test_ddtree_golden_cases():
    recs = _read_tree_cases()
    assert len(recs) == 3
    for r in recs:
        ids = np.array([[int(t) for t in g.split()] for g in r["ids"].split(";")], np.int32)
        lps = np.array([[float(t) for t in g.split()] for g in r["logp"].split(";")], np.float32)
        t = build_tree(int(r["anchor"]), ids, lps, int(r["budget"]))
        nodes = [tuple(int(v) for v in n.split(":")) for n in r["nodes"].split()]
        assert list(zip(t.tok, t.parent, t.depth)) == nodes
        anc = [sorted(int(v) for v in g.split()) for g in r["anc"].split("/")]
        assert [[m for m in range(t.n_nodes) if (t.ancestors[n] >> m) & 1]
                for n in range(t.n_nodes)] == anc
        if "argmax" in r:
            y = [int(v) for v in r["argmax"].split()]
            parts = r["accept"].split()
            a = int(parts[0])
            path = [int(v) for v in parts[parts.index("path") + 1: parts.index("emitted")]]
            emitted = [int(v) for v in parts[parts.index("emitted") + 1:]]
            assert tree_accept(t, y) == (a, path, emitted)


@pytest.mark.parametrize("depth,k,budget,seed", [(3, 2, 9, 0), (4, 3, 20, 1), (4, 3, 120, 2),
                                                 (2, 3, 5, 3), (4, 2, 30, 4)])
def test_ddtree_heap_equals_brute_force_top_n(depth, k, budget, seed):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((depth, 10)) * 2
    if seed == 3:
        logits[:] = np.round(logits)  # coarse values: many score ties
    ids = np.zeros((depth, k), np.int32)
    lps = np.zeros((depth, k), np.float32)
    for j in range(depth):
        ids[j], lps[j] = topk_logprobs(logits[j], k)
    t = build_tree(7, ids, lps, budget)
    # brute force: every prefix, scored by a float32 running sum in depth order
    allp = []
    for dd in range(1, depth + 1):
        for ranks in itertools.product(range(k), repeat=dd):
            sc = np.float32(0.0)
            for j, r in enumerate(ranks):
                sc = np.float32(sc + lps[j, r])
            allp.append(((-float(sc), dd, ranks), ranks))
    allp.sort()
    want = [r for _, r in allp[:budget]]
    got = []
    for n in range(1, t.n_nodes):
        ranks, m = [], n
        while m != 0:
            ranks.append(t.rank[m])
            m = t.parent[m]
        got.append(tuple(reversed(ranks)))
    assert got == want
    # ancestor bitset = transitive closure of the parent relation
    for n in range(t.n_nodes):
        m, chain = n, {n}
        while t.parent[m] >= 0:
            m = t.parent[m]
            chain.add(m)
        assert {x for x in range(t.n_nodes) if (t.ancestors[n] >> x) & 1} == chain
        assert t.parent[n] < n


def test_path_tree_equals_linear_verify(tiny_w, tiny_prompt):
    """k = 1 with budget B-1 gives a single path; its tree verify must give
    the same argmax as the linear causal verify of the same tokens."""
    s = TINY.shape
    prec = nm.Precision("exact")
    seq_a = Sequence1(tiny_w, s, prec, 128)
    seq_a.prefill(tiny_prompt, inject=True)
    seq_b = Sequence1(tiny_w, s, prec, 128)
    seq_b.prefill(tiny_prompt, inject=True)
    toks = [int(v) for v in tiny_prompt[:8]]
    ids = np.array(toks[1:], np.int32)[:, None]
    t = build_tree(toks[0], ids, np.full((7, 1), -0.5, np.float32), 7)
    assert t.tok == toks and t.parent == list(range(-1, 7))
    lt, ct = tree_verify(seq_a, t)
    ll, cl = seq_b.verify(toks)
    np.testing.assert_array_equal(lt, ll)
    np.testing.assert_array_equal(ct, cl)


def test_ddtree_is_lossless_and_budget_zero_is_ar(tiny_w, tiny_prompt):
    ar = greedy_ar(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, 24)
    dt, steps = ddtree_generate(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, 24,
                                16, 8, 64)
    assert dt == ar
    assert all(st[0].n_nodes == 65 for st in steps)
    d0, steps0 = ddtree_generate(tiny_w, TINY.shape, nm.Precision("exact"), tiny_prompt, 8,
                                 16, 8, 0)
    assert d0 == ar[:8] and all(st[1] == 0 and st[0].n_nodes == 1 for st in steps0)


def test_tree_commit_compacts_accepted_path(tiny_w, tiny_prompt):
    """After a tree step the cache must equal that of a causal pass over the
    committed tokens (compaction moved every accepted row to its slot)."""
    s = TINY.shape
    prec = nm.Precision("exact")
    seq = Sequence1(tiny_w, s, prec, 160)
    lg, _ = seq.prefill(tiny_prompt, inject=True)
    anchor = nm.argmax_lowest(lg[-1])
    # a tree whose path [anchor, x1, x2] will be accepted: use AR tokens at depth 1, 2
    ar = greedy_ar(tiny_w, s, prec, tiny_prompt, 4)
    ids = np.array([[7, ar[1]], [ar[2], 9], [11, 12]], np.int32)
    lps = np.array([[-0.1, -0.2], [-0.1, -0.3], [-0.5, -0.6]], np.float32)
    t = build_tree(anchor, ids, lps, 6)
    vlog, cap = tree_verify(seq, t)
    y = [nm.argmax_lowest(r) for r in vlog]
    a, path, emitted = tree_accept(t, y)
    assert a >= 2 and emitted[:2] == ar[1:3]
    tree_commit(seq, cap, path)
    ref = Sequence1(tiny_w, s, prec, 160)
    ref.prefill(list(tiny_prompt) + [anchor] + emitted[:-1], inject=True)
    n = seq.length
    assert n == ref.length
    np.testing.assert_array_equal(seq.cache.k[:, :n], ref.cache.k[:, :n])
    np.testing.assert_array_equal(seq.cache.v[:, :n], ref.cache.v[:, :n])
    np.testing.assert_allclose(seq.dcache.k[:, :n], ref.dcache.k[:, :n], rtol=0, atol=0)
