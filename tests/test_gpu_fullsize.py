"""Full-size parity in the benchmark's launch configuration: Qwen3-8B-shaped
bf16 target (36 layers, d 4096, 32/8 heads, FFN 12288, vocab 151936) with a
5-layer drafter, batch 1, B = 16, a 2048-token prompt.

The oracle cannot run the whole model at this size, so it checks sampled
outputs one by one, teacher-forced on the GPU's own caches (each check gives
the oracle exactly the inputs the GPU consumed at that point):
  * layer-0 K cache rows (embedding -> RMSNorm -> Wk -> RoPE), sampled slots;
  * the residual after layer 0 (the first captured layer) of block rows,
    attending over the GPU's layer-0 K/V cache;
  * sampled layers 1..35 one at a time for two block rows: input = the GPU's
    fp32 residual after the previous layer (dflash_debug_trace), context =
    the GPU's caches, output against the GPU's residual after the layer;
  * the lm_head logits and argmax of block rows from the GPU's final
    residual;
  * the drafter's layer-0 cache rows written by KV injection from the GPU's
    capture rows (W_fuse, then Wk / Wv of draft layer 0, RoPE);
  * every draft layer of the block draft pass over all 16 block rows,
    teacher-forced on the GPU's draft residual trace (dflash_debug_trace_draft)
    and the GPU's draft cache (no mask), and the draft logits / drafted tokens
    from the GPU's final draft residual;
  * the accept decision against the stated rule.
Tolerance: max-abs 2e-2, relative 1e-2 (bf16 path); argmax exact where the
oracle's top-1/top-2 margin exceeds 1e-2.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import numerics as nm
from oracle.decode import accept_longest_prefix
from oracle.models import Weights, _layer

from gpu_replay import check_argmax, check_close, check_draft_layer, draft_inputs, lm_logits

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-2, 1e-2
# target layers checked one by one (first, around each injected layer, last)
LAYERS = (0, 1, 2, 9, 10, 17, 18, 26, 27, 34, 35)


@pytest.fixture(scope="module")
def run():
    from block_diffusion_speculative_injection_gb300.engine import DFlashEngine
    w = wl.WORKLOADS["qwen3_8b_b1"]
    prompt = wl.prompts(w)[0]
    P = len(prompt)
    eng = DFlashEngine(w.shape, 16, 1, P + 64, max_rows=P)
    sid = eng.seq_ids(1)
    anchors = eng.prefill([prompt])
    torch.cuda.synchronize()
    # draft cache after prefill injection (layer 0), before the step adds rows
    dk0 = eng.debug_view("dk_cache", 0)[0].float().cpu().numpy()
    dv0 = eng.debug_view("dv_cache", 0)[0].float().cpu().numpy()
    from block_diffusion_speculative_injection_gb300 import capi
    trace = torch.zeros(w.shape.n_layers, P, w.shape.d_model, dtype=torch.float32, device="cuda")
    dtrace = torch.zeros(w.shape.n_draft_layers, P, w.shape.d_model, dtype=torch.float32,
                         device="cuda")
    qa = [torch.zeros(w.shape.n_draft_layers, P, w.shape.q_dim, dtype=torch.bfloat16,
                      device="cuda") for _ in range(2)]
    capi.dflash_debug_trace(eng.ctx, trace)
    capi.dflash_debug_trace_draft(eng.ctx, dtrace)
    capi.dflash_debug_trace_draft_attn(eng.ctx, *qa)
    anchor = int(anchors[0].item())
    out, dlog, vlog, margin = eng.step(sid, anchors, want_logits=True)
    torch.cuda.synchronize()
    capi.dflash_debug_trace(eng.ctx, None)
    capi.dflash_debug_trace_draft(eng.ctx, None)
    capi.dflash_debug_trace_draft_attn(eng.ctx, None, None)
    r = dict(
        w=w, prompt=prompt, P=P,
        block=out.block[0].cpu().numpy(), argmax=out.argmax[0].cpu().numpy(),
        accept=int(out.accept_len[0]), emitted=out.emitted[0].cpu().numpy(),
        vlog=vlog[0].cpu().numpy(), dlog=dlog[0].cpu().numpy(),
        capture=eng.debug_view("capture")[:16].float().cpu().numpy(),
        dk0=dk0, dv0=dv0,
        k_cache={l: eng.debug_view("k_cache", l)[0, :, : P + 16].float().cpu().numpy()
                 for l in LAYERS},
        v_cache={l: eng.debug_view("v_cache", l)[0, :, : P + 16].float().cpu().numpy()
                 for l in LAYERS},
        trace=trace[:, :16].cpu().numpy(),
        anchor=anchor, dtrace=dtrace[:, :16].cpu().numpy(),
        dq=qa[0][:, :16].float().cpu().numpy(), dao=qa[1][:, :16].float().cpu().numpy(),
        dctx={l: (eng.debug_view("dk_cache", l)[0, :, :P].float().cpu().numpy().transpose(1, 0, 2),
                  eng.debug_view("dv_cache", l)[0, :, :P].float().cpu().numpy().transpose(1, 0, 2))
              for l in range(w.shape.n_draft_layers)},
        length=eng.lengths(1)[0],
        dk_after=eng.debug_view("dk_cache", 0)[0, :, : P + 16].float().cpu().numpy(),
        dv_after=eng.debug_view("dv_cache", 0)[0, :, : P + 16].float().cpu().numpy(),
    )
    eng.close()
    r["W"] = Weights(wl.SyntheticWeights(w.shape, w.seed))
    return r


def tokens_of(r):
    return np.concatenate([r["prompt"], r["block"]]).astype(np.int64)


def test_accept_rule_and_length(run):
    a, em = accept_longest_prefix([int(t) for t in run["block"][1:]], [int(y) for y in run["argmax"]])
    assert a == run["accept"]
    assert em == [int(t) for t in run["emitted"] if t >= 0]
    assert run["length"] == run["P"] + a + 1


def test_layer0_k_cache_rows(run):
    s = run["w"].shape
    W, toks = run["W"], tokens_of(run)
    prec = nm.Precision("bf16emu")
    slots = [0, 1, 777, run["P"] - 1, run["P"], run["P"] + 15]
    h = prec.store(nm.rmsnorm(W["tok_emb"][toks[slots]], W["layers.0.attn_norm"], s.rms_eps))
    k = nm.linear(h, W["layers.0.wk"]).reshape(len(slots), s.n_kv_heads, s.head_dim)
    k = prec.store(nm.apply_rope(k, np.array(slots), s.rope_theta))
    v = prec.store(nm.linear(h, W["layers.0.wv"]).reshape(len(slots), s.n_kv_heads, s.head_dim))
    gk = run["k_cache"][0][:, slots].transpose(1, 0, 2)
    gv = run["v_cache"][0][:, slots].transpose(1, 0, 2)
    check_close(gk, k, ATOL, RTOL, "layer-0 K cache")
    check_close(gv, v, ATOL, RTOL, "layer-0 V cache")


def _row_layer(r, l, x, row):
    """Oracle layer l for block row `row` with the GPU's cache as context."""
    s = r["w"].shape
    P = r["P"]
    pos = np.array([P + row])
    kc = r["k_cache"][l].transpose(1, 0, 2)  # [slots, H_kv, hd]
    vc = r["v_cache"][l].transpose(1, 0, 2)

    def attend_rows(q, k, v):
        kk = np.concatenate([kc[: P + row], k])
        vv = np.concatenate([vc[: P + row], v])
        return np.stack([nm.attend(q[0], kk, vv)])

    return _layer(r["W"], s, nm.Precision("bf16emu"), f"layers.{l}", x, pos, attend_rows)


def test_layer0_output_of_block_rows(run):
    W, toks = run["W"], tokens_of(run)
    for row in (0, 7, 15):
        x = W["tok_emb"][toks[run["P"] + row]][None, :]
        y = _row_layer(run, 0, x, row)
        check_close(run["capture"][row, 0], y[0], ATOL, RTOL, f"layer-0 output row {row}")


@pytest.mark.parametrize("row", [3, 12])
def test_every_sampled_layer_teacher_forced(run, row):
    """Layer l of block row `row`, fed the GPU's own fp32 residual after
    layer l-1 and the GPU's caches, against the GPU's residual after layer l.
    (Layers are checked one at a time: chaining several from a rounded start
    would measure the model's sensitivity, not the kernels.)"""
    for l in LAYERS:
        if l == 0:
            continue
        x = run["trace"][l - 1, row][None, :].astype(np.float64)
        y = _row_layer(run, l, x, row)
        run["W"]._cache.clear()  # keep host memory bounded
        check_close(run["trace"][l, row], y[0], ATOL, RTOL, f"layer {l} output row {row}")


def _lm_logits(r, h_final):
    s = r["w"].shape
    sw = wl.SyntheticWeights(s, r["w"].seed)
    hn = nm.round_bf16(nm.rmsnorm(h_final[None, :], np.ones(s.d_model), s.rms_eps))[0]
    offs = sw.offsets("lm_head")
    out = np.empty(s.vocab)
    for c0 in range(0, s.vocab, 16384):
        rows = wl.pool_rows(sw.pool(), offs[c0: c0 + 16384], s.d_model).astype(np.float64)
        out[c0: c0 + len(rows)] = rows @ hn
    return out


def test_final_logits_and_argmax(run):
    for row in (0, 9):
        lg = _lm_logits(run, run["trace"][-1, row].astype(np.float64))
        check_close(run["vlog"][row], lg, ATOL, RTOL, f"verify logits row {row}")
        check_argmax([run["argmax"][row]], lg[None, :], f"verify argmax row {row}")


def test_draft_injection_cache_rows(run):
    """Rows P..P+a of draft layer 0's cache were written by KV injection from
    the step's capture rows 0..a: F = W_fuse h_cat, K = RoPE(Wk F), V = Wv F."""
    s = run["w"].shape
    W = run["W"]
    a = run["accept"]
    prec = nm.Precision("bf16emu")
    hcat = run["capture"][: a + 1].reshape(a + 1, s.n_inject * s.d_model).astype(np.float64)
    f = prec.store(nm.linear(hcat, W["draft.fuse"]))
    pos = run["P"] + np.arange(a + 1)
    k = nm.linear(f, W["draft.layers.0.wk"]).reshape(a + 1, s.n_kv_heads, s.head_dim)
    k = prec.store(nm.apply_rope(k, pos, s.rope_theta))
    v = prec.store(nm.linear(f, W["draft.layers.0.wv"]).reshape(a + 1, s.n_kv_heads, s.head_dim))
    check_close(run["dk_after"][:, pos].transpose(1, 0, 2), k, ATOL, RTOL, "injected draft K")
    check_close(run["dv_after"][:, pos].transpose(1, 0, 2), v, ATOL, RTOL, "injected draft V")
    # prompt rows injected at prefill are untouched by the step
    np.testing.assert_array_equal(run["dk_after"][:, : run["P"]], run["dk0"][:, : run["P"]])


@pytest.mark.parametrize("l", [0, 1, 2, 3, 4])
def test_draft_layer_teacher_forced(run, l):
    """Draft layer l over the 16 block rows [anchor, mask x 15] at positions
    P..P+15, input = the GPU's fp32 residual after draft layer l-1 (the
    embeddings for layer 0), context = the GPU's draft cache rows 0..P-1 (the
    injected context), no mask; checked in three stages (queries, attention
    on the GPU's queries, the rest of the layer on the GPU's attention
    output) against the GPU's traces."""
    s = run["w"].shape
    P = run["P"]
    x = (draft_inputs(s, run["w"].seed, run["anchor"], 16) if l == 0
         else run["dtrace"][l - 1].astype(np.float64))
    kc, vc = run["dctx"][l]
    check_draft_layer(run["W"], s, l, x, P, kc, vc, run["dq"][l], run["dao"][l], run["dtrace"][l],
                      f"draft layer {l}")
    run["W"]._cache.clear()


def test_draft_logits_and_argmax(run):
    """The drafter's final norm and the shared lm_head over the GPU's final
    draft residual of slots 1..15, against the GPU's draft logits; the
    drafted tokens are their argmax."""
    s = run["w"].shape
    lg = lm_logits(s, run["w"].seed, run["dtrace"][-1][1:], "draft.final_norm")
    check_close(run["dlog"], lg, ATOL, RTOL, "draft logits")
    check_argmax(run["block"][1:], lg, "drafted tokens")
