"""Block attention through dflash_block_attention against the oracle's
softmax attention, on bf16 inputs drawn N(0,1) (query length 16, 32 query
heads over 8 KV heads, head_dim 128).

Small cases run every output row (context lengths with ragged 64-key tails,
causal and bidirectional, with and without the split-KV workspace); the
full op grid (context 512..16384 x batch 1, 8, 32) checks sampled rows that
the oracle computes one by one.  Tolerance: max-abs 2e-2, relative 1e-2.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle.numerics import attend

pytestmark = pytest.mark.gpu
H, HKV, HD, BLK = 32, 8, 128, 16


def run_op(b, ctx, causal, use_ws=True, block=BLK):
    from block_diffusion_speculative_injection_gb300 import capi
    from block_diffusion_speculative_injection_gb300.engine import device_operand
    q = device_operand("q", b * block * H).view(b, block, H, HD)
    k = device_operand("k", b * HKV * (ctx + block)).view(b, HKV, ctx + block, HD)
    v = device_operand("v", b * HKV * (ctx + block)).view(b, HKV, ctx + block, HD)
    out = torch.empty_like(q)
    ws = None
    need = capi.dflash_block_attention_workspace(b, H, HKV, ctx, block)
    assert need >= 0
    if use_ws and need > 0:
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    capi.dflash_block_attention(b, H, HKV, ctx, block, causal, q, k, v, out, ws)
    torch.cuda.synchronize()
    return out


def oracle_rows(b_total, ctx, causal, picks, block=BLK):
    """picks: list of (b, j, h) -> oracle output row (fp64)."""
    n_k = ctx + block
    outs = []
    for (b, j, h) in picks:
        kvh = h // (H // HKV)
        rows = (b * HKV + kvh) * n_k + np.arange(n_k)
        kk = wl.attn_operand_rows("k", b_total * HKV * n_k, rows=rows).astype(np.float64)
        vv = wl.attn_operand_rows("v", b_total * HKV * n_k, rows=rows).astype(np.float64)
        qrow = wl.attn_operand_rows("q", b_total * block * H, rows=[(b * block + j) * H + h])
        n_vis = ctx + j + 1 if causal else n_k
        o = attend(qrow.astype(np.float64), kk[:n_vis, None, :], vv[:n_vis, None, :])
        outs.append(o[0])
    return np.stack(outs)


@pytest.mark.parametrize("b,ctx,causal,use_ws", [
    (1, 0, 0, True), (1, 37, 0, True), (2, 300, 1, True), (3, 129, 0, False),
    (1, 1000, 0, True), (2, 64, 1, False),
])
def test_block_attention_all_rows(b, ctx, causal, use_ws):
    out = run_op(b, ctx, causal, use_ws).float().cpu().numpy()
    picks = [(bb, j, h) for bb in range(b) for j in range(BLK) for h in range(0, H, 3)]
    ref = oracle_rows(b, ctx, causal, picks)
    got = np.stack([out[bb, j, h] for (bb, j, h) in picks])
    np.testing.assert_allclose(got, ref, atol=2e-2, rtol=1e-2)


def test_split_and_unsplit_agree():
    a = run_op(2, 2000, 0, True).float()
    c = run_op(2, 2000, 0, False).float()
    assert torch.allclose(a, c, atol=1e-2, rtol=1e-2)


@pytest.mark.parametrize("ctx", wl.ATTN_OP_CTX)
@pytest.mark.parametrize("b", wl.ATTN_OP_BATCH)
def test_block_attention_full_grid_sampled(b, ctx):
    out = run_op(b, ctx, 0, True).float().cpu().numpy()
    rng = np.random.default_rng(ctx + b)
    picks = [(int(rng.integers(b)), int(rng.integers(BLK)), int(rng.integers(H))) for _ in range(4)]
    picks.append((b - 1, BLK - 1, H - 1))
    ref = oracle_rows(b, ctx, 0, picks)
    got = np.stack([out[bb, j, h] for (bb, j, h) in picks])
    np.testing.assert_allclose(got, ref, atol=2e-2, rtol=1e-2)
    assert np.isfinite(out).all()


# one KV head of 4 query heads over a long context: a single CTA per split,
# so the planner spreads the keys over more than 32 splits (the merge's
# batched path)
MANY_SPLITS = (1, 4, 1, 6000)  # batch, q heads, kv heads, context


def test_many_splits_merge_path():
    from block_diffusion_speculative_injection_gb300 import capi
    b, h, hkv, ctx = MANY_SPLITS
    g = torch.Generator(device="cuda").manual_seed(11)
    q = torch.randn(b, BLK, h, HD, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(b, hkv, ctx + BLK, HD, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(b, hkv, ctx + BLK, HD, device="cuda", generator=g).to(torch.bfloat16)
    out = torch.empty_like(q)
    need = capi.dflash_block_attention_workspace(b, h, hkv, ctx, BLK)
    assert need // (b * BLK * h * (HD + 2) * 4) > 32
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for causal in (0, 1):
        capi.dflash_block_attention(b, h, hkv, ctx, BLK, causal, q, k, v, out, ws)
        torch.cuda.synchronize()
        kk = k[0, 0].float().cpu().numpy().astype(np.float64)
        vv = v[0, 0].float().cpu().numpy().astype(np.float64)
        qq = q[0].float().cpu().numpy().astype(np.float64)
        got = out[0].float().cpu().numpy()
        for j in range(BLK):
            n = ctx + j + 1 if causal else ctx + BLK
            ref = attend(qq[j], kk[:n, None, :], vv[:n, None, :])
            np.testing.assert_allclose(got[j], ref, atol=2e-2, rtol=1e-2)


def test_full_grid_covers_every_combine_regime():
    """The split merge has three code paths: up to 8 splits, up to 32 (all
    loads in flight at once) and more (batches of 32).  The sampled grid
    above and the many-splits case must reach each of them."""
    from block_diffusion_speculative_injection_gb300 import capi
    seen = set()
    shapes = [(b, H, HKV, ctx) for b in wl.ATTN_OP_BATCH for ctx in wl.ATTN_OP_CTX]
    for b, h, hkv, ctx in shapes + [MANY_SPLITS]:
        need = capi.dflash_block_attention_workspace(b, h, hkv, ctx, BLK)
        splits = need // (b * BLK * h * (HD + 2) * 4) if need > 0 else 1
        if splits > 1:
            seen.add(0 if splits <= 8 else (1 if splits <= 32 else 2))
    assert seen == {0, 1, 2}, seen


def test_misaligned_pointers_are_refused():
    from block_diffusion_speculative_injection_gb300 import capi
    b, ctx = 1, 100
    q = torch.zeros(b * BLK * H * HD + 8, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(b * HKV * (ctx + BLK) * HD, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    out = torch.zeros(b * BLK * H * HD + 8, dtype=torch.bfloat16, device="cuda")
    for qq, oo in ((q[1:], out[:-8]), (q[:-8], out[1:]), (q[4:], out[:-8])):
        with pytest.raises(capi.DFlashError) as e:
            capi.dflash_block_attention(b, H, HKV, ctx, BLK, 0, qq, k, v, oo)
        assert e.value.status == 1
    capi.dflash_block_attention(b, H, HKV, ctx, BLK, 0, q[8:], k, v, out[8:])  # 16-byte offsets pass
    torch.cuda.synchronize()
