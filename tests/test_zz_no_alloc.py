"""The allocation-free block attention entry point.

dflash_block_attention_noalloc exists for callers that cannot allocate
device memory where they run attention (an engine's per-request path that
must use its own pool, a serving loop that bans cudaMalloc after start-up,
a plugin execute call with no allocator).  It keeps the split-KV partials in
a fixed 16 MiB array inside the library instead of a caller workspace.

These tests call it through the C ABI twice in a row on the same sizes (the
second call finds the first call's leftovers in the shared array) and
compare each result with the workspace-taking entry point, within the
tolerance the other attention tests use; and they check that sizes needing
more than the fixed array are refused.  This file is collected last.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

H, HKV, HD, BLK = 32, 8, 128, 16
LIMIT = 16 << 20


def _inputs(b, ctx, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(b, BLK, H, HD, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(b, HKV, ctx + BLK, HD, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(b, HKV, ctx + BLK, HD, device="cuda", generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("b,ctx,causal", [(1, 2048, 0), (2, 1000, 1), (8, 4096, 0)])
def test_noalloc_matches_workspace_entry_twice(b, ctx, causal):
    from block_diffusion_speculative_injection_gb300 import capi
    need = capi.dflash_block_attention_workspace(b, H, HKV, ctx, BLK)
    assert 0 < need <= LIMIT  # these sizes do use the scratch array
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for call in range(2):
        q, k, v = _inputs(b, ctx, 100 * call + b)
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        capi.dflash_block_attention(b, H, HKV, ctx, BLK, causal, q, k, v, ref, ws)
        capi.dflash_block_attention_noalloc(b, H, HKV, ctx, BLK, causal, q, k, v, got)
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        torch.testing.assert_close(got.float(), ref.float(), atol=2e-2, rtol=1e-2)


def test_noalloc_refuses_sizes_beyond_its_array():
    """A shape whose split-KV partials exceed the fixed array is refused with
    DFLASH_E_CAPACITY (the first candidate that needs more than 16 MiB on this
    GPU; many heads of 64 query rows each give many CTAs, hence many
    partial rows)."""
    from block_diffusion_speculative_injection_gb300 import capi
    cands = [(32, 32, 8, 16384, 16), (1, 512, 512, 4096, 64), (2, 512, 512, 4096, 64),
             (1, 1024, 1024, 2048, 64)]
    pick = None
    for b, h, hkv, ctx, blk in cands:
        if capi.dflash_block_attention_workspace(b, h, hkv, ctx, blk) > LIMIT:
            pick = (b, h, hkv, ctx, blk)
            break
    assert pick is not None, "no candidate shape exceeds the fixed array"
    b, h, hkv, ctx, blk = pick
    q = torch.zeros(b, blk, h, HD, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(b, hkv, ctx + blk, HD, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    out = torch.empty_like(q)
    with pytest.raises(capi.DFlashError) as e:
        capi.dflash_block_attention_noalloc(b, h, hkv, ctx, blk, 0, q, k, v, out)
    assert e.value.status == 2  # DFLASH_E_CAPACITY
