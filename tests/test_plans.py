"""Launch plans of the tensor-core GEMM and the split-KV attention
(dflash_plan_gemm / dflash_plan_attention: host arithmetic, no GPU).

The Qwen3-8B cases pin the grids the ncu launch lists show for one step
(profiles/); the sweeps check the rules every plan must keep, among them
that a direct epilogue's exchange buffers and row metadata fit in the stage
memory it reuses."""
import itertools

import pytest

from block_diffusion_speculative_injection_gb300 import capi

QKV, SWIGLU, RESID, SLAB, VOCAB, VOCAB_TOP2 = 1, 2, 3, 0, 6, 7
GB300_SMS = 152


@pytest.fixture(scope="module")
def lib():
    try:
        return capi.load()
    except FileNotFoundError:
        pytest.skip("libdflash.so not built (run __graft_entry__.build())")


def grid(p):
    return (p["n_tiles"], p["m_tiles"], p["splits"])


def test_qwen3_8b_one_sequence_grids(lib):
    # 16 token rows (one block): the grids of the b = 1 launch list
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 16, 6144, 4096, QKV)) == (48, 1, 5)
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 16, 4096, 4096, RESID)) == (32, 1, 8)
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 16, 4096, 12288, RESID)) == (32, 1, 8)
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 16, 2 * 12288, 4096, SWIGLU)) == (192, 1, 1)
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 16, 151936, 4096, SLAB)) == (1187, 1, 1)
    # the lm_head with its top-2 reduction in registers: persistent at 512 rows
    p = capi.dflash_plan_gemm(GB300_SMS, 512, 151936, 4096, VOCAB_TOP2)
    assert (grid(p), p["persistent"]) == ((1187, 2, 1), GB300_SMS)
    # the lm_head with its vocabulary reduction: one CTA per 128 ids, no K split
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 16, 151936, 4096, VOCAB)) == (1187, 1, 1)
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 512, 151936, 4096, VOCAB)) == (1187, 2, 1)
    p = capi.dflash_plan_gemm(GB300_SMS, 16, 6144, 4096, QKV)
    assert (p["BN"], p["threads"]) == (16, 128)


def test_qwen3_8b_32_sequences_qkv(lib):
    # 512 token rows: QKV (48 feature tiles, unsplit) takes three 176-row
    # token tiles on 144 SMs
    p = capi.dflash_plan_gemm(GB300_SMS, 512, 6144, 4096, QKV)
    assert grid(p) == (48, 3, 1)
    assert (p["BN"], p["threads"]) == (176, 384)
    # O and down (32 feature tiles) would fill 64 SMs: two K splits per tile
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 512, 4096, 4096, RESID)) == (32, 2, 2)
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 512, 4096, 12288, RESID)) == (32, 2, 2)
    # a DDTree pass of 4 x 65 rows: two 144-row token tiles, O and down split
    assert grid(capi.dflash_plan_gemm(GB300_SMS, 260, 4096, 14336, RESID)) == (32, 2, 2)
    assert capi.dflash_plan_gemm(GB300_SMS, 260, 4096, 14336, RESID)["BN"] == 144


@pytest.mark.parametrize("sms", [GB300_SMS, 132, 20])
def test_gemm_plan_rules(lib, sms):
    shapes = [(6144, 4096, QKV), (4096, 4096, RESID), (4096, 12288, RESID),
              (24576, 4096, SWIGLU), (151936, 4096, SLAB), (2048, 8192, 4), (10240, 4096, 5),
              (151936, 4096, VOCAB), (151936, 4096, VOCAB_TOP2)]
    for M, (N, K, kind) in itertools.product(list(range(1, 80)) + [96, 128, 129, 200, 256, 257,
                                                                  300, 512, 777, 1024, 2048],
                                             shapes):
        p = capi.dflash_plan_gemm(sms, M, N, K, kind)
        BN, mt, nt, st, sp, th, smem = (p[k] for k in ("BN", "m_tiles", "n_tiles", "stages",
                                                       "splits", "threads", "smem_bytes"))
        # token tiles as wide as the MMA allows; an unsplit pass that leaves
        # SMs idle takes more (of at least 64 rows) while they fit one wave
        mt0 = (M + 255) // 256
        assert BN % 16 == 0 and 16 <= BN <= 256 and BN * mt >= M and mt >= mt0
        if mt > mt0:
            assert sp == 1 and not p["persistent"] and kind not in (SLAB, VOCAB, VOCAB_TOP2) and mt0 > 1
            assert nt * mt <= sms and BN >= 64
            assert nt * (mt + 1) > sms or -(-M // (mt + 1)) <= 48
        assert nt == (N + 127) // 128
        assert 2 <= st <= 8
        pers = p["persistent"]
        # persistent form: more tiles than SMs, wide tiles, no K split, not the lm_head
        want_pers = sp == 1 and BN > 64 and kind not in (SLAB, VOCAB) and nt * mt > sms
        assert pers == (sms if want_pers else 0)
        if pers:
            assert th == 448 and smem <= 227 * 1024
            # ring + the epilogue's own scratch (three 16 x 128 fp32 buffers, 256 x 12 B)
            assert smem >= st * (128 * 64 * 2 + BN * 64 * 2) + 3 * 16 * 128 * 4 + 256 * 12
        else:
            assert th == (384 if BN > 128 else 128)
            if BN <= 128:  # two CTAs per SM: dynamic + 3 KB static + 1 KB reserve each
                assert 2 * (smem + 3072 + 1024) <= 228 * 1024
            assert smem <= 210 * 1024  # the kernel's shared-memory attribute
        stage_mem = st * (128 * 64 * 2 + BN * 64 * 2)
        # direct epilogue: one 16 x 128 fp32 exchange buffer per group of 128
        # threads, then 256 x 8 B destination offsets and 256 x 4 B RoPE
        # offsets, in stage memory (or, persistent, in memory of their own)
        assert (th // 128) * 16 * 128 * 4 + 256 * 8 + 256 * 4 <= stage_mem or pers
        # a split tile's fp32 partial [BN][128] sits in its own stage memory
        if sp > 1:
            assert BN * 128 * 4 <= stage_mem
        assert 1 <= sp <= 8 and sp <= K // 64 // 4 or sp == 1
        if kind in (SWIGLU, SLAB, VOCAB, VOCAB_TOP2):
            assert sp == 1
        slots = (2 if BN <= 128 else 1) * sms
        if sp > 1:
            assert nt * mt * sp * 8 <= 7 * slots  # every cluster resident at once
        # a grid that fills under half of the CTA slots is split along K when
        # two splits are allowed (kind, K, partial tile, cluster residency)
        if (kind not in (SWIGLU, SLAB, VOCAB, VOCAB_TOP2) and nt * mt * 2 <= slots and K // 64 // 4 >= 2
                and BN * 128 * 4 <= stage_mem and nt * mt * 16 <= 7 * slots):
            assert sp >= 2


def test_gemm_plan_refuses_bad_sizes(lib):
    for args in [(152, 0, 4096, 4096, 1), (152, 16, 4096, 100, 1), (152, 16, 4096, 0, 1),
                 (0, 16, 4096, 4096, 1), (152, 16, 4096, 4096, 8), (152, 16, 4160, 4096, SWIGLU)]:
        with pytest.raises(capi.DFlashError):
            capi.dflash_plan_gemm(*args)


def test_attention_plan_one_sequence(lib):
    # 16 rows x 32 heads over 2048 + 16 keys: 8 KV heads, 17 key tiles of 128,
    # one tile per split, all CTAs (one per SM) in a single wave
    p = capi.dflash_plan_attention(GB300_SMS, 1, 32, 8, 16, 2048 + 16)
    assert p == {"splits": 17, "keys_per_split": 128, "ctas": 8 * 17}
    # short context: no split
    assert capi.dflash_plan_attention(GB300_SMS, 1, 32, 8, 16, 128)["splits"] == 1


@pytest.mark.parametrize("sms", [GB300_SMS, 40])
def test_attention_plan_rules(lib, sms):
    for batch, keys, min_s, (H, Hkv) in itertools.product(
            [1, 2, 4, 8, 32], [16, 64, 65, 500, 2064, 8208, 16400], [1, 2], [(32, 8), (16, 16), (64, 4)]):
        q = 16
        p = capi.dflash_plan_attention(sms, batch, H, Hkv, q, keys, min_s)
        s, kps, ctas = p["splits"], p["keys_per_split"], p["ctas"]
        tiles = (keys + 127) // 128
        assert 1 <= s <= min(256, tiles)
        base = ((q + 64 // (H // Hkv) - 1) // (64 // (H // Hkv))) * Hkv * batch
        assert ctas == base * s
        if s > 1:
            assert kps % 128 == 0
            assert s * kps >= keys and (s - 1) * kps < keys  # no split is empty
        else:
            assert kps == keys
        if min_s == 2 and tiles >= 2:
            assert s >= 2


def test_attention_plan_refuses_bad_shapes(lib):
    for args in [(152, 0, 32, 8, 16, 100), (152, 1, 32, 6, 16, 100), (152, 1, 32, 8, 0, 100),
                 (152, 1, 32, 8, 16, 0), (152, 1, 256, 2, 16, 100)]:
        with pytest.raises(capi.DFlashError):
            capi.dflash_plan_attention(*args)
