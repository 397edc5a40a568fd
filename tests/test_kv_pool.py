"""The paged KV cache's host allocator (dflash_kv_pool_*): no GPU.

Rules pinned here: a sequence holds ceil(slots / 128) pages, new pages are
the lowest free ids, a refused request changes nothing, release returns
every page, and no page is ever held twice.
"""
import random

import pytest

from block_diffusion_speculative_injection_gb300 import capi

S = capi.PAGE_SLOTS


@pytest.fixture(scope="module")
def lib():
    try:
        return capi.load()
    except FileNotFoundError:
        pytest.skip("libdflash.so not built (run __graft_entry__.build())")


def test_lowest_free_pages_first_and_reuse(lib):
    p = capi.KvPool(10, 3, 4)
    assert p.reserve(0, 200) == (0, 2) and p.pages(0) == [0, 1]
    assert p.reserve(1, 1) == (0, 1) and p.pages(1) == [2]
    assert p.reserve(0, 2 * S + 1) == (2, 1) and p.pages(0) == [0, 1, 3]
    assert p.reserve(0, 3 * S) == (3, 0)  # already covered
    assert p.release(1) == 1 and p.pages(1) == []
    # the freed page 2 goes out before 4
    assert p.reserve(2, S + 1) == (0, 2) and p.pages(2) == [2, 4]
    assert p.free() == 10 - 5
    assert p.reserve(1, 0) == (0, 0) and p.pages(1) == []


def test_refusals_change_nothing(lib):
    p = capi.KvPool(3, 2, 4)
    p.reserve(0, 2 * S)
    with pytest.raises(capi.DFlashError) as e:
        p.reserve(1, 2 * S)  # one free page, two needed
    assert e.value.status == 2
    assert p.free() == 1 and p.pages(1) == []
    with pytest.raises(capi.DFlashError) as e:
        capi.KvPool(100, 1, 4).reserve(0, 4 * S + 1)  # more than max_pages
    assert e.value.status == 2
    for seq, n in [(-1, 1), (2, 1), (0, -5)]:
        with pytest.raises(capi.DFlashError) as e:
            p.reserve(seq, n)
        assert e.value.status == 1
    assert p.release(7) == -1


def test_random_sequences_of_calls_keep_the_invariants(lib):
    rng = random.Random(11)
    n_pages, n_seq, max_pages = 40, 6, 9
    p = capi.KvPool(n_pages, n_seq, max_pages)
    free = set(range(n_pages))
    held = {s: [] for s in range(n_seq)}
    for _ in range(2000):
        s = rng.randrange(n_seq)
        if rng.random() < 0.2:
            assert p.release(s) == len(held[s])
            free |= set(held[s])
            held[s] = []
        else:
            slots = rng.randrange(0, (max_pages + 2) * S)
            need = -(-slots // S)
            add = max(0, need - len(held[s]))
            if need > max_pages or add > len(free):
                with pytest.raises(capi.DFlashError):
                    p.reserve(s, slots)
            else:
                got = sorted(free)[:add]
                assert p.reserve(s, slots) == (len(held[s]), add)
                held[s] += got
                free -= set(got)
        assert p.pages(s) == held[s]
        assert p.free() == len(free)
    owned = [x for s in held for x in held[s]]
    assert len(owned) == len(set(owned)) and not (set(owned) & free)
    assert set(owned) | free == set(range(n_pages))
