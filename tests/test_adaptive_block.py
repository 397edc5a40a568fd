"""Host policy that picks the block size of each DFlash step from the
recent acceptance lengths (block_diffusion_speculative_injection_gb300.adaptive).
The GPU side (tests/test_gpu_e2e.py) checks that any block schedule emits
the same tokens as greedy AR decoding."""
import math

import pytest

from block_diffusion_speculative_injection_gb300.adaptive import AdaptiveBlock


def test_starts_at_the_configured_block():
    assert AdaptiveBlock(16).next_block() == 16
    assert AdaptiveBlock(4).next_block() == 4


def test_one_update_by_hand():
    p = AdaptiveBlock(16, decay=0.5, slack=2)
    p.update([4, 4])  # ema = 0.5 * 15 + 0.5 * 4 = 9.5
    assert p.ema == pytest.approx(9.5)
    assert p.next_block() == math.ceil(9.5) + 1 + 2


def test_no_acceptance_settles_at_anchor_plus_slack():
    p = AdaptiveBlock(16, b_min=2, slack=2)
    for _ in range(60):
        p.update([0])
    assert p.next_block() == 3
    q = AdaptiveBlock(16, b_min=5, slack=2)
    for _ in range(60):
        q.update([0, 0, 0])
    assert q.next_block() == 5


def test_whole_blocks_accepted_grow_back_to_the_maximum():
    p = AdaptiveBlock(16, slack=2)
    for _ in range(60):
        p.update([0])
    sizes = []
    for _ in range(20):
        b = p.next_block()
        sizes.append(b)
        p.update([b - 1])  # every draft token accepted
    assert sizes[-1] == 16
    assert all(x <= y for x, y in zip(sizes, sizes[1:]))


def test_always_within_bounds_and_mean_over_the_batch():
    p = AdaptiveBlock(8, b_min=2, decay=0.25, slack=1)
    for step in range(50):
        b = p.next_block()
        assert 2 <= b <= 8
        p.update([(step * 7) % b, (step * 3) % b, 0])
    r = AdaptiveBlock(16, decay=0.0, slack=0)
    r.update([1, 2, 3, 6])  # mean 3
    assert r.next_block() == 4


def test_rejects_bad_parameters():
    with pytest.raises(ValueError):
        AdaptiveBlock(4, b_min=5)
    with pytest.raises(ValueError):
        AdaptiveBlock(4, decay=1.0)
    with pytest.raises(ValueError):
        AdaptiveBlock(4, slack=-1)
    p = AdaptiveBlock(4)
    p.update([])
    assert p.next_block() == 4
