"""Host logic of bench.py that needs no GPU: which roofline a kernel class is
reported against."""
import pytest

import bench


def test_weight_streaming_gemm_is_hbm_bound():
    # 16 token rows: 2 * 16 flops per 2-byte weight -> 16 flop/B
    nbytes = 111.4e6
    bound, achieved, peak, unit = bench.gemm_roofline(nbytes, 16 * nbytes, 0.0279, 6777.0, 1714.9)
    assert (bound, unit, peak) == ("hbm", "GB/s", 6777.0)
    assert achieved == pytest.approx(nbytes / 0.0279e-3 / 1e9)


def test_wide_token_tile_gemm_is_tensor_bound():
    # 512 token rows: 512 flop/B, above the machine balance of ~253 flop/B
    nbytes = 55.2e6
    flops = 2 * 512 * 6144 * 4096
    bound, achieved, peak, unit = bench.gemm_roofline(nbytes, flops, 0.0449, 6777.0, 1714.9)
    assert (bound, unit, peak) == ("tensor", "TFLOP/s", 1714.9)
    assert achieved == pytest.approx(flops / 0.0449e-3 / 1e12)


def test_balance_point_and_zero_time():
    hbm, tf = 6000.0, 1500.0
    balance = tf * 1e12 / (hbm * 1e9)  # 250 flop/B
    assert bench.gemm_roofline(1e6, (balance - 1) * 1e6, 1.0, hbm, tf)[0] == "hbm"
    assert bench.gemm_roofline(1e6, (balance + 1) * 1e6, 1.0, hbm, tf)[0] == "tensor"
    assert bench.gemm_roofline(1e6, 1e9, 0.0, hbm, tf) == ("hbm", 0.0, hbm, "GB/s")
