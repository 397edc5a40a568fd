"""Host-side checks of the C ABI that need no GPU: the library loads, every
function include/dflash.h declares is exported, and configuration / argument
validation rejects bad input before touching the device."""
import ctypes

import pytest

import workloads as wl
from block_diffusion_speculative_injection_gb300 import capi
from block_diffusion_speculative_injection_gb300.engine import config_for


@pytest.fixture(scope="module")
def lib():
    try:
        return capi.load()
    except FileNotFoundError:
        pytest.skip("libdflash.so not built (run __graft_entry__.build())")


def test_every_declared_function_is_exported(lib):
    names = capi.header_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(capi._SIGS)


def _create_status(cfg):
    h = ctypes.c_void_p()
    return capi.load().dflash_create(ctypes.byref(cfg), ctypes.byref(h))


@pytest.mark.parametrize("field,value", [
    ("block_size", 0), ("block_size", 17), ("n_heads", 6), ("max_batch", 0),
    ("n_inject", 0), ("max_tree_nodes", 1), ("max_tree_nodes", 200), ("max_rows", 1),
    ("dtype", 7), ("head_dim", 96), ("vocab", 1),
])
def test_create_rejects_bad_config(lib, field, value):
    cfg = config_for(wl.MINI_BF16, 16, 2, 512, 64, 0)
    setattr(cfg, field, value)
    assert _create_status(cfg) == 1  # DFLASH_E_INVALID_ARG, before any device call


def test_create_rejects_unordered_inject_layers(lib):
    cfg = config_for(wl.MINI_BF16, 16, 2, 512, 64, 0)
    cfg.inject_layers[0], cfg.inject_layers[1] = 2, 0
    assert _create_status(cfg) == 1


def test_null_context_calls_fail_cleanly(lib):
    assert lib.dflash_verify(None, 1, None, None, 1, None, 0, None, None, None, None) == 1
    assert lib.dflash_check(None) == 1
    assert lib.dflash_launch_count(None) == -1
    assert lib.dflash_seq_lengths(None) is None
    assert lib.dflash_set_block_size(None, 4) == 1
    assert lib.dflash_draft_block(None, 1, None, None, None, 0, None, None, None, None) == 1
    lib.dflash_destroy(None)
