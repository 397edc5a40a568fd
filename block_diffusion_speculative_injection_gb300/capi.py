"""ctypes binding of libdflash.so: the C ABI of include/dflash.h, same names.

Argument marshalling only: torch tensors are passed as raw device pointers
and the caller's current CUDA stream is passed as the stream handle.  Every
step of the computation runs in the library's CUDA kernels.  If the shared
library is missing, loading raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdflash.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "dflash.h")

DFLASH_F32, DFLASH_BF16, DFLASH_I32 = 0, 1, 2
DFLASH_ACCEPT_GREEDY, DFLASH_ACCEPT_ALL, DFLASH_ACCEPT_GIVEN = 0, 1, 2
DFLASH_VERIFY_LAST_ONLY = 1

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "CAPACITY", 3: "OOM", 4: "CUDA", 5: "DEVICE_CHECK",
          6: "TIMEOUT", 7: "UNSUPPORTED", 8: "STATE"}


class DFlashError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"dflash status {status} ({STATUS.get(status, '?')}): {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int32), ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32), ("vocab", ctypes.c_int32),
        ("n_target_layers", ctypes.c_int32), ("n_draft_layers", ctypes.c_int32),
        ("n_inject", ctypes.c_int32), ("inject_layers", ctypes.c_int32 * 16),
        ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
        ("block_size", ctypes.c_int32), ("max_batch", ctypes.c_int32),
        ("max_ctx", ctypes.c_int32), ("max_rows", ctypes.c_int32),
        ("max_tree_nodes", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("kv_pages", ctypes.c_int32),
    ]


PAGE_SLOTS = 128  # DFLASH_PAGE_SLOTS: cache slots per KV page


class DTree(ctypes.Structure):
    _fields_ = [
        ("tok", ctypes.c_void_p), ("parent", ctypes.c_void_p), ("depth", ctypes.c_void_p),
        ("anc", ctypes.c_void_p), ("n_nodes", ctypes.c_void_p),
        ("max_nodes", ctypes.c_int32), ("anc_words", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIGS = {
    "dflash_create": ([ctypes.POINTER(Config), ctypes.POINTER(_P)], _I),
    "dflash_set_weight": ([_P, ctypes.c_char_p, _P, _I, ctypes.POINTER(ctypes.c_int64), _I], _I),
    "dflash_reset_seq": ([_P, _I, _P], _I),
    "dflash_kv_reserve": ([_P, _I, _I, _P], _I),
    "dflash_injection_rows": ([_P, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                               ctypes.POINTER(_I)], _I),
    "dflash_advance_lengths": ([_P, _I, _P, _P, _P], _I),
    "dflash_kv_release": ([_P, _I, _P], _I),
    "dflash_kv_free_pages": ([_P], _I),
    "dflash_kv_pool_create": ([_I, _I, _I], _P),
    "dflash_kv_pool_destroy": ([_P], None),
    "dflash_kv_pool_reserve": ([_P, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)], _I),
    "dflash_kv_pool_release": ([_P, _I], _I),
    "dflash_kv_pool_pages": ([_P, _I, _P, _I], _I),
    "dflash_kv_pool_free": ([_P], _I),
    "dflash_verify": ([_P, _I, _P, _P, _I, _P, _I, _P, _P, _P, _P], _I),
    "dflash_draft_block": ([_P, _I, _P, _P, _P, _I, _P, _P, _P, _P], _I),
    "dflash_set_block_size": ([_P, _I], _I),
    "dflash_accept_commit": ([_P, _I, _P, _P, _P, ctypes.POINTER(DTree), _I, _P, _P, _P, _P], _I),
    "dflash_inject_kv": ([_P, _I, _P, _P, _P, _P], _I),
    "dtree_build": ([_P, _I, _P, _P, _P, _I, _I, ctypes.POINTER(DTree), _P], _I),
    "dtree_verify": ([_P, _I, _P, ctypes.POINTER(DTree), _P, _P, _P, _P], _I),
    "dflash_check": ([_P], _I),
    "dflash_last_error": ([_P], ctypes.c_char_p),
    "dflash_seq_lengths": ([_P], _P),
    "dflash_launch_count": ([_P], ctypes.c_int64),
    "dflash_debug_view": ([_P, ctypes.c_char_p, _I, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_int64)], _I),
    "dflash_destroy": ([_P], None),
    "dflash_block_attention": ([_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, ctypes.c_int64, _P], _I),
    "dflash_block_attention_workspace": ([_I, _I, _I, _I, _I], ctypes.c_int64),
    "dflash_block_attention_noalloc": ([_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "dflash_debug_wait_timeout": ([_P, _P], _I),
    "dflash_sample_workspace": ([_I, _I], ctypes.c_int64),
    "dflash_sample_rows": ([_I, _I, _P, _P, _P, _P, ctypes.c_int64, _P], _I),
    "dflash_spec_accept_workspace": ([_I, _I, _I], ctypes.c_int64),
    "dflash_spec_accept_sampled": ([_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int64, _P],
                                   _I),
    "dflash_plan_gemm": ([_I, _I, _I, _I, _I, _I, _P], _I),
    "dflash_plan_attention": ([_I, _I, _I, _I, _I, ctypes.c_int64, _I, _P], _I),
    "dflash_profile": ([_P, _I], _I),
    "dflash_debug_trace": ([_P, _P, ctypes.c_int64], _I),
    "dflash_debug_trace_draft": ([_P, _P, ctypes.c_int64], _I),
    "dflash_debug_trace_draft_attn": ([_P, _P, _P, ctypes.c_int64], _I),
    "dflash_profile_list": ([_P, _I, _P, _P, ctypes.c_int64], ctypes.c_int64),
    "dflash_profile_read": ([_P, _I, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double),
                             ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)], _I),
}

_lib: Optional[ctypes.CDLL] = None


def header_functions():
    """Names of the functions declared in include/dflash.h."""
    with open(HEADER) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:dflash|dtree)_[a-z_]+)\s*\(", src)))


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads libdflash.so (raises if it has not been built).  DFLASH_LIB_PATH
    names another build of the same library (e.g. one compiled with
    different tuning flags)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = os.environ.get("DFLASH_LIB_PATH", LIB_PATH)
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (args, ret) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ret
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(ctx, status: int) -> None:
    if status != 0:
        msg = load().dflash_last_error(ctx).decode() if ctx else ""
        raise DFlashError(status, msg)


# ---------------------------------------------------------------------------
# the C ABI, one wrapper per function (raises DFlashError on a non-OK status)
# ---------------------------------------------------------------------------

def dflash_create(cfg: Config) -> int:
    h = _P()
    st = load().dflash_create(ctypes.byref(cfg), ctypes.byref(h))
    if st != 0:
        raise DFlashError(st, "dflash_create rejected the configuration")
    return h.value


def dflash_destroy(ctx: int) -> None:
    load().dflash_destroy(ctx)


def dflash_set_weight(ctx: int, name: str, tensor, dtype: int) -> None:
    shape = (ctypes.c_int64 * tensor.dim())(*tensor.shape)
    _check(ctx, load().dflash_set_weight(ctx, name.encode(), _ptr(tensor), dtype, shape, tensor.dim()))


def dflash_reset_seq(ctx: int, seq_id: int, stream=None) -> None:
    _check(ctx, load().dflash_reset_seq(ctx, seq_id, _stream(stream)))


def dflash_injection_rows(ctx):
    """(hidden, row_seq, row_pos device pointers, rows) of the pending injection queue."""
    h, rs, rp, n = _P(), _P(), _P(), _I()
    _check(ctx, load().dflash_injection_rows(ctx, ctypes.byref(h), ctypes.byref(rs), ctypes.byref(rp),
                                             ctypes.byref(n)))
    return h.value, rs.value, rp.value, n.value


def dflash_advance_lengths(ctx, batch: int, seq_ids, counts, stream=None) -> None:
    _check(ctx, load().dflash_advance_lengths(ctx, batch, _ptr(seq_ids), _ptr(counts),
                                              _stream(stream)))


def dflash_kv_reserve(ctx, seq_id: int, n_slots: int, stream=None) -> None:
    _check(ctx, load().dflash_kv_reserve(ctx, seq_id, n_slots, _stream(stream)))


def dflash_kv_release(ctx, seq_id: int, stream=None) -> None:
    _check(ctx, load().dflash_kv_release(ctx, seq_id, _stream(stream)))


def dflash_kv_free_pages(ctx) -> int:
    return load().dflash_kv_free_pages(ctx)


class KvPool:
    """The host page allocator (dflash_kv_pool_*), no GPU needed."""

    def __init__(self, n_pages: int, max_seqs: int, max_pages: int):
        self.h = load().dflash_kv_pool_create(n_pages, max_seqs, max_pages)
        if not self.h:
            raise DFlashError(1, "dflash_kv_pool_create")

    def reserve(self, seq: int, n_slots: int):
        """(first new table index, pages added); raises DFlashError when refused."""
        f, n = _I(), _I()
        st = load().dflash_kv_pool_reserve(self.h, seq, n_slots, ctypes.byref(f), ctypes.byref(n))
        if st != 0:
            raise DFlashError(st, "dflash_kv_pool_reserve")
        return f.value, n.value

    def release(self, seq: int) -> int:
        return load().dflash_kv_pool_release(self.h, seq)

    def pages(self, seq: int) -> list:
        n = load().dflash_kv_pool_pages(self.h, seq, None, 0)
        if n < 0:
            raise DFlashError(1, "dflash_kv_pool_pages")
        buf = (_I * max(n, 1))()
        load().dflash_kv_pool_pages(self.h, seq, ctypes.addressof(buf), n)
        return list(buf)[:n]

    def free(self) -> int:
        return load().dflash_kv_pool_free(self.h)

    def close(self) -> None:
        if self.h:
            load().dflash_kv_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dflash_verify(ctx, batch, seq_ids, tokens, q, q_lens, flags, argmax, margin=None, logits=None,
                  stream=None) -> None:
    _check(ctx, load().dflash_verify(ctx, batch, _ptr(seq_ids), _ptr(tokens), q, _ptr(q_lens), flags,
                                     _ptr(argmax), _ptr(margin), _ptr(logits), _stream(stream)))


def dflash_set_block_size(ctx, block: int) -> None:
    _check(ctx, load().dflash_set_block_size(ctx, block))


def dflash_draft_block(ctx, batch, seq_ids, anchor, block, topk=0, topk_ids=None, topk_logp=None,
                       logits=None, stream=None) -> None:
    _check(ctx, load().dflash_draft_block(ctx, batch, _ptr(seq_ids), _ptr(anchor), _ptr(block), topk,
                                          _ptr(topk_ids), _ptr(topk_logp), _ptr(logits),
                                          _stream(stream)))


def dflash_accept_commit(ctx, batch, seq_ids, block, argmax, tree, mode, accept_len, next_anchor,
                         emitted, stream=None) -> None:
    tp = ctypes.byref(tree) if tree is not None else None
    _check(ctx, load().dflash_accept_commit(ctx, batch, _ptr(seq_ids), _ptr(block), _ptr(argmax), tp,
                                            mode, _ptr(accept_len), _ptr(next_anchor), _ptr(emitted),
                                            _stream(stream)))


def dflash_inject_kv(ctx, n_rows=0, row_seq=None, row_pos=None, hidden=None, stream=None) -> None:
    _check(ctx, load().dflash_inject_kv(ctx, n_rows, _ptr(row_seq), _ptr(row_pos), _ptr(hidden),
                                        _stream(stream)))


def dtree_build(ctx, batch, anchor, topk_ids, topk_logp, topk, budget, tree: DTree,
                stream=None) -> None:
    _check(ctx, load().dtree_build(ctx, batch, _ptr(anchor), _ptr(topk_ids), _ptr(topk_logp), topk,
                                   budget, ctypes.byref(tree), _stream(stream)))


def dtree_verify(ctx, batch, seq_ids, tree: DTree, node_argmax, margin=None, logits=None,
                 stream=None) -> None:
    _check(ctx, load().dtree_verify(ctx, batch, _ptr(seq_ids), ctypes.byref(tree), _ptr(node_argmax),
                                    _ptr(margin), _ptr(logits), _stream(stream)))


def dflash_check(ctx) -> None:
    _check(ctx, load().dflash_check(ctx))


def dflash_last_error(ctx) -> str:
    return load().dflash_last_error(ctx).decode()


def dflash_seq_lengths(ctx) -> int:
    return load().dflash_seq_lengths(ctx)


def dflash_launch_count(ctx) -> int:
    return int(load().dflash_launch_count(ctx))


def dflash_debug_view(ctx, name: str, layer: int = 0):
    p = _P()
    n = ctypes.c_int64()
    _check(ctx, load().dflash_debug_view(ctx, name.encode(), layer, ctypes.byref(p), ctypes.byref(n)))
    return p.value, n.value


def dflash_block_attention(batch, n_heads, n_kv_heads, ctx_len, block, causal, q, k, v, out,
                           workspace=None, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().dflash_block_attention(batch, n_heads, n_kv_heads, ctx_len, block, causal, _ptr(q),
                                       _ptr(k), _ptr(v), _ptr(out), _ptr(workspace), nbytes,
                                       _stream(stream))
    if st != 0:
        raise DFlashError(st, "dflash_block_attention")


def dflash_block_attention_workspace(batch, n_heads, n_kv_heads, ctx_len, block) -> int:
    return int(load().dflash_block_attention_workspace(batch, n_heads, n_kv_heads, ctx_len, block))


def dflash_plan_gemm(sm_count, M, N, K, kind, max_splits=8) -> dict:
    """Launch plan of the tensor-core GEMM (host arithmetic; no GPU needed)."""
    out = (ctypes.c_int32 * 8)()
    st = load().dflash_plan_gemm(sm_count, M, N, K, kind, max_splits, ctypes.addressof(out))
    if st != 0:
        raise DFlashError(st, "dflash_plan_gemm")
    keys = ("BN", "m_tiles", "n_tiles", "stages", "splits", "threads", "smem_bytes", "persistent")
    return dict(zip(keys, list(out)))


def dflash_plan_attention(sm_count, batch, n_heads, n_kv_heads, q_per_seq, max_keys,
                          min_splits=1) -> dict:
    """Split-KV plan of the bf16 attention (host arithmetic; no GPU needed)."""
    out = (ctypes.c_int32 * 3)()
    st = load().dflash_plan_attention(sm_count, batch, n_heads, n_kv_heads, q_per_seq, max_keys,
                                      min_splits, ctypes.addressof(out))
    if st != 0:
        raise DFlashError(st, "dflash_plan_attention")
    return dict(zip(("splits", "keys_per_split", "ctas"), list(out)))


def dflash_profile(ctx, enable: bool) -> None:
    _check(ctx, load().dflash_profile(ctx, 1 if enable else 0))


PROF_GEMM, PROF_ATTN, PROF_ROW, PROF_VOCAB, PROF_SPEC, PROF_ALL = 0, 1, 2, 3, 4, -1


def dflash_profile_list(ctx, kind: int):
    """Per-launch (ms, flops) of the recorded launches of one class."""
    n = load().dflash_profile_list(ctx, kind, None, None, 0)
    if n < 0:
        raise DFlashError(4, "dflash_profile_list")
    ms = (ctypes.c_double * max(n, 1))()
    fl = (ctypes.c_double * max(n, 1))()
    load().dflash_profile_list(ctx, kind, ctypes.addressof(ms), ctypes.addressof(fl), n)
    return list(zip(list(ms)[:n], list(fl)[:n]))


def dflash_profile_read(ctx, kind: int):
    """(launches, ms, algorithmic bytes, flops) of one kernel class."""
    n = ctypes.c_int64()
    ms, b, f = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(ctx, load().dflash_profile_read(ctx, kind, ctypes.byref(n), ctypes.byref(ms),
                                           ctypes.byref(b), ctypes.byref(f)))
    return n.value, ms.value, b.value, f.value


def dflash_block_attention_noalloc(batch, n_heads, n_kv_heads, ctx_len, block, causal, q, k, v, out,
                                   stream=None) -> None:
    """Block attention with the library's fixed scratch array (no allocation)."""
    st = load().dflash_block_attention_noalloc(batch, n_heads, n_kv_heads, ctx_len, block, causal,
                                               _ptr(q), _ptr(k), _ptr(v), _ptr(out), _stream(stream))
    if st != 0:
        raise DFlashError(st, "dflash_block_attention_noalloc")


def dflash_debug_wait_timeout(ctx, stream=None) -> None:
    """Runs a bounded wait that expires (about 2 s) and records a timeout."""
    st = load().dflash_debug_wait_timeout(ctx, _stream(stream))
    if st != 0:
        raise DFlashError(st, "dflash_debug_wait_timeout")


def dflash_sample_workspace(rows, vocab) -> int:
    return int(load().dflash_sample_workspace(rows, vocab))


def dflash_sample_rows(rows, vocab, logits, u, tokens, workspace, stream=None) -> None:
    """One temperature-1 draw per row of fp32 logits [rows][vocab] (uniforms u [rows])."""
    nbytes = workspace.numel() * workspace.element_size()
    st = load().dflash_sample_rows(rows, vocab, _ptr(logits), _ptr(u), _ptr(tokens), _ptr(workspace),
                                   nbytes, _stream(stream))
    if st != 0:
        raise DFlashError(st, "dflash_sample_rows")


def dflash_spec_accept_workspace(batch, block, vocab) -> int:
    return int(load().dflash_spec_accept_workspace(batch, block, vocab))


def dflash_spec_accept_sampled(batch, block, vocab, draft_logits, target_logits, tokens, u_accept,
                               u_resample, accept_len, emitted, workspace, stream=None) -> None:
    """Temperature-1 acceptance of one block per sequence (speculative rejection rule)."""
    nbytes = workspace.numel() * workspace.element_size()
    st = load().dflash_spec_accept_sampled(batch, block, vocab, _ptr(draft_logits), _ptr(target_logits),
                                           _ptr(tokens), _ptr(u_accept), _ptr(u_resample),
                                           _ptr(accept_len), _ptr(emitted), _ptr(workspace), nbytes,
                                           _stream(stream))
    if st != 0:
        raise DFlashError(st, "dflash_spec_accept_sampled")


def dflash_debug_trace(ctx, dst=None) -> None:
    """Registers (or clears with None) a [L][max_rows][d] fp32 residual trace."""
    nbytes = dst.numel() * dst.element_size() if dst is not None else 0
    _check(ctx, load().dflash_debug_trace(ctx, _ptr(dst), nbytes))


def dflash_debug_trace_draft(ctx, dst=None) -> None:
    """Registers (or clears with None) a [L_d][max_rows][d] fp32 residual trace
    of the draft passes."""
    nbytes = dst.numel() * dst.element_size() if dst is not None else 0
    _check(ctx, load().dflash_debug_trace_draft(ctx, _ptr(dst), nbytes))


def dflash_debug_trace_draft_attn(ctx, q=None, attn=None) -> None:
    """Registers (or clears with None) per-draft-layer copies of the roped
    queries and of the attention output, [L_d][max_rows][H*hd] each."""
    t = q if q is not None else attn
    nbytes = t.numel() * t.element_size() if t is not None else 0
    _check(ctx, load().dflash_debug_trace_draft_attn(ctx, _ptr(q), _ptr(attn), nbytes))
