"""ctypes loader for libpagedattn.so (the C ABI declared in include/pagedattn.h).

The library is built in-tree by ``paged_kv_decode_17_gb300.build``.  There is
no fallback: if the shared library is missing every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

c_void_p = ctypes.c_void_p
c_int = ctypes.c_int
c_float = ctypes.c_float
c_size_t = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/pagedattn.h
SIGNATURES = {
    "pa_abi_version": (c_int, []),
    "pa_status_string": (ctypes.c_char_p, [c_int]),
    "pa_decode_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int]),
    "attn_decode_paged": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,  # out, lse, q, k_pool, v_pool
        c_int, c_void_p, c_int,  # num_pages, block_table, max_pages_per_seq
        c_void_p, c_int, c_int, c_int,  # seq_lens, batch, max_seq_len, page_size
        c_int, c_int, c_int, c_float,  # Hq, Hkv, D, scale
        c_void_p, c_size_t, c_void_p, c_void_p,  # workspace, bytes, status, stream
    ]),
    "attn_decode_paged_append": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,  # out, lse, q, k_pool, v_pool
        c_void_p, c_void_p,  # k_new, v_new
        c_int, c_void_p, c_int,  # num_pages, block_table, max_pages_per_seq
        c_void_p, c_int, c_int, c_int,  # seq_lens, batch, max_seq_len, page_size
        c_int, c_int, c_int, c_float,  # Hq, Hkv, D, scale
        c_void_p, c_size_t, c_void_p, c_void_p,  # workspace, bytes, status, stream
    ]),
    "attn_decode_paged_noalloc": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,  # out, lse, q, k_pool, v_pool
        c_int, c_void_p, c_int,  # num_pages, block_table, max_pages_per_seq
        c_void_p, c_int, c_int, c_int,  # seq_lens, batch, max_seq_len, page_size
        c_int, c_int, c_int, c_float,  # Hq, Hkv, D, scale
        c_void_p, c_void_p,  # status, stream
    ]),
    "pa_decode_multiquery_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_decode_multiquery_paged": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,  # out, lse, q, k_pool, v_pool
        c_int, c_void_p, c_int,  # num_pages, block_table, max_pages_per_seq
        c_void_p, c_void_p,  # cu_seqlens_q, seq_lens
        c_int, c_int, c_int, c_int,  # batch, total_q, max_q_len, max_seq_len
        c_int, c_int, c_int, c_int, c_float,  # page_size, Hq, Hkv, D, scale
        c_void_p, c_size_t, c_void_p, c_void_p,  # workspace, bytes, status, stream
    ]),
    "attn_decode_multiquery_paged_append": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,  # out, lse, q, k_pool, v_pool
        c_void_p, c_void_p,  # k_new, v_new
        c_int, c_void_p, c_int,  # num_pages, block_table, max_pages_per_seq
        c_void_p, c_void_p,  # cu_seqlens_q, seq_lens
        c_int, c_int, c_int, c_int,  # batch, total_q, max_q_len, max_seq_len
        c_int, c_int, c_int, c_int, c_float,  # page_size, Hq, Hkv, D, scale
        c_void_p, c_size_t, c_void_p, c_void_p,  # workspace, bytes, status, stream
    ]),
    "pa_prefill_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_prefill_varlen_causal": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,  # out, lse, q, k_pool, v_pool
        c_int, c_void_p, c_int,  # num_pages, block_table, max_pages_per_seq
        c_void_p, c_void_p,  # cu_seqlens_q, seq_lens
        c_int, c_int, c_int, c_int,  # batch, total_q, max_q_len, max_seq_len
        c_int, c_int, c_int, c_int, c_float,  # page_size, Hq, Hkv, D, scale
        c_void_p, c_size_t, c_void_p, c_void_p,  # workspace, bytes, status, stream
    ]),
    "kv_write_paged_rope": (c_int, [
        c_void_p, c_void_p, c_int, c_void_p, c_void_p,  # k_pool, v_pool, num_pages, k_new, v_new
        c_void_p, c_int,  # q (nullable), num_q_heads
        c_void_p, c_void_p, c_void_p, c_int,  # cu_seqlens_new, seq_lens, block_table, max_pages
        c_int, c_int, c_int, c_int, c_int,  # batch, total_new, page_size, Hkv, D
        c_float, c_void_p, c_void_p, c_float,  # rope_base, q_norm_weight, k_norm_weight, norm_eps
        c_void_p, c_void_p,  # status, stream
    ]),
    "kv_write_paged_fp8": (c_int, [
        c_void_p, c_void_p, c_int, c_void_p, c_void_p,  # k_pool, v_pool, num_pages, k_new, v_new
        c_void_p, c_void_p,  # k_scale, v_scale
        c_void_p, c_void_p, c_void_p, c_int,  # cu_seqlens_new, seq_lens, block_table, max_pages
        c_int, c_int, c_int, c_int, c_int,  # batch, total_new, page_size, Hkv, D
        c_void_p, c_void_p,  # status, stream
    ]),
    "attn_decode_paged_fp8": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,  # out, lse, q, k_pool, v_pool
        c_void_p, c_void_p,  # k_scale, v_scale
        c_int, c_void_p, c_int,  # num_pages, block_table, max_pages_per_seq
        c_void_p, c_int, c_int, c_int,  # seq_lens, batch, max_seq_len, page_size
        c_int, c_int, c_int, c_float,  # Hq, Hkv, D, scale
        c_void_p, c_size_t, c_void_p, c_void_p,  # workspace, bytes, status, stream
    ]),
    "kv_write_paged": (c_int, [
        c_void_p, c_void_p, c_int, c_void_p, c_void_p,  # k_pool, v_pool, num_pages, k_new, v_new
        c_void_p, c_void_p, c_void_p, c_int,  # cu_seqlens_new, seq_lens, block_table, max_pages
        c_int, c_int, c_int, c_int, c_int,  # batch, total_new, page_size, Hkv, D
        c_void_p, c_void_p,  # status, stream
    ]),
}


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libpagedattn.so (optionally building it first)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    "libpagedattn.so is not built (expected at %s); run "
                    "paged_kv_decode_17_gb300.build.build() first" % path)
            _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name, None)
            if fn is None:
                continue  # reported by missing_symbols()
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def missing_symbols(lib: ctypes.CDLL, names) -> list:
    out = []
    for n in names:
        try:
            getattr(lib, n)
        except AttributeError:
            out.append(n)
    return out


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = "unknown"
        try:
            msg = load().pa_status_string(code).decode()
        except Exception:  # pragma: no cover - message lookup only
            pass
        super().__init__("%s failed: status %d (%s)" % (where, code, msg))
        self.code = code


def check(code: int, where: str) -> None:
    if code != 0:
        raise PagedAttnError(code, where)
