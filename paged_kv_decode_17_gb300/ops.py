"""Torch-facing wrappers of the C ABI: argument marshalling only.

Every function takes CUDA tensors (the decode and writeback calls also take
pinned host tensors for their small per-step arguments: q, out, lse, the new
K/V rows, seq_lens, cu_seqlens), checks dtypes/shapes/contiguity, passes raw
pointers and the current CUDA stream to libpagedattn.so, and raises
``PagedAttnError`` on a non-zero status.  No arithmetic of the method happens
here and there is no CPU path.
"""

from __future__ import annotations

import math
from typing import Optional, Tuple

import torch

from . import _lib

_ws_cache = {}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t: torch.Tensor, name: str, dtype, ndim: int, host_ok: bool = False) -> None:
    """Check a tensor argument.  ``host_ok``: a pinned (page-locked) host
    tensor is accepted too; the kernels read or write it in place over the
    CPU-GPU link (NVLink-C2C on GB300), which for a decode step's small
    per-step tensors is cheaper than staging copies."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not (t.is_cuda or (host_ok and t.is_pinned())):
        raise ValueError("%s must be a CUDA tensor%s (there is no CPU path)"
                         % (name, " or a pinned host tensor" if host_ok else ""))
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.dim() != ndim:
        raise ValueError("%s must have %d dims, got shape %s" % (name, ndim, tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


class Workspace:
    """Device scratch for the split partials (and each sequence's first work
    unit).  Every call writes what it reads, so it needs no initialisation
    and may serve calls of any size that fits.  One workspace per stream that
    may run a call concurrently."""

    def __init__(self, nbytes: int, device):
        self.nbytes = int(max(nbytes, 256))
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


def decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(_lib.load().pa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim))


def decode_multiquery_workspace_bytes(batch: int, max_q_len: int, num_q_heads: int, num_kv_heads: int,
                                      head_dim: int) -> int:
    return int(_lib.load().pa_decode_multiquery_workspace_bytes(batch, max_q_len, num_q_heads, num_kv_heads,
                                                                head_dim))


def prefill_workspace_bytes(batch: int, total_q: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(_lib.load().pa_prefill_workspace_bytes(batch, total_q, num_q_heads, num_kv_heads, head_dim))


def _cached_ws(kind: str, nbytes: int, device) -> Workspace:
    key = (kind, torch.device(device).index, torch.cuda.current_stream(device).cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.nbytes < nbytes:
        ws = Workspace(nbytes, device)
        _ws_cache[key] = ws
    return ws


def new_status(device) -> torch.Tensor:
    """A zeroed int32 device status word."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(status: torch.Tensor, where: str = "kernel") -> None:
    """Synchronise and raise if a kernel recorded a device-side error."""
    v = int(status.item())
    if v != 0:
        raise _lib.PagedAttnError(v, where)


def kv_write_paged(k_pool: torch.Tensor, v_pool: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   cu_seqlens_new: torch.Tensor, seq_lens: torch.Tensor, block_table: torch.Tensor,
                   status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write the new K/V rows into their pages (in place on k_pool/v_pool)."""
    lib = _lib.load()
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(k_new, "k_new", torch.bfloat16, 3, host_ok=True)
    _need(v_new, "v_new", torch.bfloat16, 3, host_ok=True)
    _need(cu_seqlens_new, "cu_seqlens_new", torch.int32, 1, host_ok=True)
    _need(seq_lens, "seq_lens", torch.int32, 1, host_ok=True)
    _need(block_table, "block_table", torch.int32, 2)
    P, Hkv, ps, D = k_pool.shape
    if v_pool.shape != k_pool.shape or k_new.shape != v_new.shape or k_new.shape[1:] != (Hkv, D):
        raise ValueError("inconsistent K/V shapes")
    B = seq_lens.shape[0]
    if cu_seqlens_new.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens_new must have batch+1 entries and block_table batch rows")
    rc = lib.kv_write_paged(_ptr(k_pool), _ptr(v_pool), P, _ptr(k_new), _ptr(v_new), _ptr(cu_seqlens_new),
                            _ptr(seq_lens), _ptr(block_table), block_table.shape[1], B, k_new.shape[0], ps, Hkv, D,
                            _ptr(status), _stream_handle(stream))
    _lib.check(rc, "kv_write_paged")


def kv_write_paged_rope(k_pool: torch.Tensor, v_pool: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                        cu_seqlens_new: torch.Tensor, seq_lens: torch.Tensor, block_table: torch.Tensor,
                        rope_base: float = 10000.0, *, q: Optional[torch.Tensor] = None,
                        q_norm_weight: Optional[torch.Tensor] = None, k_norm_weight: Optional[torch.Tensor] = None,
                        norm_eps: float = 1e-6, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Writeback with the Q/K RMS norm (optional) and rotary embedding fused in.

    K rows are normalised (if ``k_norm_weight``) and rotated at their
    position before they are written; V rows are copied; ``q`` (the same
    tokens' queries, [total_new][Hq][D]) is normalised / rotated in place.
    """
    lib = _lib.load()
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(k_new, "k_new", torch.bfloat16, 3, host_ok=True)
    _need(v_new, "v_new", torch.bfloat16, 3, host_ok=True)
    _need(cu_seqlens_new, "cu_seqlens_new", torch.int32, 1, host_ok=True)
    _need(seq_lens, "seq_lens", torch.int32, 1, host_ok=True)
    _need(block_table, "block_table", torch.int32, 2)
    P, Hkv, ps, D = k_pool.shape
    if v_pool.shape != k_pool.shape or k_new.shape != v_new.shape or k_new.shape[1:] != (Hkv, D):
        raise ValueError("inconsistent K/V shapes")
    Hq = 0
    if q is not None:
        _need(q, "q", torch.bfloat16, 3, host_ok=True)
        if q.shape[0] != k_new.shape[0] or q.shape[2] != D:
            raise ValueError("q must be [total_new][Hq][head_dim]")
        Hq = q.shape[1]
    for name, w in (("q_norm_weight", q_norm_weight), ("k_norm_weight", k_norm_weight)):
        if w is not None:
            _need(w, name, torch.bfloat16, 1)
            if w.shape[0] != D:
                raise ValueError("%s must have head_dim entries" % name)
    B = seq_lens.shape[0]
    if cu_seqlens_new.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens_new must have batch+1 entries and block_table batch rows")
    rc = lib.kv_write_paged_rope(_ptr(k_pool), _ptr(v_pool), P, _ptr(k_new), _ptr(v_new), _ptr(q), Hq,
                                 _ptr(cu_seqlens_new), _ptr(seq_lens), _ptr(block_table), block_table.shape[1], B,
                                 k_new.shape[0], ps, Hkv, D, float(rope_base), _ptr(q_norm_weight),
                                 _ptr(k_norm_weight), float(norm_eps), _ptr(status), _stream_handle(stream))
    _lib.check(rc, "kv_write_paged_rope")


def _need_fp8_pools(k_pool, v_pool, k_scale, v_scale):
    _need(k_pool, "k_pool", torch.uint8, 4)
    _need(v_pool, "v_pool", torch.uint8, 4)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(v_scale, "v_scale", torch.float32, 1)
    P, Hkv, ps, D = k_pool.shape
    if v_pool.shape != (P, Hkv, D, ps):
        raise ValueError("v_pool must be [num_pages][Hkv][head_dim][page_size] (transposed per page block)")
    if k_scale.shape[0] != Hkv or v_scale.shape[0] != Hkv:
        raise ValueError("k_scale / v_scale must have one entry per KV head")
    return P, Hkv, ps, D


def kv_write_paged_fp8(k_pool: torch.Tensor, v_pool: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                       k_scale: torch.Tensor, v_scale: torch.Tensor, cu_seqlens_new: torch.Tensor,
                       seq_lens: torch.Tensor, block_table: torch.Tensor, status: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """Quantise the new K/V rows to e4m3 (x / scale[g], round to nearest even,
    saturating) and write them into the FP8 pools (V transposed per page block)."""
    lib = _lib.load()
    P, Hkv, ps, D = _need_fp8_pools(k_pool, v_pool, k_scale, v_scale)
    _need(k_new, "k_new", torch.bfloat16, 3, host_ok=True)
    _need(v_new, "v_new", torch.bfloat16, 3, host_ok=True)
    _need(cu_seqlens_new, "cu_seqlens_new", torch.int32, 1, host_ok=True)
    _need(seq_lens, "seq_lens", torch.int32, 1, host_ok=True)
    _need(block_table, "block_table", torch.int32, 2)
    if k_new.shape != v_new.shape or k_new.shape[1:] != (Hkv, D):
        raise ValueError("k_new / v_new must be [total_new][Hkv][head_dim]")
    B = seq_lens.shape[0]
    if cu_seqlens_new.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens_new must have batch+1 entries and block_table batch rows")
    rc = lib.kv_write_paged_fp8(_ptr(k_pool), _ptr(v_pool), P, _ptr(k_new), _ptr(v_new), _ptr(k_scale),
                                _ptr(v_scale), _ptr(cu_seqlens_new), _ptr(seq_lens), _ptr(block_table),
                                block_table.shape[1], B, k_new.shape[0], ps, Hkv, D, _ptr(status),
                                _stream_handle(stream))
    _lib.check(rc, "kv_write_paged_fp8")


def attn_decode_paged_fp8(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, k_scale: torch.Tensor,
                          v_scale: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                          softmax_scale: Optional[float] = None, *, max_seq_len: Optional[int] = None,
                          out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          return_lse: bool = False, workspace: Optional[Workspace] = None,
                          status: Optional[torch.Tensor] = None, stream=None):
    """Split-K paged decode over an FP8 (e4m3) cache with per-KV-head scales."""
    lib = _lib.load()
    _need(q, "q", torch.bfloat16, 3, host_ok=True)
    P, Hkv, ps, D = _need_fp8_pools(k_pool, v_pool, k_scale, v_scale)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1, host_ok=True)
    B, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("inconsistent head_dim")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens must have batch rows")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if max_seq_len is None:
        max_seq_len = block_table.shape[1] * ps
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=k_pool.device)
    else:
        _need(out, "out", torch.bfloat16, 3, host_ok=True)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=k_pool.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, host_ok=True)
    need = int(lib.pa_decode_workspace_bytes(B, Hq, Hkv, D)) if B > 0 else 0
    if workspace is None:
        workspace = _cached_ws("decode", need, k_pool.device)
    rc = lib.attn_decode_paged_fp8(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
                                   _ptr(v_scale), P, _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
                                   int(max_seq_len), ps, Hq, Hkv, D, float(softmax_scale), workspace.ptr,
                                   workspace.nbytes, _ptr(status), _stream_handle(stream))
    _lib.check(rc, "attn_decode_paged_fp8")
    return (out, lse) if return_lse else out


def attn_decode_paged(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, block_table: torch.Tensor,
                      seq_lens: torch.Tensor, softmax_scale: Optional[float] = None, *,
                      max_seq_len: Optional[int] = None, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, return_lse: bool = False,
                      workspace: Optional[Workspace] = None, status: Optional[torch.Tensor] = None,
                      k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                      stream=None):
    """Split-K paged decode, one query row per sequence.

    q [B][Hq][D] bf16; pools [P][Hkv][page_size][D] bf16; block_table
    [B][max_pages] int32; seq_lens [B] int32 (device).  ``max_seq_len`` is a
    host upper bound of seq_lens used only to size the launch (default: the
    table's capacity).  With ``k_new``/``v_new`` ([B][Hkv][D] bf16: each
    sequence's newest row, at position seq_lens[b] - 1) the rows are written
    into their pool slots by the same kernel (attn_decode_paged_append)
    instead of needing a kv_write_paged call first.  Returns out (and lse if
    requested).
    """
    lib = _lib.load()
    _need(q, "q", torch.bfloat16, 3, host_ok=True)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1, host_ok=True)
    B, Hq, D = q.shape
    P, Hkv, ps, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("inconsistent head_dim / pool shapes")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens must have batch rows")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if max_seq_len is None:
        max_seq_len = block_table.shape[1] * ps
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=k_pool.device)
    else:
        _need(out, "out", torch.bfloat16, 3, host_ok=True)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=k_pool.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, host_ok=True)
    need = int(lib.pa_decode_workspace_bytes(B, Hq, Hkv, D)) if B > 0 else 0
    if workspace is None:
        workspace = _cached_ws("decode", need, k_pool.device)
    if (k_new is None) != (v_new is None):
        raise ValueError("pass both k_new and v_new, or neither")
    if k_new is not None:
        _need(k_new, "k_new", torch.bfloat16, 3, host_ok=True)
        _need(v_new, "v_new", torch.bfloat16, 3, host_ok=True)
        if k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape:
            raise ValueError("k_new / v_new must be [batch][Hkv][head_dim]")
        rc = lib.attn_decode_paged_append(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_new),
                                          _ptr(v_new), P, _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                          B, int(max_seq_len), ps, Hq, Hkv, D, float(softmax_scale), workspace.ptr,
                                          workspace.nbytes, _ptr(status), _stream_handle(stream))
        _lib.check(rc, "attn_decode_paged_append")
    else:
        rc = lib.attn_decode_paged(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_pool), _ptr(v_pool), P, _ptr(block_table),
                                   block_table.shape[1], _ptr(seq_lens), B, int(max_seq_len), ps, Hq, Hkv, D,
                                   float(softmax_scale), workspace.ptr, workspace.nbytes, _ptr(status),
                                   _stream_handle(stream))
        _lib.check(rc, "attn_decode_paged")
    return (out, lse) if return_lse else out


def attn_decode_multiquery_paged(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                 block_table: torch.Tensor, cu_seqlens_q: torch.Tensor, seq_lens: torch.Tensor,
                                 softmax_scale: Optional[float] = None, *, max_q_len: Optional[int] = None,
                                 max_seq_len: Optional[int] = None, out: Optional[torch.Tensor] = None,
                                 lse: Optional[torch.Tensor] = None, return_lse: bool = False,
                                 workspace: Optional[Workspace] = None, status: Optional[torch.Tensor] = None,
                                 k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                                 stream=None):
    """Multi-query decode: 1..8 query rows per sequence, causal inside the block.

    q [total_q][Hq][D] bf16; cu_seqlens_q [B+1] int32; seq_lens [B] int32
    (total keys, the query rows' own K/V already written).  ``max_q_len``
    (1..8, default min(8, total_q)) is a host upper bound of the per-entry
    row counts; it sizes the workspace and the launch.  With ``k_new`` /
    ``v_new`` ([total_q][Hkv][D] bf16, the query tokens' own K/V rows) the
    rows are written into their pool slots by the same kernel
    (attn_decode_multiquery_paged_append) instead of needing kv_write_paged
    first.
    """
    lib = _lib.load()
    _need(q, "q", torch.bfloat16, 3, host_ok=True)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, host_ok=True)
    _need(seq_lens, "seq_lens", torch.int32, 1, host_ok=True)
    Tq, Hq, D = q.shape
    P, Hkv, ps, D2 = k_pool.shape
    B = seq_lens.shape[0]
    if D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("inconsistent head_dim / pool shapes")
    if cu_seqlens_q.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens_q must have batch+1 entries and block_table batch rows")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if max_seq_len is None:
        max_seq_len = block_table.shape[1] * ps
    if max_q_len is None:
        max_q_len = max(1, min(8, Tq))
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=k_pool.device)
    else:
        _need(out, "out", torch.bfloat16, 3, host_ok=True)
    if return_lse and lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=k_pool.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, host_ok=True)
    need = int(lib.pa_decode_multiquery_workspace_bytes(B, int(max_q_len), Hq, Hkv, D)) if B > 0 else 0
    if workspace is None:
        workspace = _cached_ws("decode", need, k_pool.device)
    if (k_new is None) != (v_new is None):
        raise ValueError("pass both k_new and v_new, or neither")
    if k_new is not None:
        _need(k_new, "k_new", torch.bfloat16, 3, host_ok=True)
        _need(v_new, "v_new", torch.bfloat16, 3, host_ok=True)
        if k_new.shape != (Tq, Hkv, D) or v_new.shape != k_new.shape:
            raise ValueError("k_new / v_new must be [total_q][Hkv][head_dim]")
        rc = lib.attn_decode_multiquery_paged_append(
            _ptr(out), _ptr(lse), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new), P,
            _ptr(block_table), block_table.shape[1], _ptr(cu_seqlens_q), _ptr(seq_lens), B, Tq, int(max_q_len),
            int(max_seq_len), ps, Hq, Hkv, D, float(softmax_scale), workspace.ptr, workspace.nbytes, _ptr(status),
            _stream_handle(stream))
        _lib.check(rc, "attn_decode_multiquery_paged_append")
    else:
        rc = lib.attn_decode_multiquery_paged(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_pool), _ptr(v_pool), P,
                                              _ptr(block_table), block_table.shape[1], _ptr(cu_seqlens_q),
                                              _ptr(seq_lens), B, Tq, int(max_q_len), int(max_seq_len), ps, Hq, Hkv,
                                              D, float(softmax_scale), workspace.ptr, workspace.nbytes, _ptr(status),
                                              _stream_handle(stream))
        _lib.check(rc, "attn_decode_multiquery_paged")
    return (out, lse) if return_lse else out


def attn_prefill_varlen_causal(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                               block_table: torch.Tensor, cu_seqlens_q: torch.Tensor, seq_lens: torch.Tensor,
                               softmax_scale: Optional[float] = None, *, max_q_len: Optional[int] = None,
                               max_seq_len: Optional[int] = None, out: Optional[torch.Tensor] = None,
                               lse: Optional[torch.Tensor] = None, return_lse: bool = False,
                               workspace: Optional[Workspace] = None, status: Optional[torch.Tensor] = None,
                               stream=None):
    """Varlen causal attention over paged K/V (bottom-right aligned).

    q [total_q][Hq][D] bf16; cu_seqlens_q [B+1] int32; seq_lens [B] int32
    (total keys per sequence, the query rows' own K/V already written).
    ``max_q_len``/``max_seq_len`` are host upper bounds used only to size the
    launch (defaults: total_q and the table's capacity).
    """
    lib = _lib.load()
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    Tq, Hq, D = q.shape
    P, Hkv, ps, D2 = k_pool.shape
    B = seq_lens.shape[0]
    if D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("inconsistent head_dim / pool shapes")
    if cu_seqlens_q.shape[0] != B + 1 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens_q must have batch+1 entries and block_table batch rows")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if max_seq_len is None:
        max_seq_len = block_table.shape[1] * ps
    if max_q_len is None:
        max_q_len = Tq
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, 3)
    if return_lse and lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    need = int(lib.pa_prefill_workspace_bytes(B, Tq, Hq, Hkv, D)) if B > 0 else 0
    if workspace is None:
        workspace = _cached_ws("prefill", need, q.device)
    rc = lib.attn_prefill_varlen_causal(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_pool), _ptr(v_pool), P,
                                        _ptr(block_table), block_table.shape[1], _ptr(cu_seqlens_q), _ptr(seq_lens),
                                        B, Tq, int(max_q_len), int(max_seq_len), ps, Hq, Hkv, D,
                                        float(softmax_scale), workspace.ptr, workspace.nbytes, _ptr(status),
                                        _stream_handle(stream))
    _lib.check(rc, "attn_prefill_varlen_causal")
    return (out, lse) if return_lse else out
