"""The C ABI without a GPU: the library builds, loads, exports every function
include/pagedattn.h declares, and rejects bad arguments on the host before
touching the device."""

import ctypes
import os
import re

import pytest

import paged_kv_decode_17_gb300 as pa
from paged_kv_decode_17_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedattn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"#[^\n]*", "", text)
    names = re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\([^;{}]*\)\s*;", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_three_operations():
    names = _declared_functions()
    for n in ("attn_decode_paged", "attn_prefill_varlen_causal", "kv_write_paged"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    names = _declared_functions()
    missing = _lib.missing_symbols(lib, names)
    assert not missing, "declared but not exported: %s" % missing
    # and the binding knows every one of them
    assert set(names) <= set(_lib.SIGNATURES), set(names) - set(_lib.SIGNATURES)


def test_status_strings(lib):
    assert lib.pa_abi_version() >= 1
    for code in range(-8, 1):
        s = lib.pa_status_string(code).decode()
        assert s and s != "unknown status"


def _decode_args(**over):
    a = dict(out=1 << 20, lse=None, q=1 << 20, k=1 << 20, v=1 << 20, num_pages=16, bt=1 << 20, maxp=8,
             lens=1 << 20, batch=2, max_seq_len=100, ps=16, hq=4, hkv=2, d=64, scale=0.125, ws=None, wsb=0,
             status=None, stream=None)
    a.update(over)
    return [a[k] for k in ("out", "lse", "q", "k", "v", "num_pages", "bt", "maxp", "lens", "batch", "max_seq_len",
                           "ps", "hq", "hkv", "d", "scale", "ws", "wsb", "status", "stream")]


@pytest.mark.parametrize("over,code", [
    (dict(hq=3), -2),            # Hq not a multiple of Hkv
    (dict(d=96), -2),            # unsupported head_dim
    (dict(ps=8), -2),            # page size not a multiple of 16
    (dict(ps=24), -2),
    (dict(max_seq_len=1000), -2),  # more than the table can hold
    (dict(q=None), -1),
    (dict(bt=None), -1),
    (dict(batch=-1), -2),
])
def test_decode_host_validation(lib, over, code):
    assert lib.attn_decode_paged(*_decode_args(**over)) == code


def _append_args(k_new=1 << 20, v_new=1 << 20, **over):
    a = _decode_args(**over)
    return a[:5] + [k_new, v_new] + a[5:]


@pytest.mark.parametrize("kw,code", [
    (dict(k_new=None), -1),           # the new rows are required
    (dict(v_new=None), -1),
    (dict(k_new=(1 << 20) + 8), -2),  # 16-byte alignment
    (dict(hq=3), -2),
    (dict(q=None), -1),
])
def test_append_host_validation(lib, kw, code):
    assert lib.attn_decode_paged_append(*_append_args(**kw)) == code


def test_multiquery_append_host_validation(lib):
    f = lib.attn_decode_multiquery_paged_append
    P = 1 << 20
    # out, lse, q, k, v, k_new, v_new, num_pages, bt, maxp, cu_q, lens, batch, total_q, max_q_len, max_seq_len,
    # ps, hq, hkv, d, scale, ws, wsb, status, stream
    args = [P, None, P, P, P, P, P, 16, P, 8, P, P, 2, 4, 2, 100, 16, 4, 2, 64, 0.125, None, 0, None, None]
    for i, code in ((5, -1), (6, -1), (10, -1)):  # k_new, v_new, cu_seqlens_q missing
        bad = list(args)
        bad[i] = None
        assert f(*bad) == code
    bad = list(args)
    bad[14] = 9  # more than 8 query rows
    assert f(*bad) == -2
    bad = list(args)
    bad[17] = 3  # Hq not a multiple of Hkv
    assert f(*bad) == -2


def test_append_empty_batch_is_a_noop(lib):
    assert lib.attn_decode_paged_append(*_append_args(k_new=None, v_new=None, batch=0, q=None, out=None)) == 0


def test_decode_empty_batch_is_a_noop(lib):
    assert lib.attn_decode_paged(*_decode_args(batch=0, q=None, out=None)) == 0


def test_kv_write_host_validation(lib):
    f = lib.kv_write_paged
    P = 1 << 20
    assert f(P, P, 8, P, P, P, P, P, 4, 2, 10, 16, 2, 96, None, None) == -2
    assert f(P, P, 8, P, P, P, P, P, 4, 2, 10, 12, 2, 64, None, None) == -2
    assert f(None, P, 8, P, P, P, P, P, 4, 2, 10, 16, 2, 64, None, None) == -1
    assert f(P, P, 8, P, P, P, P, P, 4, 0, 0, 16, 2, 64, None, None) == 0  # nothing to write


def test_prefill_host_validation(lib):
    f = lib.attn_prefill_varlen_causal
    P = 1 << 20
    args = [P, None, P, P, P, 16, P, 8, P, P, 2, 10, 8, 100, 16, 4, 2, 64, 0.125, None, 0, None, None]
    bad_heads = list(args)
    bad_heads[15] = 3
    assert f(*bad_heads) == -2
    bad_q = list(args)
    bad_q[2] = None
    assert f(*bad_q) == -1


def test_ops_refuse_cpu_tensors():
    import torch
    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    kp = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16)
    bt = torch.zeros(2, 2, dtype=torch.int32)
    lens = torch.ones(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        pa.attn_decode_paged(q, kp, kp, bt, lens)


def test_multiquery_host_validation(lib):
    f = lib.attn_decode_multiquery_paged
    P = 1 << 20
    # out, lse, q, k, v, num_pages, bt, maxp, cu, lens, batch, total_q, max_q_len, max_seq_len, ps, hq, hkv, d, ...
    args = [P, None, P, P, P, 16, P, 8, P, P, 2, 8, 4, 100, 16, 4, 2, 64, 0.125, None, 0, None, None]
    for bad_q in (0, 9):  # the block must hold 1..8 query rows
        a = list(args)
        a[12] = bad_q
        assert f(*a) == -2
    a = list(args)
    a[8] = None  # cu_seqlens_q
    assert f(*a) == -1
    a = list(args)
    a[15] = 3  # Hq not a multiple of Hkv
    assert f(*a) == -2
    a = list(args)
    a[10], a[2] = 0, None  # empty batch: nothing to do
    assert f(*a) == 0


def test_kv_write_rope_host_validation(lib):
    f = lib.kv_write_paged_rope
    P = 1 << 20
    # k_pool, v_pool, num_pages, k_new, v_new, q, Hq, cu, lens, bt, maxp, batch, total, ps, Hkv, D, base, qw, kw, eps
    args = [P, P, 8, P, P, None, 0, P, P, P, 4, 2, 10, 16, 2, 64, 10000.0, None, None, 1e-6, None, None]
    for i, bad in ((16, 1.0), (16, float("nan")), (16, float("inf")), (19, -1.0), (15, 96)):
        a = list(args)
        a[i] = bad
        assert f(*a) == -2, (i, bad)
    a = list(args)
    a[5], a[6] = P, 3  # q given with Hq not a multiple of Hkv
    assert f(*a) == -2
    a = list(args)
    a[0] = None
    assert f(*a) == -1
    a = list(args)
    a[11] = 0  # empty batch
    assert f(*a) == 0


def test_fp8_host_validation(lib):
    P = 1 << 20
    w = lib.kv_write_paged_fp8
    # k_pool, v_pool, num_pages, k_new, v_new, k_scale, v_scale, cu, lens, bt, maxp, batch, total, ps, Hkv, D
    args = [P, P, 8, P, P, P, P, P, P, P, 4, 2, 10, 16, 2, 64, None, None]
    a = list(args)
    a[15] = 96
    assert w(*a) == -2
    a = list(args)
    a[5] = None  # k_scale
    assert w(*a) == -1
    a = list(args)
    a[11] = 0
    assert w(*a) == 0
    d = lib.attn_decode_paged_fp8
    # out, lse, q, k, v, k_scale, v_scale, num_pages, bt, maxp, lens, batch, max_seq_len, ps, hq, hkv, d, scale, ...
    args = [P, None, P, P, P, P, P, 16, P, 8, P, 2, 100, 16, 4, 2, 64, 0.125, None, 0, None, None]
    a = list(args)
    a[6] = None  # v_scale
    assert d(*a) == -1
    a = list(args)
    a[14] = 3  # Hq not a multiple of Hkv
    assert d(*a) == -2
