"""kv_write_paged_rope on the GPU against the fp64 oracle: K rows normalised
and rotated within one bf16 ulp, V rows and every untouched byte bit-exact,
queries rotated in place, and attention over the rotated cache."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.conftest import assert_attention_close, bits, np_i32, oracle_args

pytestmark = pytest.mark.gpu


def _pa():
    return pytest.importorskip("paged_kv_decode_17_gb300")


def _bf16_bits_of(x64):
    """bf16 bit patterns of float64 values, rounded to nearest even."""
    f = oracle.round_to_bf16_f64(x64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _assert_within_ulp(gpu_bits, ref, what, min_exact=0.99):
    g = oracle.bf16_bits_to_f64(gpu_bits)
    err = np.abs(g - ref)
    bound = oracle.bf16_ulp(ref) + 1e-6 * np.sqrt(np.mean(ref * ref))
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), "%s: err %.3g at %s (ref %.6g gpu %.6g)" % (what, err[worst], worst, ref[worst],
                                                                             g[worst])
    exact = np.mean(gpu_bits == _bf16_bits_of(ref))
    assert exact >= min_exact, "%s: only %.4f of the elements round like the oracle" % (what, exact)


def _weights(D, seed):
    g = torch.Generator().manual_seed(seed)
    return (0.5 + torch.rand(D, generator=g)).to(torch.bfloat16)


CASES = [
    # name, seq_lens, n_new, Hq, Hkv, D, page_size, base, norm, with_q
    ("decode_rows", [37, 100, 5000], [1, 1, 1], 8, 2, 128, 16, 10000.0, False, True),
    ("prefill_rows", [300, 77], [300, 20], 4, 2, 128, 16, 1e6, True, True),
    ("d64_page32", [129, 64], [64, 1], 6, 3, 64, 32, 500000.0, True, False),
    ("k_only_norm", [50, 17], [9, 17], 8, 1, 128, 16, 10000.0, True, False),
    ("long_positions", [131072, 70000], [2, 3], 4, 2, 128, 64, 10000.0, False, True),
]


@pytest.mark.parametrize("name,seq_lens,n_new,hq,hkv,d,ps,base,norm,with_q", CASES, ids=[c[0] for c in CASES])
def test_rope_writeback_matches_oracle(cuda_device, name, seq_lens, n_new, hq, hkv, d, ps, base, norm, with_q):
    pa = _pa()
    case = workloads.make_paged_case(name, seq_lens, n_new, hq, hkv, d, page_size=ps, prewritten=False,
                                     seed=len(name) * 3 + d)
    kw = _weights(d, 1) if norm else None
    qw = _weights(d, 2) if (norm and with_q) else None
    k0, v0, q0 = bits(case.k_pool), bits(case.v_pool), bits(case.q)
    cu, lens = np_i32(case.cu_seqlens_q), case.seq_lens_host
    # oracle: rotated rows, and where every row goes (the pinned scatter)
    k_ref, q_ref, pos = oracle.rope_writeback_rows(bits(case.k_new), q0 if with_q else None, cu, lens, base,
                                                   None if kw is None else bits(kw),
                                                   None if qw is None else bits(qw), eps=1e-6)
    marker_k = np.zeros_like(bits(case.k_new))
    kp_ref, vp_ref = oracle.kv_write_paged(k0, v0, marker_k, bits(case.v_new), cu, lens,
                                           np_i32(case.block_table), ps)
    g = case.to(cuda_device)
    status = pa.new_status(cuda_device)
    pa.kv_write_paged_rope(g.k_pool, g.v_pool, g.k_new, g.v_new, g.cu_seqlens_q, g.seq_lens, g.block_table, base,
                           q=g.q if with_q else None, q_norm_weight=None if qw is None else qw.to(cuda_device),
                           k_norm_weight=None if kw is None else kw.to(cuda_device), norm_eps=1e-6, status=status)
    pa.check_status(status, "kv_write_paged_rope")
    kp, vp = bits(g.k_pool), bits(g.v_pool)
    assert np.array_equal(vp, vp_ref), "V pool differs"
    # K: written slots within one ulp, all other bytes untouched
    written = np.zeros(kp.shape[:1] + kp.shape[2:3], dtype=bool)  # [page][slot]
    rows = []
    bt = np_i32(case.block_table)
    for t in range(len(pos)):
        b = int(np.searchsorted(cu, t, side="right") - 1)
        phys, slot = int(bt[b][pos[t] // ps]), int(pos[t] % ps)
        written[phys, slot] = True
        rows.append(kp[phys, :, slot, :])
    untouched = ~written[:, None, :, None].repeat(kp.shape[1], 1).repeat(kp.shape[3], 3)
    assert np.array_equal(kp[untouched], k0[untouched]), "K bytes outside the written slots changed"
    _assert_within_ulp(np.stack(rows), k_ref, "K rows")
    if with_q:
        _assert_within_ulp(bits(g.q), q_ref, "q rows")
    else:
        assert np.array_equal(bits(g.q), q0)


def test_attention_over_rotated_cache(cuda_device):
    """Serving order with RoPE: fused writeback of the chunk's rows (rotating
    K and the queries), then prefill over the pages.  The oracle rotates and
    rounds the same rows itself and attends over them."""
    pa = _pa()
    base = 1e6
    case = workloads.make_paged_case("rope_attn", [700, 2000, 64], [200, 1, 64], 16, 2, 128, prewritten=False,
                                     seed=81)
    kw, qw = _weights(128, 3), _weights(128, 4)
    cu, lens, ps = np_i32(case.cu_seqlens_q), case.seq_lens_host, case.page_size
    k_ref, q_ref, _ = oracle.rope_writeback_rows(bits(case.k_new), bits(case.q), cu, lens, base, bits(kw),
                                                 bits(qw), eps=1e-6)
    kp, vp = oracle.kv_write_paged(bits(case.k_pool), bits(case.v_pool), _bf16_bits_of(k_ref), bits(case.v_new),
                                   cu, lens, np_i32(case.block_table), ps)
    args = oracle_args(case)
    args.update(q_bits=_bf16_bits_of(q_ref), k_pool_bits=kp, v_pool_bits=vp)
    ref_out, ref_lse = oracle.paged_attention(**args)
    g = case.to(cuda_device)
    pa.kv_write_paged_rope(g.k_pool, g.v_pool, g.k_new, g.v_new, g.cu_seqlens_q, g.seq_lens, g.block_table, base,
                           q=g.q, q_norm_weight=qw.to(cuda_device), k_norm_weight=kw.to(cuda_device))
    out, lse = pa.attn_prefill_varlen_causal(g.q, g.k_pool, g.v_pool, g.block_table, g.cu_seqlens_q, g.seq_lens,
                                             g.softmax_scale, return_lse=True)
    assert_attention_close(out, ref_out, lse, ref_lse, what="attention over rotated cache")


def test_rope_writeback_bad_page_reports_status(cuda_device):
    pa = _pa()
    case = workloads.make_paged_case("rope_bad", [40], [40], 4, 2, 128, prewritten=False, seed=82).to(cuda_device)
    case.block_table[0, 1] = -5
    status = pa.new_status(cuda_device)
    pa.kv_write_paged_rope(case.k_pool, case.v_pool, case.k_new, case.v_new, case.cu_seqlens_q, case.seq_lens,
                           case.block_table, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
