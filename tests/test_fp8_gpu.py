"""FP8 (e4m3) KV cache on the GPU: the quantising writeback bit for bit
against the oracle's codes, and decode over FP8 pages against attention over
the oracle-dequantised pages.  Slots no sequence owns hold the NaN code
0x7F, so a read of them would show in the output."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.conftest import assert_attention_close, bits, compact_for_oracle, np_i32

pytestmark = pytest.mark.gpu


def _pa():
    return pytest.importorskip("paged_kv_decode_17_gb300")


def _scales(hkv, seed, base):
    g = np.random.default_rng(seed)
    return (base * (0.5 + g.random(hkv))).astype(np.float32)


def _fp8_pools(case, ks, vs):
    """Oracle codes of a case's bf16 pools (NaN slots become 0x7F), V transposed per page block."""
    kb, vb = bits(case.k_pool), bits(case.v_pool)
    kc = np.stack([oracle.fp8.quantize(kb[:, g], float(ks[g])) for g in range(kb.shape[1])], axis=1)
    vc = np.stack([oracle.fp8.quantize(vb[:, g], float(vs[g])) for g in range(vb.shape[1])], axis=1)
    return kc, np.ascontiguousarray(np.swapaxes(vc, 2, 3))


def _decode_fp8(case, kc, vc, ks, vs, dev):
    pa = _pa()
    g = case.to(dev)
    status = pa.new_status(dev)
    out, lse = pa.attn_decode_paged_fp8(g.q, torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev),
                                        torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev),
                                        g.block_table, g.seq_lens, g.softmax_scale,
                                        max_seq_len=max(1, case.max_seq_len), return_lse=True, status=status)
    pa.check_status(status, "attn_decode_paged_fp8")
    return out, lse


CASES = [
    # name, seq_lens, Hq, Hkv, D, page_size
    ("tiny_d64", [37, 100], 4, 2, 64, 16),
    ("qwen_like", [900, 1, 17, 3000], 28, 4, 128, 16),
    ("ragged_page64", [5000, 130, 64, 1], 8, 2, 128, 64),
    ("mha_d64", [700, 33], 4, 4, 64, 32),
    ("group16", [1200, 77], 32, 2, 128, 16),
    ("empty_seq", [0, 300], 8, 2, 128, 16),
    ("page256", [2100, 513], 8, 1, 128, 256),
]


@pytest.mark.parametrize("name,seq_lens,hq,hkv,d,ps", CASES, ids=[c[0] for c in CASES])
def test_fp8_decode_matches_oracle(cuda_device, name, seq_lens, hq, hkv, d, ps):
    case = workloads.make_paged_case(name, seq_lens, [1] * len(seq_lens), hq, hkv, d, page_size=ps,
                                     seed=len(name) * 5 + d)
    ks, vs = _scales(hkv, 1, 0.012), _scales(hkv, 2, 0.009)
    kc, vc = _fp8_pools(case, ks, vs)
    ref_out, ref_lse = oracle.paged_attention_fp8(bits(case.q), kc, vc, ks, vs, np_i32(case.block_table),
                                                  case.seq_lens_host, np_i32(case.cu_seqlens_q), hq, hkv, ps,
                                                  case.softmax_scale)
    out, lse = _decode_fp8(case, kc, vc, ks, vs, cuda_device)
    assert_attention_close(out, ref_out, lse, ref_lse, what=name)


def test_fp8_sharp_logits(cuda_device):
    case = workloads.make_paged_case("fp8_sharp", [700, 2000], [1, 1], 16, 2, 128, k_scale=8.0, seed=90)
    ks, vs = _scales(2, 3, 0.09), _scales(2, 4, 0.01)
    kc, vc = _fp8_pools(case, ks, vs)
    ref_out, ref_lse = oracle.paged_attention_fp8(bits(case.q), kc, vc, ks, vs, np_i32(case.block_table),
                                                  case.seq_lens_host, np_i32(case.cu_seqlens_q), 16, 2, 16,
                                                  case.softmax_scale)
    out, lse = _decode_fp8(case, kc, vc, ks, vs, cuda_device)
    assert_attention_close(out, ref_out, lse, ref_lse, what="fp8 sharp")


@pytest.mark.parametrize("d,ps", [(128, 16), (64, 32), (128, 64)])
def test_fp8_writeback_bit_exact(cuda_device, d, ps):
    pa = _pa()
    case = workloads.make_paged_case("fp8_wb", [300, 17, 90], [300, 5, 1], 8, 2, d, page_size=ps,
                                     prewritten=False, seed=91 + d)
    ks, vs = _scales(2, 5, 0.01), _scales(2, 6, 0.02)
    P, Hkv = case.num_pages, 2
    rng = np.random.default_rng(7)
    k0 = rng.integers(0, 256, (P, Hkv, ps, d), dtype=np.uint8)  # arbitrary old contents
    v0 = rng.integers(0, 256, (P, Hkv, d, ps), dtype=np.uint8)
    want_k, want_v = oracle.kv_write_paged_fp8(k0, v0, bits(case.k_new), bits(case.v_new), ks, vs,
                                               np_i32(case.cu_seqlens_q), case.seq_lens_host,
                                               np_i32(case.block_table), ps)
    g = case.to(cuda_device)
    kp, vp = torch.from_numpy(k0).to(cuda_device), torch.from_numpy(v0).to(cuda_device)
    status = pa.new_status(cuda_device)
    pa.kv_write_paged_fp8(kp, vp, g.k_new, g.v_new, torch.from_numpy(ks).to(cuda_device),
                          torch.from_numpy(vs).to(cuda_device), g.cu_seqlens_q, g.seq_lens, g.block_table,
                          status=status)
    pa.check_status(status, "kv_write_paged_fp8")
    assert np.array_equal(kp.cpu().numpy(), want_k), "K codes differ"
    assert np.array_equal(vp.cpu().numpy(), want_v), "V codes differ"


def test_fp8_writeback_then_decode(cuda_device):
    """Serving order on an FP8 cache: quantising writeback of each sequence's
    newest row on the GPU, then decode; the oracle quantises and attends itself."""
    pa = _pa()
    case = workloads.make_paged_case("fp8_e2e", [1000, 64, 3333], [1, 1, 1], 28, 4, 128, prewritten=False,
                                     seed=92)
    ks, vs = _scales(4, 7, 0.011), _scales(4, 8, 0.008)
    kc, vc = _fp8_pools(case, ks, vs)  # the pre-write pages (the new rows' slots hold NaN codes)
    want_k, want_v = oracle.kv_write_paged_fp8(kc, vc, bits(case.k_new), bits(case.v_new), ks, vs,
                                               np_i32(case.cu_seqlens_q), case.seq_lens_host,
                                               np_i32(case.block_table), 16)
    ref_out, ref_lse = oracle.paged_attention_fp8(bits(case.q), want_k, want_v, ks, vs, np_i32(case.block_table),
                                                  case.seq_lens_host, np_i32(case.cu_seqlens_q), 28, 4, 16,
                                                  case.softmax_scale)
    g = case.to(cuda_device)
    kp, vp = torch.from_numpy(kc).to(cuda_device), torch.from_numpy(vc).to(cuda_device)
    kst, vst = torch.from_numpy(ks).to(cuda_device), torch.from_numpy(vs).to(cuda_device)
    pa.kv_write_paged_fp8(kp, vp, g.k_new, g.v_new, kst, vst, g.cu_seqlens_q, g.seq_lens, g.block_table)
    out, lse = pa.attn_decode_paged_fp8(g.q, kp, vp, kst, vst, g.block_table, g.seq_lens, g.softmax_scale,
                                        return_lse=True)
    assert_attention_close(out, ref_out, lse, ref_lse, what="fp8 writeback + decode")


def test_fp8_page_permutation_and_determinism(cuda_device):
    case = workloads.make_paged_case("fp8_perm", [700, 33, 1500], [1, 1, 1], 8, 2, 128, num_pages=160, seed=93)
    ks, vs = _scales(2, 9, 0.01), _scales(2, 10, 0.01)
    kc, vc = _fp8_pools(case, ks, vs)
    o1, l1 = _decode_fp8(case, kc, vc, ks, vs, cuda_device)
    o1b, l1b = _decode_fp8(case, kc, vc, ks, vs, cuda_device)
    assert torch.equal(o1.view(torch.int16), o1b.view(torch.int16)) and torch.equal(l1, l1b)
    perm = np.random.default_rng(4).permutation(case.num_pages)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    c2 = workloads.PagedCase(**{**case.__dict__})
    bt = case.block_table.clone()
    m = bt >= 0
    bt[m] = torch.from_numpy(inv)[bt[m].long()].to(torch.int32)
    c2.block_table = bt
    o2, l2 = _decode_fp8(c2, kc[perm], vc[perm], ks, vs, cuda_device)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


@pytest.mark.slow
def test_fp8_qwen7b_full_size_sampled(cuda_device):
    """The Qwen2.5-7B decode shape (batch 32 x 8192) on an FP8 cache: the whole
    pool quantised by the oracle, three sequences checked against it."""
    case = workloads.qwen7b_decode()
    ks, vs = _scales(4, 11, 0.012), _scales(4, 12, 0.009)
    kc, vc = _fp8_pools(case, ks, vs)
    out, lse = _decode_fp8(case, kc, vc, ks, vs, cuda_device)
    assert torch.isfinite(out.float()).all()
    seqs = [0, 17, 31]
    ref_out, ref_lse = oracle.paged_attention_fp8(bits(case.q), kc, vc, ks, vs, np_i32(case.block_table),
                                                  case.seq_lens_host, np_i32(case.cu_seqlens_q), 28, 4, 16,
                                                  case.softmax_scale, seqs=seqs)
    assert_attention_close(out[seqs], ref_out[seqs], lse[seqs], ref_lse[seqs], what="fp8 qwen7b sampled")


def test_fp8_subnormal_codes(cuda_device):
    """Every K and V code in the e4m3 subnormal range (|code value| < 2^-6), with
    scales large enough that they dominate the result: the exact decode of
    subnormal codes (no flushing to zero) is visible in the output."""
    case = workloads.make_paged_case("fp8_sub", [300, 77], [1, 1], 8, 2, 128, seed=95)
    rng = np.random.default_rng(96)
    P = case.num_pages
    kc = rng.integers(1, 8, (P, 2, 16, 128), dtype=np.uint8) | (rng.integers(0, 2, (P, 2, 16, 128), dtype=np.uint8) << 7)
    vc = rng.integers(1, 8, (P, 2, 128, 16), dtype=np.uint8) | (rng.integers(0, 2, (P, 2, 128, 16), dtype=np.uint8) << 7)
    ks = np.array([64.0, 32.0], dtype=np.float32)  # code 1 -> 2^-9 * 64 = 0.125
    vs = np.array([512.0, 256.0], dtype=np.float32)
    ref_out, ref_lse = oracle.paged_attention_fp8(bits(case.q), kc, vc, ks, vs, np_i32(case.block_table),
                                                  case.seq_lens_host, np_i32(case.cu_seqlens_q), 8, 2, 16,
                                                  case.softmax_scale)
    assert np.abs(ref_out).max() > 0.1  # the subnormal values carry the output
    out, lse = _decode_fp8(case, kc, vc, ks, vs, cuda_device)
    assert_attention_close(out, ref_out, lse, ref_lse, what="fp8 subnormal codes")


@pytest.mark.parametrize("ps", [16, 64])
def test_fp8_bad_page_reports_status(cuda_device, ps):
    """A block-table entry outside the pool is reported (PA_ERR_BAD_PAGE) and its unit
    skipped, both when 16-token pages are staged by bulk copies (the stage's barrier
    phase still completes) and when larger pages are staged per lane; the call ends."""
    pa = _pa()
    case = workloads.make_paged_case("fp8_bad", [900, 300], [1, 1], 8, 2, 128, page_size=ps, seed=97)
    ks, vs = _scales(2, 13, 0.01), _scales(2, 14, 0.01)
    kc, vc = _fp8_pools(case, ks, vs)
    g = case.to(cuda_device)
    g.block_table[0, 2] = 10 ** 6
    g.block_table[1, 0] = -3
    status = pa.new_status(cuda_device)
    pa.attn_decode_paged_fp8(g.q, torch.from_numpy(kc).to(cuda_device), torch.from_numpy(vc).to(cuda_device),
                             torch.from_numpy(ks).to(cuda_device), torch.from_numpy(vs).to(cuda_device),
                             g.block_table, g.seq_lens, g.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
