"""attn_decode_multiquery_paged (1-8 query rows per sequence, causal inside
the block) on the GPU against the fp64 oracle, the same entries inside a
mixed attn_prefill_varlen_causal call, and the bit-exact invariants."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.conftest import assert_attention_close, compact_for_oracle, oracle_args

pytestmark = pytest.mark.gpu


def _pa():
    return pytest.importorskip("paged_kv_decode_17_gb300")


def _mq(case, dev, **kw):
    pa = _pa()
    g = case.to(dev) if case.q.device != dev else case
    status = pa.new_status(dev)
    out, lse = pa.attn_decode_multiquery_paged(g.q, g.k_pool, g.v_pool, g.block_table, g.cu_seqlens_q,
                                               g.seq_lens, g.softmax_scale, max_q_len=max(1, case.max_q_len),
                                               max_seq_len=max(1, case.max_seq_len), return_lse=True,
                                               status=status, **kw)
    pa.check_status(status, "attn_decode_multiquery_paged")
    return out, lse


def _check(case, dev):
    ref_out, ref_lse = oracle.paged_attention(**oracle_args(case))
    out, lse = _mq(case, dev)
    return assert_attention_close(out, ref_out, lse, ref_lse, what=case.name)


CASES = [
    # name, seq_lens, q_lens, Hq, Hkv, D, page_size
    ("q2_g7", [900, 2, 37], [2, 2, 2], 28, 4, 128, 16),        # 14 rows: one row block
    ("q3_g7", [1000, 17, 300], [3, 3, 3], 14, 2, 128, 16),     # 21 rows: two row blocks
    ("q4_g7", [2000, 4, 129, 700], [4, 4, 4, 4], 28, 4, 128, 16),  # 28 rows
    ("q8_g7", [3000, 8, 77], [8, 8, 8], 7, 1, 128, 16),        # 56 rows: four row blocks
    ("q4_g4", [1500, 600], [4, 4], 32, 8, 128, 16),            # 16 rows exactly
    ("q8_mha", [800, 9], [8, 8], 4, 4, 128, 16),               # group 1
    ("q8_g16", [1200, 333], [8, 8], 32, 2, 128, 16),           # 128 rows: two segments
    ("q3_g32", [700, 50], [3, 3], 32, 1, 64, 16),              # 96 rows, D 64
    ("ragged_q", [400, 1, 65, 5000, 3], [1, 1, 5, 8, 3], 16, 2, 128, 16),
    ("q_zero", [300, 90, 120], [2, 0, 6], 8, 2, 128, 16),      # an entry with no query row
    ("page64", [1000, 260], [5, 7], 8, 2, 128, 64),
    ("page256_d64", [2000, 513], [6, 2], 12, 2, 64, 256),
]


@pytest.mark.parametrize("name,seq_lens,q_lens,hq,hkv,d,ps", CASES, ids=[c[0] for c in CASES])
def test_multiquery_matches_oracle(cuda_device, name, seq_lens, q_lens, hq, hkv, d, ps):
    case = workloads.make_paged_case(name, seq_lens, q_lens, hq, hkv, d, page_size=ps, seed=len(name) * 13 + d)
    _check(case, cuda_device)


def test_multiquery_sharp_logits(cuda_device):
    case = workloads.make_paged_case("mq_sharp", [700, 40], [6, 4], 28, 4, 128, k_scale=8.0, seed=70)
    _check(case, cuda_device)


@pytest.mark.parametrize("seed", [71, 72, 73])
def test_multiquery_random(cuda_device, seed):
    gen = torch.Generator().manual_seed(seed)
    B = int(torch.randint(1, 24, (1,), generator=gen))
    q_lens = torch.randint(1, 9, (B,), generator=gen).tolist()
    lens = [q + int(x) for q, x in zip(q_lens, torch.randint(0, 4000, (B,), generator=gen).tolist())]
    Hkv = int(torch.randint(1, 5, (1,), generator=gen))
    group = int(torch.randint(1, 17, (1,), generator=gen))
    D = 64 if seed % 2 else 128
    case = workloads.make_paged_case("mqrand%d" % seed, lens, q_lens, Hkv * group, Hkv, D, seed=seed)
    _check(case, cuda_device)


def test_rows_equal_truncated_decodes(cuda_device):
    """Row i of a q_len block = a one-row decode of the sequence cut to
    seq_len - q_len + i + 1 keys (within the tolerance: the split plans differ)."""
    pa = _pa()
    q_len, L = 5, 3000
    case = workloads.make_paged_case("mq_trunc", [L], [q_len], 16, 2, 128, seed=74).to(cuda_device)
    out, lse = _mq(case, cuda_device)
    for i in range(q_len):
        lens = torch.tensor([L - q_len + i + 1], dtype=torch.int32, device=cuda_device)
        o1, l1 = pa.attn_decode_paged(case.q[i:i + 1].contiguous(), case.k_pool, case.v_pool, case.block_table,
                                      lens, case.softmax_scale, return_lse=True)
        d = (out[i].float() - o1[0].float()).abs()
        assert bool((d <= 2e-2 + 2e-2 * o1[0].float().abs()).all())
        assert float((lse[i] - l1[0]).abs().max()) < 1e-3


def test_future_keys_do_not_matter(cuda_device):
    """Row i is bit-identical when K/V at positions after it change."""
    q_len, L = 6, 1000
    case = workloads.make_paged_case("mq_causal", [L], [q_len], 14, 2, 128, seed=75)
    out1, _ = _mq(case, cuda_device)
    k, v = case.k_pool.clone(), case.v_pool.clone()
    t = L - q_len + 2  # rows 0..2 see keys < t + 1
    for pos in range(t + 1, L):
        phys = int(case.block_table[0, pos // 16])
        k[phys, :, pos % 16] = 3.0
        v[phys, :, pos % 16] = -5.0
    case.k_pool, case.v_pool = k, v
    out2, _ = _mq(case, cuda_device)
    assert torch.equal(out1[:3].view(torch.int16), out2[:3].view(torch.int16))
    assert not torch.equal(out1[3:].view(torch.int16), out2[3:].view(torch.int16))


def test_multiquery_page_permutation_and_determinism(cuda_device):
    case = workloads.make_paged_case("mq_perm", [700, 33, 1500], [4, 2, 8], 28, 4, 128, num_pages=200, seed=76)
    g = case.to(cuda_device)
    o1, l1 = _mq(g, cuda_device)
    o1b, l1b = _mq(g, cuda_device)
    assert torch.equal(o1.view(torch.int16), o1b.view(torch.int16)) and torch.equal(l1, l1b)
    P = case.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    c2 = workloads.PagedCase(**{**case.__dict__})
    c2.k_pool = case.k_pool[perm].contiguous()
    c2.v_pool = case.v_pool[perm].contiguous()
    bt = case.block_table.clone()
    m = bt >= 0
    bt[m] = inv[bt[m].long()].to(torch.int32)
    c2.block_table = bt
    o2, l2 = _mq(c2, cuda_device)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_mixed_call_routes_short_blocks_to_decode(cuda_device):
    """A mixed step with q_len 1, 2..8 and long prefill chunks in one call:
    the short entries give the same bits as the multi-query entry point."""
    pa = _pa()
    case = workloads.make_paged_case("mq_mixed", [900, 300, 2000, 64, 5000], [1, 4, 256, 8, 129], 28, 4, 128,
                                     seed=77)
    ref_out, ref_lse = oracle.paged_attention(**oracle_args(case))
    g = case.to(cuda_device)
    status = pa.new_status(cuda_device)
    out, lse = pa.attn_prefill_varlen_causal(g.q, g.k_pool, g.v_pool, g.block_table, g.cu_seqlens_q, g.seq_lens,
                                             g.softmax_scale, max_q_len=g.max_q_len, max_seq_len=g.max_seq_len,
                                             return_lse=True, status=status)
    pa.check_status(status, "attn_prefill_varlen_causal")
    assert_attention_close(out, ref_out, lse, ref_lse, what="mixed with short blocks")


def test_qlen_above_bound_reports_status(cuda_device):
    pa = _pa()
    case = workloads.make_paged_case("mq_bad", [300, 200], [3, 6], 8, 2, 128, seed=78).to(cuda_device)
    status = pa.new_status(cuda_device)
    pa.attn_decode_multiquery_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.cu_seqlens_q,
                                    case.seq_lens, max_q_len=4, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -7


@pytest.mark.slow
def test_qwen7b_multiquery_full_size_sampled(cuda_device):
    """The Qwen2.5-7B decode shape (batch 32 x 8192, Hq 28, Hkv 4) with 4
    query rows per sequence: three sequences against the oracle on every head."""
    case = workloads.qwen7b_multiquery(device=cuda_device)
    out, lse = _mq(case, cuda_device)
    assert torch.isfinite(out.float()).all()
    seqs = [0, 17, 31]
    args, rows = compact_for_oracle(case, seqs)
    ref_out, ref_lse = oracle.paged_attention(**args)
    assert_attention_close(out[rows], ref_out, lse[rows], ref_lse, what="qwen7b_multiquery sampled")


@pytest.mark.parametrize("lens,qlens,hq,hkv,d,ps", [
    ([900, 2, 37, 18], [2, 2, 3, 3], 28, 4, 128, 16),      # 21 rows: two row blocks; new rows 15-17 span two units
    ([16, 300, 65], [8, 4, 1], 32, 4, 64, 16),             # 64 rows: four row blocks; head_dim 64
    ([40, 1000], [4, 2], 16, 8, 128, 32),                  # group 2 x 4 rows = 8: swapped variant, 32-token pages
])
def test_multiquery_append_matches_writeback_then_decode(cuda_device, lens, qlens, hq, hkv, d, ps):
    """attn_decode_multiquery_paged_append = kv_write_paged (cu_seqlens_new =
    cu_seqlens_q) + attn_decode_multiquery_paged, bit for bit (output, lse and
    the pools), and matches the oracle."""
    pa = _pa()
    dev = cuda_device
    case = workloads.make_paged_case("mq_append", lens, qlens, hq, hkv, d, page_size=ps, seed=93,
                                     prewritten=False, device=dev)
    k2, v2 = case.k_pool.clone(), case.v_pool.clone()
    pa.kv_write_paged(case.k_pool, case.v_pool, case.k_new, case.v_new, case.cu_seqlens_q, case.seq_lens,
                      case.block_table)
    out1, lse1 = _mq(case, dev)
    status = pa.new_status(dev)
    out2, lse2 = pa.attn_decode_multiquery_paged(case.q, k2, v2, case.block_table, case.cu_seqlens_q, case.seq_lens,
                                                 case.softmax_scale, max_q_len=max(qlens),
                                                 max_seq_len=case.max_seq_len, return_lse=True, status=status,
                                                 k_new=case.k_new, v_new=case.v_new)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    assert torch.equal(k2.view(torch.int16), case.k_pool.view(torch.int16))
    assert torch.equal(v2.view(torch.int16), case.v_pool.view(torch.int16))
    ref_out, ref_lse = oracle.paged_attention(**oracle_args(case))
    assert_attention_close(out2, ref_out, lse2, ref_lse, what="mq_append")


@pytest.mark.parametrize("chunk", ["1", "5"])
def test_multiquery_small_chunks(cuda_device, monkeypatch, chunk):
    """Small split-K chunks (PAGEDATTN_DECODE_CHUNK, in 16-key units): many CTA
    ranges per segment, so range boundaries fall between the row blocks of one
    key block (segments of 2 and 4 row blocks), and a ragged call mixes segments
    of 1, 2 and 4 row blocks.  Against the oracle, and bit-identical run to run."""
    monkeypatch.setenv("PAGEDATTN_DECODE_CHUNK", chunk)
    for name, lens, qlens, hq, hkv, d in [("sc_q4_g7", [2000, 4, 129, 700], [4, 4, 4, 4], 28, 4, 128),
                                         ("sc_q8_g7", [3000, 8, 77], [8, 8, 8], 7, 1, 128),
                                         ("sc_ragged", [400, 1, 65, 5000, 3, 999], [1, 1, 5, 8, 3, 2], 16, 2, 128),
                                         ("sc_d64", [700, 50, 333], [3, 3, 7], 32, 2, 64)]:
        case = workloads.make_paged_case(name, lens, qlens, hq, hkv, d, page_size=16, seed=len(name) * 7 + d)
        _check(case, cuda_device)
        a, la = _mq(case, cuda_device)
        b, lb = _mq(case, cuda_device)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)) and torch.equal(la, lb)
