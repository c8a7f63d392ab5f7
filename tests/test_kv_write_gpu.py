"""kv_write_paged on the GPU against the oracle's scatter: bit-exact, every byte."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.conftest import bits, np_i32

pytestmark = pytest.mark.gpu


def _run_and_compare(case, dev):
    pa = pytest.importorskip("paged_kv_decode_17_gb300")
    kp0, vp0 = bits(case.k_pool), bits(case.v_pool)
    want_k, want_v = oracle.kv_write_paged(kp0, vp0, bits(case.k_new), bits(case.v_new),
                                           np_i32(case.cu_seqlens_q), case.seq_lens_host,
                                           np_i32(case.block_table), case.page_size)
    g = case.to(dev)
    status = pa.new_status(dev)
    pa.kv_write_paged(g.k_pool, g.v_pool, g.k_new, g.v_new, g.cu_seqlens_q, g.seq_lens, g.block_table,
                      status=status)
    pa.check_status(status, "kv_write_paged")
    got_k, got_v = bits(g.k_pool), bits(g.v_pool)
    assert (got_k == want_k).all(), "K pool differs from the oracle scatter"
    assert (got_v == want_v).all(), "V pool differs from the oracle scatter"


@pytest.mark.parametrize("D,Hkv,ps", [(128, 4, 16), (64, 2, 16), (128, 8, 64), (64, 1, 32)])
def test_kv_write_prefill_rows(cuda_device, D, Hkv, ps):
    case = workloads.make_paged_case("wb", [40, 17, 5, 300, 1], [9, 17, 1, 120, 1], 2 * Hkv, Hkv, D, page_size=ps,
                                     prewritten=False, seed=31 + D + ps)
    _run_and_compare(case, cuda_device)


def test_kv_write_decode_step(cuda_device):
    # one new token per sequence, the serving decode step
    case = workloads.make_paged_case("wb_dec", [8192] * 4 + [1, 17], [1] * 6, 28, 4, 128, prewritten=False, seed=32)
    _run_and_compare(case, cuda_device)


def test_kv_write_empty_sequences(cuda_device):
    case = workloads.make_paged_case("wb_empty", [0, 20, 0, 33], [0, 20, 0, 2], 4, 2, 64, prewritten=False,
                                     num_pages=8, seed=33)
    _run_and_compare(case, cuda_device)


@pytest.mark.slow
def test_kv_write_varlen_prefill_full_size(cuda_device):
    # 16 sequences, 512..4096 new tokens each, Hkv=4, D=128
    case = workloads.varlen_prefill(device="cpu")
    _run_and_compare(case, cuda_device)


def test_kv_write_bad_page_reports_status(cuda_device):
    pa = pytest.importorskip("paged_kv_decode_17_gb300")
    case = workloads.make_paged_case("wb_bad", [40, 17], [9, 17], 4, 2, 64, prewritten=False, seed=34, num_pages=5)
    g = case.to(cuda_device)
    bt = g.block_table.clone()
    bt[1, 0] = 1000  # outside the pool
    before_k = bits(g.k_pool)
    status = pa.new_status(cuda_device)
    pa.kv_write_paged(g.k_pool, g.v_pool, g.k_new, g.v_new, g.cu_seqlens_q, g.seq_lens, bt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6  # PA_ERR_BAD_PAGE
    # sequence 0 was still written, the bad rows were skipped
    after_k = bits(g.k_pool)
    assert (after_k != before_k).any()


def test_kv_write_many_sequences(cuda_device):
    # more than 32 sequences (the row -> sequence count spans several 32-entry chunks of cu_seqlens),
    # an odd number of new rows, and rows past the 64 vectors a warp holds (Hkv 8, D 128)
    gen = torch.Generator().manual_seed(35)
    B = 70
    q_lens = torch.randint(0, 7, (B,), generator=gen).tolist()
    seq_lens = [q + int(torch.randint(0, 90, (1,), generator=gen)) for q in q_lens]
    case = workloads.make_paged_case("wb_many", seq_lens, q_lens, 16, 8, 128, prewritten=False, seed=35)
    _run_and_compare(case, cuda_device)
