import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def oracle_args(case):
    """Numpy views of a workloads.PagedCase for the oracle."""
    return dict(
        q_bits=bits(case.q),
        k_pool_bits=bits(case.k_pool),
        v_pool_bits=bits(case.v_pool),
        block_table=np_i32(case.block_table),
        seq_lens=case.seq_lens_host,
        cu_seqlens_q=np_i32(case.cu_seqlens_q),
        num_q_heads=case.num_q_heads,
        num_kv_heads=case.num_kv_heads,
        page_size=case.page_size,
        scale=case.softmax_scale,
    )


@pytest.fixture(scope="session")
def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


# ---------------------------------------------------------------- parity helpers
# Tolerance of the bf16 outputs against the fp64 oracle: |gpu - ref| <= 2e-2 + 2e-2 |ref|
# element-wise, plus two stricter guards because the absolute bound alone is weak at long
# context (output magnitudes shrink like 1/sqrt(context)): relative L2 error per
# (row, head) <= 1e-2 and |lse error| <= 1e-3.
ATOL = 2e-2
RTOL = 2e-2
REL_L2 = 1e-2
LSE_ATOL = 1e-3


def assert_attention_close(out_gpu, ref_out, lse_gpu=None, ref_lse=None, rows=None, heads=None, what=""):
    """Compare a GPU bf16 output (torch) with the oracle's float64 arrays."""
    o = out_gpu.detach().float().cpu().double().numpy()
    if rows is not None:
        o = o[rows]
        ref_out = ref_out[rows]
    if heads is not None:
        o = o[:, heads]
        ref_out = ref_out[:, heads]
    assert np.isfinite(o).all(), "%s: non-finite GPU output" % what
    err = np.abs(o - ref_out)
    bound = ATOL + RTOL * np.abs(ref_out)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), "%s: max abs err %.3g at %s (ref %.4g, gpu %.4g)" % (
        what, err.max(), worst, ref_out[worst], o[worst])
    num = np.sqrt(((o - ref_out) ** 2).sum(-1))
    den = np.sqrt((ref_out ** 2).sum(-1))
    nz = den > 0
    rel = np.where(nz, num / np.where(nz, den, 1), num)
    assert rel.max() <= REL_L2, "%s: rel-L2 %.3g" % (what, rel.max())
    if lse_gpu is not None:
        l = lse_gpu.detach().cpu().double().numpy()
        rl = ref_lse
        if rows is not None:
            l = l[rows]
            rl = rl[rows]
        if heads is not None:
            l = l[:, heads]
            rl = rl[:, heads]
        fin = np.isfinite(rl)
        assert (np.isfinite(l) == fin).all(), "%s: lse finiteness differs" % what
        assert (l[~fin] == rl[~fin]).all(), "%s: lse of empty rows" % what
        if fin.any():
            assert np.abs(l[fin] - rl[fin]).max() <= LSE_ATOL, "%s: lse err %.3g" % (
                what, np.abs(l[fin] - rl[fin]).max())
    return float(err.max())


def compact_for_oracle(case, seqs):
    """Oracle inputs restricted to sequences `seqs` of a (possibly huge, on-device)
    case: their pages are copied out (each sequence's pages in table order) and
    the block table is renumbered to the compact pool.  Query rows of those
    sequences only; cu_seqlens renumbered.  Returns (args dict, row index list)."""
    ps = case.page_size
    pages, tables, seq_lens, cu, rows = [], [], [], [0], []
    cu_full = case.cu_seqlens_q.cpu().tolist()
    next_page = 0
    maxp = 1
    for b in seqs:
        L = case.seq_lens_host[b]
        n = -(-L // ps)
        phys = case.block_table[b, :n].long()
        pages.append(phys)
        tables.append(list(range(next_page, next_page + n)))
        next_page += n
        maxp = max(maxp, n)
        seq_lens.append(L)
        r0, r1 = cu_full[b], cu_full[b + 1]
        rows.extend(range(r0, r1))
        cu.append(cu[-1] + (r1 - r0))
    idx = torch.cat(pages) if pages else torch.zeros(0, dtype=torch.long, device=case.k_pool.device)
    kp = bits(case.k_pool[idx]) if len(idx) else np.zeros((1,) + tuple(case.k_pool.shape[1:]), np.uint16)
    vp = bits(case.v_pool[idx]) if len(idx) else np.zeros((1,) + tuple(case.v_pool.shape[1:]), np.uint16)
    bt = np.full((len(seqs), maxp), -1, dtype=np.int64)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    row_idx = torch.tensor(rows, dtype=torch.long, device=case.q.device)
    args = dict(q_bits=bits(case.q[row_idx]), k_pool_bits=kp, v_pool_bits=vp, block_table=bt,
                seq_lens=seq_lens, cu_seqlens_q=np.array(cu), num_q_heads=case.num_q_heads,
                num_kv_heads=case.num_kv_heads, page_size=ps, scale=case.softmax_scale)
    return args, rows
