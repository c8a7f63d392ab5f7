"""attn_decode_paged on the GPU against the fp64 oracle, plus the invariants
that must hold bit for bit (page permutation, run-to-run determinism)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.conftest import assert_attention_close, bits, compact_for_oracle, oracle_args

pytestmark = pytest.mark.gpu


def _pa():
    return pytest.importorskip("paged_kv_decode_17_gb300")


def _decode(case, dev, **kw):
    pa = _pa()
    g = case.to(dev) if case.q.device != dev else case
    status = pa.new_status(dev)
    out, lse = pa.attn_decode_paged(g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.softmax_scale,
                                    max_seq_len=max(1, case.max_seq_len), return_lse=True, status=status, **kw)
    pa.check_status(status, "attn_decode_paged")
    return out, lse


def _check(case, dev):
    ref_out, ref_lse = oracle.paged_attention(**oracle_args(case))
    out, lse = _decode(case, dev)
    return assert_attention_close(out, ref_out, lse, ref_lse, what=case.name)


@pytest.mark.parametrize("sharp", [False, True])
def test_tiny_decode(cuda_device, sharp):
    _check(workloads.tiny_decode(seed=0, sharp=sharp), cuda_device)


@pytest.mark.parametrize("name", sorted(workloads.awkward_cases().keys()))
def test_awkward_decode(cuda_device, name):
    _check(workloads.awkward_cases()[name], cuda_device)


@pytest.mark.parametrize("seed", [40, 41, 42])
def test_random_ragged_decode(cuda_device, seed):
    gen = torch.Generator().manual_seed(seed)
    B = int(torch.randint(1, 40, (1,), generator=gen))
    lens = torch.randint(1, 3000, (B,), generator=gen).tolist()
    Hkv = int(torch.randint(1, 5, (1,), generator=gen))
    group = int(torch.randint(1, 9, (1,), generator=gen))
    D = 64 if seed % 2 else 128
    case = workloads.make_paged_case("rand%d" % seed, lens, [1] * B, Hkv * group, Hkv, D, seed=seed)
    _check(case, cuda_device)


def test_page_permutation_bit_exact(cuda_device):
    case = workloads.make_paged_case("perm", [700, 33, 1500], [1, 1, 1], 8, 2, 128, num_pages=160, seed=43)
    out1, lse1 = _decode(case, cuda_device)
    P = case.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    case2 = workloads.PagedCase(**{**case.__dict__})
    case2.k_pool = case.k_pool[perm].contiguous()
    case2.v_pool = case.v_pool[perm].contiguous()
    bt = case.block_table.clone()
    m = bt >= 0
    bt[m] = inv[bt[m].long()].to(torch.int32)
    case2.block_table = bt
    out2, lse2 = _decode(case2, cuda_device)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_run_twice_bit_exact(cuda_device):
    case = workloads.make_paged_case("twice", [5000, 12000, 77], [1, 1, 1], 32, 8, 128, seed=44)
    g = case.to(cuda_device)
    o1, l1 = _decode(g, cuda_device)
    o2, l2 = _decode(g, cuda_device)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_tail_slots_never_read(cuda_device):
    # overwrite every slot past each sequence's end with +inf; outputs must not move
    case = workloads.make_paged_case("tail", [17, 33, 250], [1, 1, 1], 8, 4, 64, num_pages=40, seed=45)
    o1, l1 = _decode(case, cuda_device)
    k = case.k_pool.clone()
    v = case.v_pool.clone()
    for b, L in enumerate(case.seq_lens_host):
        last = int(case.block_table[b, (L - 1) // 16])
        k[last, :, L % 16 or 16:, :] = float("inf")
        v[last, :, L % 16 or 16:, :] = float("inf")
    case.k_pool, case.v_pool = k, v
    o2, l2 = _decode(case, cuda_device)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_bad_page_reports_status(cuda_device):
    pa = _pa()
    case = workloads.make_paged_case("bad", [100, 60], [1, 1], 4, 2, 64, seed=46, num_pages=12)
    g = case.to(cuda_device)
    g.block_table[1, 2] = -5
    status = pa.new_status(cuda_device)
    pa.attn_decode_paged(g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    # the workspace needs no reset after a device error: the next call runs clean
    _check(case, cuda_device)


def test_seq_len_beyond_table_reports_status(cuda_device):
    pa = _pa()
    case = workloads.make_paged_case("badlen", [30, 20], [1, 1], 4, 2, 64, seed=47)
    g = case.to(cuda_device)
    g.seq_lens[0] = 10 ** 6
    status = pa.new_status(cuda_device)
    pa.attn_decode_paged(g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, max_seq_len=32, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -7


def test_host_validation_errors(cuda_device):
    pa = _pa()
    case = workloads.tiny_decode().to(cuda_device)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.attn_decode_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                             workspace=pa.Workspace(256, cuda_device))
    assert e.value.code == -3  # workspace too small
    q3 = case.q[:, :3].contiguous()  # 3 query heads over 2 KV heads
    with pytest.raises(pa.PagedAttnError) as e:
        pa.attn_decode_paged(q3, case.k_pool, case.v_pool, case.block_table, case.seq_lens)
    assert e.value.code == -2


def _sampled_full_size(case, seqs, dev):
    out, lse = _decode(case, dev)
    args, rows = compact_for_oracle(case, seqs)
    ref_out, ref_lse = oracle.paged_attention(**args)
    assert_attention_close(out[rows], ref_out, lse[rows], ref_lse, what=case.name + " sampled")
    # no NaN anywhere in the full output
    assert torch.isfinite(out.float()).all()
    return out


@pytest.mark.slow
def test_qwen7b_decode_full_size_sampled(cuda_device):
    case = workloads.qwen7b_decode(device=cuda_device)
    _sampled_full_size(case, [0, 13, 31], cuda_device)


@pytest.mark.slow
def test_llama8b_ragged_decode_full_size_sampled(cuda_device):
    case = workloads.llama8b_ragged_decode(device=cuda_device)
    lens = case.seq_lens_host
    order = sorted(range(len(lens)), key=lambda b: lens[b])
    seqs = [order[0], order[len(order) // 2], order[-1]]  # shortest, median, longest
    _sampled_full_size(case, seqs, cuda_device)


def test_pinned_host_arguments_match_device(cuda_device):
    """q, out, lse, the new K/V rows, seq_lens and cu_seqlens in pinned host
    memory (read and written in place by the kernels) give the same bits as
    device copies: writeback, decode and multi-query decode."""
    pa = _pa()
    dev = cuda_device
    case = workloads.make_paged_case("pinned", [700, 33, 4096, 1], [1, 1, 1, 1], 28, 4, 128, seed=81,
                                     prewritten=False, device=dev)
    pools = (case.k_pool.clone(), case.v_pool.clone())
    ones = torch.arange(case.batch + 1, dtype=torch.int32, device=dev)
    # device path
    pa.kv_write_paged(case.k_pool, case.v_pool, case.k_new, case.v_new, ones, case.seq_lens, case.block_table)
    out_d, lse_d = pa.attn_decode_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                        case.softmax_scale, max_seq_len=case.max_seq_len, return_lse=True)
    # pinned host path on fresh pools
    k2, v2 = pools
    h = {n: getattr(case, n).cpu().pin_memory() for n in ("q", "k_new", "v_new", "seq_lens")}
    h_ones = ones.cpu().pin_memory()
    out_h = torch.full(case.q.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.full((case.batch, case.num_q_heads), float("nan"), dtype=torch.float32).pin_memory()
    status = pa.new_status(dev)
    pa.kv_write_paged(k2, v2, h["k_new"], h["v_new"], h_ones, h["seq_lens"], case.block_table, status=status)
    pa.attn_decode_paged(h["q"], k2, v2, case.block_table, h["seq_lens"], case.softmax_scale,
                         max_seq_len=case.max_seq_len, out=out_h, lse=lse_h, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(k2.view(torch.int16), case.k_pool.view(torch.int16))
    assert torch.equal(v2.view(torch.int16), case.v_pool.view(torch.int16))
    assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16))
    assert torch.equal(lse_h, lse_d.cpu())
    # multi-query decode (2 rows per sequence) with host q / out / cu_seqlens_q / seq_lens
    mq = workloads.make_paged_case("pinned_mq", [300, 64, 2000], [2, 2, 2], 28, 4, 128, seed=82, device=dev)
    ref = pa.attn_decode_multiquery_paged(mq.q, mq.k_pool, mq.v_pool, mq.block_table, mq.cu_seqlens_q, mq.seq_lens,
                                          mq.softmax_scale, max_q_len=2, max_seq_len=mq.max_seq_len)
    hq = mq.q.cpu().pin_memory()
    hout = torch.empty(mq.q.shape, dtype=torch.bfloat16).pin_memory()
    pa.attn_decode_multiquery_paged(hq, mq.k_pool, mq.v_pool, mq.block_table, mq.cu_seqlens_q.cpu().pin_memory(),
                                    mq.seq_lens.cpu().pin_memory(), mq.softmax_scale, max_q_len=2,
                                    max_seq_len=mq.max_seq_len, out=hout)
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("lens,hq,hkv,d,ps", [
    ([1, 16, 17, 31, 32, 500], 28, 4, 128, 16),   # group 7: swapped variant; page-boundary positions
    ([1, 64, 65, 1000], 16, 2, 64, 64),           # group 8, head_dim 64, 64-token pages
    ([5, 300, 4097], 32, 2, 128, 16),             # group 16: unswapped
    ([3, 129, 2048], 64, 2, 128, 32),             # group 32: two row blocks, one writer per key block
])
def test_append_matches_writeback_then_decode(cuda_device, lens, hq, hkv, d, ps):
    """attn_decode_paged_append = kv_write_paged + attn_decode_paged, bit for
    bit (output, lse and the pools), and matches the oracle."""
    pa = _pa()
    dev = cuda_device
    case = workloads.make_paged_case("append", lens, [1] * len(lens), hq, hkv, d, page_size=ps, seed=91,
                                     prewritten=False, device=dev)
    k2, v2 = case.k_pool.clone(), case.v_pool.clone()
    ones = torch.arange(case.batch + 1, dtype=torch.int32, device=dev)
    pa.kv_write_paged(case.k_pool, case.v_pool, case.k_new, case.v_new, ones, case.seq_lens, case.block_table)
    out1, lse1 = pa.attn_decode_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                      case.softmax_scale, max_seq_len=case.max_seq_len, return_lse=True)
    status = pa.new_status(dev)
    out2, lse2 = pa.attn_decode_paged(case.q, k2, v2, case.block_table, case.seq_lens, case.softmax_scale,
                                      max_seq_len=case.max_seq_len, return_lse=True, status=status,
                                      k_new=case.k_new, v_new=case.v_new)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    assert torch.equal(k2.view(torch.int16), case.k_pool.view(torch.int16))
    assert torch.equal(v2.view(torch.int16), case.v_pool.view(torch.int16))
    ref_out, ref_lse = oracle.paged_attention(**oracle_args(case))
    assert_attention_close(out2, ref_out, lse2, ref_lse, what="append")


def test_append_with_pinned_host_rows(cuda_device):
    """The appended rows (and q / out) may be pinned host tensors."""
    pa = _pa()
    dev = cuda_device
    case = workloads.make_paged_case("append_host", [40, 7, 900], [1, 1, 1], 28, 4, 128, seed=92,
                                     prewritten=False, device=dev)
    k2, v2 = case.k_pool.clone(), case.v_pool.clone()
    ref = pa.attn_decode_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                               case.softmax_scale, max_seq_len=case.max_seq_len, k_new=case.k_new, v_new=case.v_new)
    hout = torch.empty(case.q.shape, dtype=torch.bfloat16).pin_memory()
    pa.attn_decode_paged(case.q.cpu().pin_memory(), k2, v2, case.block_table, case.seq_lens, case.softmax_scale,
                         max_seq_len=case.max_seq_len, out=hout, k_new=case.k_new.cpu().pin_memory(),
                         v_new=case.v_new.cpu().pin_memory())
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(k2.view(torch.int16), case.k_pool.view(torch.int16))


@pytest.mark.parametrize("chunk", ["1", "3"])
def test_forced_small_chunks(cuda_device, monkeypatch, chunk):
    """PAGEDATTN_DECODE_CHUNK shrinks the split-K chunks (in 16-key units), so even
    tiny problems are split across many CTAs and merged; the result stays within
    tolerance and run-to-run bit-identical."""
    monkeypatch.setenv("PAGEDATTN_DECODE_CHUNK", chunk)
    for case in (workloads.tiny_decode(seed=1), workloads.tiny_decode(seed=2, sharp=True),
                 workloads.make_paged_case("chunks", [1, 700, 33, 2049], [1] * 4, 28, 4, 128, seed=44)):
        _check(case, cuda_device)
        a, la = _decode(case, cuda_device)
        b, lb = _decode(case, cuda_device)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)) and torch.equal(la, lb)


def test_config_log_once_per_configuration(cuda_device, tmp_path):
    """PAGEDATTN_LOG prints the chosen launch configuration once per distinct
    configuration (a child process, so the environment is read fresh)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import torch, workloads, paged_kv_decode_17_gb300 as pa\n"
        "dev = torch.device('cuda:0')\n"
        "c = workloads.tiny_decode(seed=0).to(dev)\n"
        "for _ in range(3):\n"
        "    pa.attn_decode_paged(c.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, c.softmax_scale, max_seq_len=100)\n"
        "m = workloads.make_paged_case('log', [300, 1], [200, 1], 8, 2, 128, seed=1).to(dev)\n"
        "pa.attn_prefill_varlen_causal(m.q, m.k_pool, m.v_pool, m.block_table, m.cu_seqlens_q, m.seq_lens)\n"
        "torch.cuda.synchronize()\n" % root)
    env = dict(os.environ, PAGEDATTN_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stderr.splitlines() if l.startswith("[pagedattn]")]
    dec = [l for l in lines if "split-K decode" in l]
    assert len([l for l in dec if "head_dim 64" in l]) == 1, lines  # three identical calls, one line
    assert any("per segment" in l for l in dec), lines  # the prefill call's one-row entries
    assert any("mixed step in one launch" in l for l in lines), lines  # the default path of that call
    env["PAGEDATTN_LOG"] = "0"
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "[pagedattn]" not in r.stderr
