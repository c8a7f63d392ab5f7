"""attn_prefill_varlen_causal (and writeback + prefill) on the GPU against the
fp64 oracle, including mixed prefill + decode entries and the bit-exact
invariants."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.conftest import assert_attention_close, bits, compact_for_oracle, np_i32, oracle_args

pytestmark = pytest.mark.gpu


def _pa():
    return pytest.importorskip("paged_kv_decode_17_gb300")


def _prefill(g, dev, **kw):
    pa = _pa()
    status = pa.new_status(dev)
    out, lse = pa.attn_prefill_varlen_causal(g.q, g.k_pool, g.v_pool, g.block_table, g.cu_seqlens_q, g.seq_lens,
                                             g.softmax_scale, max_q_len=max(1, g.max_q_len),
                                             max_seq_len=max(1, g.max_seq_len), return_lse=True, status=status, **kw)
    pa.check_status(status, "attn_prefill_varlen_causal")
    return out, lse


def _check(case, dev):
    ref_out, ref_lse = oracle.paged_attention(**oracle_args(case))
    out, lse = _prefill(case.to(dev), dev)
    return assert_attention_close(out, ref_out, lse, ref_lse, what=case.name)


CASES = [
    # name, seq_lens, q_lens, Hq, Hkv, D, page_size
    ("single_37", [37], [37], 2, 1, 128, 16),
    ("tile_exact", [128, 64], [128, 64], 4, 2, 128, 16),
    ("tile_plus1", [129, 65, 200], [129, 65, 200], 8, 2, 128, 16),
    ("ragged_many", [300, 17, 513, 2], [300, 17, 513, 2], 28, 4, 128, 16),
    ("prior_chunk", [1000, 700], [200, 129], 8, 2, 128, 16),
    ("prior_small_q", [333, 90], [5, 3], 8, 4, 128, 16),
    ("odd_group", [150, 260], [150, 100], 6, 2, 128, 16),
    ("mha", [190], [190], 4, 4, 128, 16),
    ("d64", [400, 129], [400, 60], 8, 2, 64, 16),
    ("page32", [500, 77], [300, 77], 8, 2, 128, 32),
    ("page64", [260, 1000], [260, 500], 4, 1, 128, 64),
    # the boundary between the two paths: 8 rows (split-K decode) next to 9 rows (prefill tiles),
    # with and without cached tokens before them
    ("q8_q9_boundary", [9, 500, 8, 300, 17], [9, 9, 8, 8, 17], 8, 2, 128, 16),
    # several 16-key blocks per page (one TMA box per block)
    ("page128", [700, 300], [700, 130], 8, 2, 128, 128),
    ("page256", [1100, 513], [600, 513], 4, 2, 128, 256),
    ("mixed_decode_rows", [900, 1, 77, 3000, 256], [256, 1, 1, 1, 256], 32, 8, 128, 16),
    # one-row entries (swapped operand order: group x 1 <= 8 rows) next to 2-8-row blocks (plain
    # order) and a prefill chunk in the same call
    ("mixed_orders_g4", [2000, 1, 600, 77, 1500, 9], [1, 1, 3, 8, 300, 1], 16, 4, 128, 16),
    ("mixed_orders_g8", [40, 5000, 333, 700], [1, 5, 1, 150], 16, 2, 128, 16),
    ("mixed_orders_d64", [1200, 64, 900], [1, 2, 129], 8, 2, 64, 16),
]


PATHS = ["fused", "separate"]  # one persistent launch for decode rows + prefill tiles, or separate kernels


def _set_path(monkeypatch, path):
    """fused / separate (stand-alone prefill, single CTAs by default) / pairs (stand-alone
    prefill as CTA pairs, head_dim 128) / singles (stand-alone prefill, single CTAs)."""
    monkeypatch.setenv("PAGEDATTN_PREFILL_PATH", "fused" if path == "fused" else "separate")
    if path == "pairs":
        monkeypatch.setenv("PAGEDATTN_PREFILL_PAIR", "1")
    elif path == "singles":
        monkeypatch.setenv("PAGEDATTN_PREFILL_PAIR", "0")
    else:
        monkeypatch.delenv("PAGEDATTN_PREFILL_PAIR", raising=False)


@pytest.mark.parametrize("path", PATHS + ["pairs", "singles"])
@pytest.mark.parametrize("name,seq_lens,q_lens,hq,hkv,d,ps", CASES, ids=[c[0] for c in CASES])
def test_prefill_matches_oracle(cuda_device, monkeypatch, path, name, seq_lens, q_lens, hq, hkv, d, ps):
    _set_path(monkeypatch, path)
    case = workloads.make_paged_case(name, seq_lens, q_lens, hq, hkv, d, page_size=ps, seed=len(name) * 7 + d)
    _check(case, cuda_device)


@pytest.mark.parametrize("name,seq_lens,q_lens,hq,hkv,d,ps", [c for c in CASES if c[5] == 128],
                         ids=[c[0] for c in CASES if c[5] == 128])
def test_pairs_and_singles_bit_identical(cuda_device, monkeypatch, name, seq_lens, q_lens, hq, hkv, d, ps):
    """A CTA pair computes each tile's S = Q K^T and O += P V as one M = 256 MMA over two
    SMs, but every row sees the same keys in the same order and the same softmax: the
    prefill rows come out bit-identical to single CTAs'."""
    case = workloads.make_paged_case(name, seq_lens, q_lens, hq, hkv, d, page_size=ps, seed=len(name) * 7 + d)
    g = case.to(cuda_device)
    res = {}
    for path in ("pairs", "singles"):
        _set_path(monkeypatch, path)
        res[path] = _prefill(g, cuda_device)
    cu = case.cu_seqlens_q.tolist()
    rows = [r for b, q in enumerate(case.q_lens_host) if q > 8 for r in range(cu[b], cu[b + 1])]
    if rows:
        ri = torch.tensor(rows, device=cuda_device)
        (op, lp), (os_, ls) = res["pairs"], res["singles"]
        assert torch.equal(op[ri].view(torch.int16), os_[ri].view(torch.int16))
        assert torch.equal(lp[ri], ls[ri])


@pytest.mark.parametrize("name,seq_lens,q_lens,hq,hkv,d,ps", [CASES[3], CASES[-3], CASES[-1]],
                         ids=["ragged_many", "mixed_orders_g4", "mixed_orders_d64"])
def test_fused_and_separate_paths_agree(cuda_device, monkeypatch, name, seq_lens, q_lens, hq, hkv, d, ps):
    """Prefill rows are computed item by item the same way on both paths (bit-identical);
    decode rows may be split differently (same result within rounding)."""
    case = workloads.make_paged_case(name, seq_lens, q_lens, hq, hkv, d, page_size=ps, seed=len(name) * 7 + d)
    g = case.to(cuda_device)
    res = {}
    for path in PATHS:
        monkeypatch.setenv("PAGEDATTN_PREFILL_PATH", path)
        res[path] = _prefill(g, cuda_device)
    cu = case.cu_seqlens_q.tolist()
    long_rows = [r for b, q in enumerate(case.q_lens_host) if q > 8 for r in range(cu[b], cu[b + 1])]
    short_rows = [r for b, q in enumerate(case.q_lens_host) if q <= 8 for r in range(cu[b], cu[b + 1])]
    (of, lf), (os_, ls) = res["fused"], res["separate"]
    if long_rows:
        lr = torch.tensor(long_rows, device=cuda_device)
        assert torch.equal(of[lr].view(torch.int16), os_[lr].view(torch.int16))
        assert torch.equal(lf[lr], ls[lr])
    if short_rows:
        sr = torch.tensor(short_rows, device=cuda_device)
        d_ = (of[sr].float() - os_[sr].float()).abs()
        assert bool((d_ <= 2e-2 + 2e-2 * os_[sr].float().abs()).all())
        assert float((lf[sr] - ls[sr]).abs().max()) < 1e-3


def test_fused_path_repeated_calls_bit_identical(cuda_device):
    """The plan flag and item counter of the fused launch are tagged per launch and
    reset after it: back-to-back calls (different inputs in between) stay exact."""
    a = workloads.make_paged_case("rep_a", [900, 1, 3000, 400], [300, 1, 1, 400], 16, 4, 128, seed=70).to(cuda_device)
    b = workloads.make_paged_case("rep_b", [2000, 77], [1000, 1], 16, 4, 128, seed=71).to(cuda_device)
    oa1, la1 = _prefill(a, cuda_device)
    ob1, lb1 = _prefill(b, cuda_device)
    oa2, la2 = _prefill(a, cuda_device)
    ob2, lb2 = _prefill(b, cuda_device)
    assert torch.equal(oa1.view(torch.int16), oa2.view(torch.int16)) and torch.equal(la1, la2)
    assert torch.equal(ob1.view(torch.int16), ob2.view(torch.int16)) and torch.equal(lb1, lb2)


def test_fused_path_back_to_back_calls_share_a_workspace(cuda_device):
    """32 mixed calls queued back to back on one stream (each launch may start while
    the previous one's merge runs) with one workspace and one status word: the
    status stays clean and the last result equals a lone call's."""
    pa = _pa()
    c = workloads.make_paged_case("b2b", [1500, 1, 3000, 64, 700], [400, 1, 1, 64, 129], 32, 8, 128,
                                  seed=72).to(cuda_device)
    ws = pa.Workspace(pa.prefill_workspace_bytes(c.batch, c.total_q, c.num_q_heads, c.num_kv_heads, c.head_dim),
                      cuda_device)
    status = pa.new_status(cuda_device)
    out = torch.empty_like(c.q)

    def call():
        pa.attn_prefill_varlen_causal(c.q, c.k_pool, c.v_pool, c.block_table, c.cu_seqlens_q, c.seq_lens,
                                      c.softmax_scale, max_q_len=c.max_q_len, max_seq_len=c.max_seq_len, out=out,
                                      workspace=ws, status=status)

    call()
    torch.cuda.synchronize()
    want = out.clone()
    for _ in range(32):
        call()
    torch.cuda.synchronize()
    pa.check_status(status, "back-to-back mixed calls")
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))


def test_prefill_sharp_logits(cuda_device):
    case = workloads.make_paged_case("sharp", [700, 300], [700, 150], 8, 2, 128, k_scale=8.0, seed=60)
    _check(case, cuda_device)


def test_writeback_then_prefill(cuda_device):
    """The serving order: write the new rows into their pages, then attend."""
    pa = _pa()
    case = workloads.make_paged_case("wb_prefill", [600, 333, 90], [200, 333, 90], 8, 2, 128, prewritten=False,
                                     seed=61)
    kp, vp = oracle.kv_write_paged(bits(case.k_pool), bits(case.v_pool), bits(case.k_new), bits(case.v_new),
                                   np_i32(case.cu_seqlens_q), case.seq_lens_host, np_i32(case.block_table),
                                   case.page_size)
    args = oracle_args(case)
    args["k_pool_bits"], args["v_pool_bits"] = kp, vp
    ref_out, ref_lse = oracle.paged_attention(**args)
    g = case.to(cuda_device)
    pa.kv_write_paged(g.k_pool, g.v_pool, g.k_new, g.v_new, g.cu_seqlens_q, g.seq_lens, g.block_table)
    out, lse = _prefill(g, cuda_device)
    assert_attention_close(out, ref_out, lse, ref_lse, what="writeback+prefill")


def test_decode_rows_equal_decode_entry_point(cuda_device):
    """q_len = 1 entries of the prefill call give the same rows as attn_decode_paged."""
    pa = _pa()
    case = workloads.make_paged_case("dec_eq", [5000, 1, 333, 70], [1, 1, 1, 1], 16, 2, 128, seed=62).to(cuda_device)
    out_p, lse_p = _prefill(case, cuda_device)
    out_d, lse_d = pa.attn_decode_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                        case.softmax_scale, return_lse=True)
    d = (out_p.float() - out_d.float()).abs()
    assert bool((d <= 2e-2 + 2e-2 * out_d.float().abs()).all())
    assert float((lse_p - lse_d).abs().max()) < 1e-3


def test_causal_future_keys_do_not_matter(cuda_device):
    """Rows at positions < t are bit-identical when K/V at positions >= t change."""
    case = workloads.make_paged_case("causal", [400], [400], 4, 2, 128, seed=63)
    out1, _ = _prefill(case.to(cuda_device), cuda_device)
    t = 250
    k, v = case.k_pool.clone(), case.v_pool.clone()
    for pos in range(t, 400):
        phys = int(case.block_table[0, pos // 16])
        k[phys, :, pos % 16] = 3.0
        v[phys, :, pos % 16] = -5.0
    case.k_pool, case.v_pool = k, v
    out2, _ = _prefill(case.to(cuda_device), cuda_device)
    assert torch.equal(out1[:t].view(torch.int16), out2[:t].view(torch.int16))
    assert not torch.equal(out1[t:].view(torch.int16), out2[t:].view(torch.int16))


def test_prefill_page_permutation_and_determinism(cuda_device):
    case = workloads.make_paged_case("perm", [520, 130], [520, 60], 8, 2, 128, num_pages=60, seed=64)
    g = case.to(cuda_device)
    o1, l1 = _prefill(g, cuda_device)
    o1b, l1b = _prefill(g, cuda_device)
    assert torch.equal(o1.view(torch.int16), o1b.view(torch.int16)) and torch.equal(l1, l1b)
    P = case.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    c2 = workloads.PagedCase(**{**case.__dict__})
    c2.k_pool = case.k_pool[perm].contiguous()
    c2.v_pool = case.v_pool[perm].contiguous()
    bt = case.block_table.clone()
    m = bt >= 0
    bt[m] = inv[bt[m].long()].to(torch.int32)
    c2.block_table = bt
    o2, l2 = _prefill(c2.to(cuda_device), cuda_device)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_prefill_bad_page_reports_status(cuda_device):
    pa = _pa()
    case = workloads.make_paged_case("bad", [300], [300], 4, 2, 128, seed=65).to(cuda_device)
    case.block_table[0, 3] = 10 ** 6
    status = pa.new_status(cuda_device)
    pa.attn_prefill_varlen_causal(case.q, case.k_pool, case.v_pool, case.block_table, case.cu_seqlens_q,
                                  case.seq_lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6


@pytest.mark.parametrize("path", ["fused", "pairs", "singles"])
def test_wait_timeout_reports_status_and_context_survives(cuda_device, monkeypatch, path):
    """With the prefill's wait limit cut to 1 ns (PAGEDATTN_PREFILL_WAIT_NS), waits
    run out: the call returns, the status word holds PA_ERR_TIMEOUT (-5), every
    CTA drains its copies and tensor-core work and exits, and the next call with
    the normal limit is clean and correct."""
    import time
    pa = _pa()
    case = workloads.make_paged_case("timeout", [3000, 2000, 1000, 600], [3000, 2000, 1000, 300], 8, 2, 128, seed=66)
    g = case.to(cuda_device)
    _set_path(monkeypatch, path)
    monkeypatch.setenv("PAGEDATTN_PREFILL_WAIT_NS", "1")
    status = pa.new_status(cuda_device)
    t0 = time.time()
    pa.attn_prefill_varlen_causal(g.q, g.k_pool, g.v_pool, g.block_table, g.cu_seqlens_q, g.seq_lens,
                                  g.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert time.time() - t0 < 60.0
    assert int(status.item()) == -5
    monkeypatch.delenv("PAGEDATTN_PREFILL_WAIT_NS")
    _check(case, cuda_device)  # clean status, oracle parity


@pytest.mark.slow
@pytest.mark.parametrize("path", PATHS)
def test_varlen_prefill_full_size_sampled(cuda_device, monkeypatch, path):
    """16 sequences of 512..4096 tokens, Hq=28, Hkv=4: writeback then prefill;
    the shortest and the longest sequence checked against the oracle on every head."""
    pa = _pa()
    _set_path(monkeypatch, path)
    case = workloads.varlen_prefill(device=cuda_device)
    lens = case.seq_lens_host
    seqs = [int(np.argmin(lens)), int(np.argmax(lens))]
    # oracle inputs: the generator's pre-write pages of those sequences, written by the oracle's scatter
    args, rows = compact_for_oracle(case, seqs)
    ri = torch.tensor(rows, device=cuda_device)
    args["k_pool_bits"], args["v_pool_bits"] = oracle.kv_write_paged(
        args["k_pool_bits"], args["v_pool_bits"], bits(case.k_new[ri]), bits(case.v_new[ri]),
        args["cu_seqlens_q"], args["seq_lens"], args["block_table"], case.page_size)
    pa.kv_write_paged(case.k_pool, case.v_pool, case.k_new, case.v_new, case.cu_seqlens_q, case.seq_lens,
                      case.block_table)
    out, lse = _prefill(case, cuda_device)
    assert torch.isfinite(out.float()).all()
    ref_out, ref_lse = oracle.paged_attention(**args)  # every head of the sampled sequences
    assert_attention_close(out[rows], ref_out, lse[rows], ref_lse, what="varlen_prefill sampled")


@pytest.mark.slow
@pytest.mark.parametrize("path", PATHS)
def test_mixed_step_full_size_sampled(cuda_device, monkeypatch, path):
    """The mixed serving step in one call (4 prefill chunks of 2048 tokens after
    0..8192 cached tokens, 60 decodes of 1k..64k, one 131,072-token decode;
    Hq=32, Hkv=8): the chunk with the most prior tokens, the longest decode and
    a mid-length decode against the oracle on every head; both paths."""
    monkeypatch.setenv("PAGEDATTN_PREFILL_PATH", path)
    case = workloads.mixed_step(device=cuda_device)
    out, lse = _prefill(case, cuda_device)
    assert torch.isfinite(out.float()).all()
    lens = case.seq_lens_host
    chunks = [b for b in range(4)]
    chunk = max(chunks, key=lambda b: lens[b])
    decs = list(range(4, len(lens)))
    longest = max(decs, key=lambda b: lens[b])
    mid = sorted(decs, key=lambda b: lens[b])[len(decs) // 2]
    seqs = [chunk, mid, longest]
    args, rows = compact_for_oracle(case, seqs)
    ref_out, ref_lse = oracle.paged_attention(**args)  # every head of the sampled sequences
    assert_attention_close(out[rows], ref_out, lse[rows], ref_lse, what="mixed_step sampled")


@pytest.mark.parametrize("name,seq_lens,q_lens,hq,hkv,d,ps", [CASES[-3], CASES[-1]], ids=["g4", "d64"])
def test_mixed_call_with_every_segment_split(cuda_device, monkeypatch, name, seq_lens, q_lens, hq, hkv, d, ps):
    """PAGEDATTN_DECODE_CHUNK=1 cuts the decode rows' KV into one-unit chunks, so
    every short entry's result comes out of the log-sum-exp merge."""
    monkeypatch.setenv("PAGEDATTN_DECODE_CHUNK", "1")
    case = workloads.make_paged_case(name, seq_lens, q_lens, hq, hkv, d, page_size=ps, seed=len(name) * 7 + d)
    _check(case, cuda_device)
