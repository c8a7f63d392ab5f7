"""Pins for the CPU oracle: it is checked against things other than itself.

* an independent scalar pure-Python restatement (``oracle.brute``) on tiny
  inputs;
* a library special case: torch's CPU ``scaled_dot_product_attention`` in
  float64 on contiguous K/V;
* the tiled online-softmax recurrence and the split-KV log-sum-exp combine
  ("The Stack Below the Stack, Part 2", sections 2.1 and 2.2) equal the
  materialised result;
* closed forms and invariants the pages and the mathematics fix;
* planted mistakes in copies of the oracle fail these pins.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute, tiled
from oracle.attention import attention_rows, bf16_bits_to_f64, gather_kv_rows, paged_attention
from paged_kv_decode_17_gb300 import roofline
import workloads
from tests.conftest import bits, np_i32, oracle_args

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _brute_from_case(case):
    a = oracle_args(case)
    out, lse = brute.attention(
        a["q_bits"].tolist(), a["k_pool_bits"].tolist(), a["v_pool_bits"].tolist(), a["block_table"].tolist(),
        a["seq_lens"], a["cu_seqlens_q"].tolist(), a["num_q_heads"], a["num_kv_heads"], a["page_size"],
        a["scale"])
    return np.array(out), np.array(lse)


def _small_cases():
    cs = [workloads.tiny_decode(seed=0), workloads.tiny_decode(seed=0, sharp=True)]
    cs.append(workloads.make_paged_case("prefill_prior", [40, 23], [9, 23], 6, 2, 16, page_size=4, seed=5))
    cs.append(workloads.make_paged_case("mha", [17, 5, 33], [1, 2, 3], 3, 3, 8, page_size=16, seed=6))
    cs.append(workloads.make_paged_case("mqa_empty", [0, 12], [1, 4], 4, 1, 8, page_size=8, seed=7, num_pages=5))
    return cs


@pytest.mark.parametrize("idx", range(5))
def test_oracle_matches_brute_force(idx):
    case = _small_cases()[idx]
    out, lse = paged_attention(**oracle_args(case))
    bout, blse = _brute_from_case(case)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, bout, rtol=0, atol=1e-12)
    fin = np.isfinite(blse)
    assert (np.isfinite(lse) == fin).all()
    np.testing.assert_allclose(lse[fin], blse[fin], rtol=0, atol=1e-12)


def _contiguous_kv(case, b, g):
    """Logical K, V of sequence b / KV head g via torch indexing (not the oracle's gather)."""
    L = case.seq_lens_host[b]
    ps = case.page_size
    pos = torch.arange(L)
    phys = case.block_table[b].long()[pos // ps]
    K = case.k_pool[phys, g, pos % ps, :].double()
    V = case.v_pool[phys, g, pos % ps, :].double()
    return K, V


@pytest.mark.parametrize("name,seq_lens,q_lens", [
    ("noprior", [64, 33], [64, 33]),
    ("prior", [70, 40], [20, 1]),
])
def test_oracle_matches_torch_sdpa_fp64(name, seq_lens, q_lens):
    case = workloads.make_paged_case(name, seq_lens, q_lens, 8, 2, 32, page_size=16, seed=11)
    out, lse = paged_attention(**oracle_args(case))
    group = case.num_q_heads // case.num_kv_heads
    cu = case.cu_seqlens_q.tolist()
    for b in range(case.batch):
        L, ql = seq_lens[b], q_lens[b]
        for h in range(case.num_q_heads):
            K, V = _contiguous_kv(case, b, h // group)
            q = case.q[cu[b]:cu[b + 1], h, :].double()
            if ql == L:
                ref = torch.nn.functional.scaled_dot_product_attention(
                    q[None, None], K[None, None], V[None, None], is_causal=True, scale=case.softmax_scale)[0, 0]
            else:
                i = torch.arange(ql)[:, None]
                j = torch.arange(L)[None, :]
                mask = j <= (L - ql + i)
                ref = torch.nn.functional.scaled_dot_product_attention(
                    q[None, None], K[None, None], V[None, None], attn_mask=mask[None, None],
                    scale=case.softmax_scale)[0, 0]
            np.testing.assert_allclose(out[cu[b]:cu[b + 1], h, :], ref.numpy(), rtol=0, atol=1e-10)


def test_multiquery_rows_are_truncated_decodes():
    """A block of q_len query rows at the end of a sequence: row i is exactly a
    one-row decode of the same sequence cut to seq_len - q_len + i + 1 keys
    (causal inside the block, every earlier token visible).  Pins the
    position offset of short query blocks against the oracle's decode."""
    q_lens = [4, 8, 1, 3]
    seq_lens = [40, 8, 17, 3]
    case = workloads.make_paged_case("mq_pin", seq_lens, q_lens, 14, 2, 16, page_size=8, seed=41)
    a = oracle_args(case)
    out, lse = paged_attention(**a)
    cu = case.cu_seqlens_q.tolist()
    for b, (L, ql) in enumerate(zip(seq_lens, q_lens)):
        for i in range(ql):
            row = cu[b] + i
            one = dict(a)
            one["q_bits"] = a["q_bits"][row:row + 1]
            one["block_table"] = a["block_table"][b:b + 1]
            one["seq_lens"] = [L - ql + i + 1]
            one["cu_seqlens_q"] = np.array([0, 1], dtype=np.int32)
            o1, l1 = paged_attention(**one)
            np.testing.assert_allclose(out[row], o1[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[row], l1[0], rtol=0, atol=1e-12)


def test_tiled_online_softmax_equals_untiled():
    rng = np.random.default_rng(3)
    for trial in range(20):
        n = int(rng.integers(1, 300))
        D = int(rng.choice([4, 16, 64]))
        q = rng.standard_normal(D)
        K = rng.standard_normal((n, D)) * (1 + 3 * (trial % 3))
        V = rng.standard_normal((n, D))
        scale = 1 / math.sqrt(D)
        ref_o, ref_lse = attention_rows(q[None], K, V, [n - 1], scale)
        tiles = [int(x) for x in rng.integers(1, 40, size=5)] + [1]
        nchunks = int(rng.integers(1, 9))
        bounds = sorted(set([0, n] + [int(x) for x in rng.integers(0, n + 1, size=nchunks)]))
        o, lse = tiled.split_decode(q, K, V, scale, bounds, tiles)
        np.testing.assert_allclose(o, ref_o[0], rtol=0, atol=1e-12)
        assert abs(lse - ref_lse[0]) < 1e-12
        # one tile, one chunk, and tile size 1 all agree too
        for tl in ([1], [n]):
            o1, l1 = tiled.split_decode(q, K, V, scale, [0, n], tl)
            np.testing.assert_allclose(o1, ref_o[0], rtol=0, atol=1e-12)


def test_combine_skips_empty_chunks():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((10, 8))
    V = rng.standard_normal((10, 8))
    q = rng.standard_normal(8)
    o, lse = tiled.split_decode(q, K, V, 0.3, [0, 0, 4, 4, 10, 10], [3])
    ref_o, ref_lse = attention_rows(q[None], K, V, [9], 0.3)
    np.testing.assert_allclose(o, ref_o[0], atol=1e-12)
    o_e, lse_e = tiled.combine([(np.zeros(8), -math.inf)] * 3)
    assert lse_e == -math.inf and (o_e == 0).all()


def test_two_key_closed_form():
    # two keys: weights are the logistic function of the score difference
    q = np.array([1.0, -2.0, 0.5])
    K = np.array([[0.3, 0.1, -1.0], [1.5, -0.2, 0.4]])
    V = np.array([[1.0, 0.0, 2.0], [-1.0, 3.0, 0.0]])
    s = 0.7 * (K @ q)
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    o, lse = attention_rows(q[None], K, V, [1], 0.7)
    np.testing.assert_allclose(o[0], w0 * V[0] + (1 - w0) * V[1], atol=1e-15)
    assert abs(lse[0] - math.log(math.exp(s[0]) + math.exp(s[1]))) < 1e-14
    # position 0 sees only key 0: the output is V[0] exactly, lse = s0
    o, lse = attention_rows(q[None], K, V, [0], 0.7)
    assert (o[0] == V[0]).all() and lse[0] == s[0]


def test_identical_keys_give_mean_of_values():
    case = workloads.make_paged_case("ident", [45], [1], 2, 1, 16, seed=21)
    k = case.k_pool.clone()
    phys = case.block_table[0, :3].long()
    row = k[phys[0], 0, 0, :].clone()
    for j in range(45):
        k[phys[j // 16], 0, j % 16, :] = row
    case.k_pool = k
    out, lse = paged_attention(**oracle_args(case))
    K, V = _contiguous_kv(case, 0, 0)
    np.testing.assert_allclose(out[0, 0], V.mean(0).numpy(), atol=1e-13)
    qv = bf16_bits_to_f64(bits(case.q)[0, 0])
    s = case.softmax_scale * float(qv @ bf16_bits_to_f64(bits(row)))
    assert abs(lse[0, 0] - (s + math.log(45))) < 1e-12


def test_single_key_returns_its_value_row():
    case = workloads.make_paged_case("one", [1, 1], [1, 1], 4, 2, 64, seed=22)
    out, _ = paged_attention(**oracle_args(case))
    for b in range(2):
        for h in range(4):
            phys = int(case.block_table[b, 0])
            v = bf16_bits_to_f64(bits(case.v_pool)[phys, h // 2, 0])
            assert (out[b, h] == v).all()


def test_causal_mask_hides_future_positions():
    case = workloads.make_paged_case("causal", [50], [12], 4, 2, 32, page_size=16, seed=23)
    out, lse = paged_attention(**oracle_args(case))
    # overwrite K/V at positions >= 45: query rows at positions < 45 must not change
    L, ql = 50, 12
    k = case.k_pool.clone()
    v = case.v_pool.clone()
    for pos in range(45, 50):
        phys = int(case.block_table[0, pos // 16])
        k[phys, :, pos % 16, :] = 7.0
        v[phys, :, pos % 16, :] = -9.0
    case.k_pool, case.v_pool = k, v
    out2, lse2 = paged_attention(**oracle_args(case))
    n_unchanged = 45 - (L - ql)
    assert (out2[:n_unchanged] == out[:n_unchanged]).all()
    assert (lse2[:n_unchanged] == lse[:n_unchanged]).all()
    assert not np.allclose(out2[n_unchanged:], out[n_unchanged:])


def test_page_permutation_leaves_output_unchanged():
    case = workloads.make_paged_case("perm", [70, 33], [3, 1], 4, 2, 16, page_size=16, num_pages=12, seed=24)
    out, lse = paged_attention(**oracle_args(case))
    perm = torch.randperm(12, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(12)
    case2 = workloads.PagedCase(**{**case.__dict__})
    case2.k_pool = case.k_pool[perm]  # new page i holds old page perm[i]
    case2.v_pool = case.v_pool[perm]
    bt = case.block_table.clone()
    valid = bt >= 0
    bt[valid] = inv[bt[valid].long()].to(torch.int32)
    case2.block_table = bt
    out2, lse2 = paged_attention(**oracle_args(case2))
    assert (out2 == out).all() and (lse2 == lse).all()


def test_softmax_shift_invariance():
    rng = np.random.default_rng(25)
    D = 16
    q = rng.standard_normal(D)
    K = rng.standard_normal((30, D))
    V = rng.standard_normal((30, D))
    u = rng.standard_normal(D)
    o, lse = attention_rows(q[None], K, V, [29], 0.25)
    o2, lse2 = attention_rows(q[None], K + u[None, :], V, [29], 0.25)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    assert abs((lse2[0] - lse[0]) - 0.25 * float(q @ u)) < 1e-12


def test_nan_in_unread_memory_is_never_read():
    case = workloads.tiny_decode(seed=1)
    # the generator NaN-poisons unused pages and tail slots
    kb = bits(case.k_pool)
    assert (kb == workloads.BF16_NAN_BITS).any()
    out, lse = paged_attention(**oracle_args(case))
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_empty_sequence_defined_result():
    case = workloads.awkward_cases()["empty_seq"]
    out, lse = paged_attention(**oracle_args(case))
    for b, L in enumerate(case.seq_lens_host):
        if L == 0:
            assert (out[b] == 0).all() and np.isneginf(lse[b]).all()
        else:
            assert np.isfinite(out[b]).all()


def test_bf16_decoding():
    # exact values of a few bf16 patterns (IEEE binary32 upper halves)
    pats = np.array([0x3F80, 0xBF80, 0x4000, 0x3F00, 0x0000, 0x8000, 0x7F80, 0x0001, 0x4049], dtype=np.uint16)
    want = [1.0, -1.0, 2.0, 0.5, 0.0, -0.0, math.inf, 2.0 ** -133, 3.140625]
    got = bf16_bits_to_f64(pats)
    assert got.tolist() == want
    # agrees with torch's bf16 -> float64 on random patterns (excluding NaN)
    r = np.random.default_rng(0).integers(0, 1 << 16, size=4096).astype(np.uint16)
    r = r[(r & 0x7F80) != 0x7F80]
    t = torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert (bf16_bits_to_f64(r) == t).all()


def test_kv_write_oracle_bit_exact_and_roundtrip():
    case = workloads.make_paged_case("wb", [40, 17, 5], [9, 17, 1], 4, 2, 16, page_size=16, prewritten=False,
                                     num_pages=9, seed=26)
    a = oracle_args(case)
    kp, vp = oracle.kv_write_paged(a["k_pool_bits"], a["v_pool_bits"], bits(case.k_new), bits(case.v_new),
                                   a["cu_seqlens_q"], a["seq_lens"], a["block_table"], case.page_size)
    # brute force restatement: iterate over every pool slot and decide what it must hold
    want_k = a["k_pool_bits"].copy()
    want_v = a["v_pool_bits"].copy()
    kn, vn = bits(case.k_new), bits(case.v_new)
    cu = a["cu_seqlens_q"]
    for b, L in enumerate(case.seq_lens_host):
        n = int(cu[b + 1] - cu[b])
        for p in range(a["block_table"].shape[1]):
            phys = int(a["block_table"][b, p])
            if phys < 0:
                continue
            for slot in range(case.page_size):
                pos = p * case.page_size + slot
                if L - n <= pos < L:
                    want_k[phys, :, slot] = kn[cu[b] + pos - (L - n)]
                    want_v[phys, :, slot] = vn[cu[b] + pos - (L - n)]
    assert (kp == want_k).all() and (vp == want_v).all()
    # untouched bytes unchanged
    changed = (kp != a["k_pool_bits"]).any(axis=(1, 3))
    assert changed.sum() <= sum(case.q_lens_host)
    # reading back through the table returns the written rows
    for b, L in enumerate(case.seq_lens_host):
        n = int(cu[b + 1] - cu[b])
        K = gather_kv_rows(kp, a["block_table"][b], L, 1, case.page_size)
        np.testing.assert_array_equal(K[L - n:], bf16_bits_to_f64(kn[cu[b]:cu[b + 1], 1]))
    # after the writeback nothing NaN is visible to attention
    out, _ = paged_attention(**{**a, "k_pool_bits": kp, "v_pool_bits": vp})
    assert np.isfinite(out).all()


def _golden(name):
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    vals = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = int(v)
    return vals


def test_traffic_byte_model_matches_pages():
    g = _golden("attention_traffic.txt")
    # one head, 4,096 tokens, D = 128, bf16: K and V read once = 2 MiB
    assert roofline.decode_kv_bytes([4096], num_kv_heads=1, head_dim=128) == g["tiled_kv_bytes_per_head"]
    assert roofline.decode_kv_bytes([4096], 1, 128) == g["decode_kv_bytes_per_head_ctx4096"]
    # the naive score matrix figures are products the page prints
    assert 4096 * 4096 * 2 == g["naive_score_matrix_bytes_per_head"]
    assert 3 * g["naive_score_matrix_bytes_per_head"] == g["naive_three_pass_bytes_per_head"]
    assert 4096 * 2 == g["decode_score_vector_bytes_ctx4096"]
    assert 32768 ** 2 * 2 == g["score_matrix_bytes_n32768_fp16"]
    # ~50x less traffic tiled vs naive, as the page says
    assert 40 < g["naive_three_pass_bytes_per_head"] / g["tiled_kv_bytes_per_head"] < 60
    # visible pairs: a causal L x L block keeps L(L+1)/2 pairs; with P prior keys q*P more
    assert roofline.visible_pairs([4], [4]) == 10
    assert roofline.visible_pairs([2], [5]) == 2 * 3 + 3
    assert roofline.visible_pairs([1], [9]) == 9
    # qwen-shaped decode: 32 x 8192 tokens, 4 KV heads, D=128 -> 512 MiB
    assert roofline.decode_kv_bytes([8192] * 32, 4, 128) == 536870912


# ---- planted mistakes: copies of the oracle with one plausible bug each must fail a pin ----

def _mut_top_left_causal(**kw):
    # bug: query i sees keys 0..i (top-left alignment) instead of prior+i
    from oracle import attention as A
    orig = A.attention_rows

    def wrong(q_rows, keys, values, positions, scale):
        prior = positions[0] - 0 if len(positions) else 0
        return orig(q_rows, keys, values, [p - positions[0] for p in positions], scale)
    A.attention_rows, saved = wrong, orig
    try:
        return paged_attention(**kw)
    finally:
        A.attention_rows = saved


def _mut_gqa_modulo(**kw):
    # bug: query head h reads KV head h % Hkv (interleaved) instead of h // group
    q = kw["q_bits"]
    Hq, Hkv = kw["num_q_heads"], kw["num_kv_heads"]
    g = Hq // Hkv
    perm = [(h % Hkv) * g + h // Hkv for h in range(Hq)]
    kw2 = dict(kw)
    kw2["q_bits"] = q[:, np.argsort(perm), :]
    out, lse = paged_attention(**kw2)
    return out[:, perm, :], lse[:, perm]


def _mut_no_scale(**kw):
    return paged_attention(**{**kw, "scale": 1.0})


def _mut_off_by_one_page(**kw):
    bt = kw["block_table"].copy()
    bt[:, :] = np.roll(bt, 1, axis=1)
    bt[bt < 0] = 0
    return paged_attention(**{**kw, "block_table": bt})


@pytest.mark.parametrize("mutant", [_mut_top_left_causal, _mut_gqa_modulo, _mut_no_scale, _mut_off_by_one_page])
def test_planted_oracle_mistakes_are_caught(mutant):
    case = workloads.make_paged_case("mut", [40, 23], [9, 3], 4, 2, 16, page_size=8, seed=27)
    a = oracle_args(case)
    bout, _ = _brute_from_case(case)
    with np.errstate(all="ignore"):
        out, _ = mutant(**a)
    assert not (np.isfinite(out).all() and np.allclose(out, bout, atol=1e-6)), "planted mistake went unnoticed"


# ------------------------------------------------------------------ rotary embedding / RMS norm
def test_rope_position_zero_is_identity():
    x = np.random.default_rng(50).standard_normal((3, 128))
    np.testing.assert_array_equal(oracle.rope_rotate_half(x, 0, 10000.0), x)


def test_rope_two_dims_is_a_plane_rotation():
    """D = 2: one pair with frequency base**0 = 1, rotated by `pos` radians."""
    x = np.array([0.3, -1.7])
    for pos in (1, 5, 1000):
        c, s = math.cos(pos), math.sin(pos)
        want = np.array([0.3 * c + 1.7 * s, -1.7 * c + 0.3 * s])
        np.testing.assert_allclose(oracle.rope_rotate_half(x, pos, 500.0), want, rtol=0, atol=1e-12)


def test_rope_worked_example_rotate_half_pairing():
    """D = 4, base 10000: pair 0 = dims (0, 2) turns by pos rad, pair 1 = dims
    (1, 3) by pos * 10000**(-1/2) = pos / 100 rad.  Unit vectors show the pairing."""
    e0 = np.array([1.0, 0.0, 0.0, 0.0])
    e1 = np.array([0.0, 1.0, 0.0, 0.0])
    np.testing.assert_allclose(oracle.rope_rotate_half(e0, 1, 10000.0),
                               [math.cos(1.0), 0.0, math.sin(1.0), 0.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.rope_rotate_half(e1, 100, 10000.0),
                               [0.0, math.cos(1.0), 0.0, math.sin(1.0)], rtol=0, atol=1e-12)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(51)
    x = rng.standard_normal(128)
    y = oracle.rope_rotate_half(x, 12345, 1e6)
    np.testing.assert_allclose(np.hypot(y[:64], y[64:]), np.hypot(x[:64], x[64:]), rtol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    """The defining property of rotary embeddings: <R(m) q, R(n) k> = <q, R(n - m) k>."""
    rng = np.random.default_rng(52)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n in ((0, 7), (100, 37), (5000, 5003), (131071, 2)):
        lhs = oracle.rope_rotate_half(q, m, 10000.0) @ oracle.rope_rotate_half(k, n, 10000.0)
        rhs = q @ oracle.rope_rotate_half(k, n - m, 10000.0)
        assert abs(lhs - rhs) <= 1e-9 * (1 + abs(rhs))


def test_rms_norm_closed_forms():
    np.testing.assert_allclose(oracle.rms_norm(np.array([3.0, 4.0]), None, 0.0),
                               np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15)
    x = np.random.default_rng(53).standard_normal(128)
    y = oracle.rms_norm(x, None, 0.0)
    assert abs(np.mean(y * y) - 1.0) < 1e-13
    np.testing.assert_allclose(oracle.rms_norm(7.5 * x, None, 0.0), y, rtol=1e-13)
    w = np.linspace(0.5, 2.0, 128)
    np.testing.assert_allclose(oracle.rms_norm(x, w, 1e-6), oracle.rms_norm(x, None, 1e-6) * w, rtol=1e-15)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: rounds to the even one (1)
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.0 - 2.0 ** -7, 1.0 + 2.0 ** -9, 3.0])
    want = np.array([1.0, 1.0 + 2.0 ** -6, -2.0, 1.0, 3.0])
    np.testing.assert_array_equal(oracle.round_to_bf16_f64(v), want)
    np.testing.assert_array_equal(oracle.bf16_ulp(np.array([1.0, 1.5, 2.0, -0.75])),
                                  [2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -8])


def test_rope_writeback_rows_positions_and_norm_order():
    """Row i of n new rows of a sequence of length L is rotated at L - n + i,
    after its RMS norm (the rotation keeps the norm, so the normalised row's
    mean square survives it)."""
    rng = np.random.default_rng(54)
    T, Hkv, D = 5, 2, 16
    k = (rng.standard_normal((T, Hkv, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    cu, lens = [0, 3, 5], [10, 2]
    w = np.full(D, 0x3F80, dtype=np.uint16)  # bf16 1.0
    out, _, pos = oracle.rope_writeback_rows(k, None, cu, lens, 10000.0, k_norm_weight_bits=w, eps=0.0)
    np.testing.assert_array_equal(pos, [7, 8, 9, 0, 1])
    np.testing.assert_allclose(np.mean(out * out, axis=-1), 1.0, rtol=1e-12)
    kf = oracle.bf16_bits_to_f64(k)
    np.testing.assert_allclose(out[3], oracle.rms_norm(kf[3], None, 0.0), rtol=0, atol=1e-15)  # position 0


# ------------------------------------------------------------------ FP8 (e4m3) KV cache
def test_e4m3_decode_matches_torch_for_every_code():
    """All 256 codes against torch's float8_e4m3fn (an independent library decoder)."""
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(codes)
    assert (np.isnan(got) == np.isnan(want)).all()
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


def test_e4m3_closed_forms_and_round_trip():
    vals = oracle.e4m3_decode(np.array([0x7E, 0x01, 0x08, 0x38, 0xB8, 0x80, 0x00], dtype=np.uint8))
    np.testing.assert_array_equal(vals, [448.0, 2.0 ** -9, 2.0 ** -6, 1.0, -1.0, -0.0, 0.0])
    assert np.signbit(vals[5])
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_decode(finite)), finite)


def test_e4m3_encode_rounding_and_saturation():
    x = np.array([1.0625, 1.1875, 2.0 ** -10, 1.5 * 2.0 ** -10, 1000.0, -1e9, 464.0, float("nan")])
    # 1.0625 is halfway 1 (0x38) / 1.125 (0x39) -> even 0x38; 1.1875 halfway 1.125 / 1.25 -> even 0x3A;
    # 2^-10 halfway 0 / 2^-9 -> 0; beyond 448 saturates; NaN -> 0x7F
    np.testing.assert_array_equal(oracle.e4m3_encode(x), [0x38, 0x3A, 0x00, 0x01, 0x7E, 0xFE, 0x7E, 0x7F])


def test_e4m3_encode_matches_torch_in_range():
    """torch's float32 -> float8_e4m3fn cast rounds to nearest even; in range it is the same map."""
    rng = np.random.default_rng(60)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 1e-2]).astype(np.float32)
    x = x[np.abs(x) < 440]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x), want)


def test_fp8_attention_equals_bf16_attention_on_the_same_values():
    """With power-of-two scales every dequantised value is exact in bf16: the
    FP8 oracle must then equal the (pinned) bf16 oracle on those values."""
    rng = np.random.default_rng(61)
    P, Hkv, ps, D, Hq = 12, 2, 16, 32, 6
    kc = rng.integers(0, 256, (P, Hkv, ps, D), dtype=np.uint8)
    vc = rng.integers(0, 256, (P, Hkv, D, ps), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x10  # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x22
    ks, vs = [0.25, 2.0], [0.5, 1.0 / 64]
    bt = np.array([[3, 7, 1, -1], [0, 11, 5, 9]])
    lens, qlens = [40, 61], [1, 5]
    cu = np.array([0, 1, 6])
    q = (rng.standard_normal((6, Hq, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

    def bf16_bits(v):
        return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

    kf = oracle.e4m3_decode(kc) * np.array(ks)[None, :, None, None]
    vf = np.swapaxes(oracle.e4m3_decode(vc) * np.array(vs)[None, :, None, None], 2, 3)
    want = paged_attention(q, bf16_bits(kf), bf16_bits(vf), bt, lens, cu, Hq, Hkv, ps, 0.2)
    got = oracle.paged_attention_fp8(q, kc, vc, ks, vs, bt, lens, cu, Hq, Hkv, ps, 0.2)
    np.testing.assert_allclose(got[0], want[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[1], want[1], rtol=0, atol=1e-12)


def test_fp8_writeback_placement_and_error_bound():
    """Rows land at (page, slot) of their position, V transposed; every code
    reads back within half an e4m3 step of x / scale (relative 2^-4, or 2^-10
    absolute in the subnormal range)."""
    rng = np.random.default_rng(62)
    P, Hkv, ps, D = 6, 2, 16, 16
    k0 = np.zeros((P, Hkv, ps, D), np.uint8)
    v0 = np.zeros((P, Hkv, D, ps), np.uint8)
    kn = (rng.standard_normal((3, Hkv, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    vn = (rng.standard_normal((3, Hkv, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ks, vs = [0.01, 0.02], [0.03, 0.005]
    bt = np.array([[4, 2], [1, 0]])
    kp, vp = oracle.kv_write_paged_fp8(k0, v0, kn, vn, ks, vs, [0, 2, 3], [17, 1], bt, ps)
    # sequence 0: rows at positions 15 (page 4 slot 15) and 16 (page 2 slot 0); sequence 1: position 0
    for (t, page, slot) in ((0, 4, 15), (1, 2, 0), (2, 1, 0)):
        for g in range(Hkv):
            x = bf16_bits_to_f64(kn[t, g]) / ks[g]
            back = oracle.e4m3_decode(kp[page, g, slot])
            assert (np.abs(back - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10) + 1e-12).all()
            xv = bf16_bits_to_f64(vn[t, g]) / vs[g]
            np.testing.assert_array_equal(vp[page, g, :, slot], oracle.e4m3_encode(xv.astype(np.float32)))
    written = np.zeros((P, ps), bool)
    written[4, 15] = written[2, 0] = written[1, 0] = True
    assert (np.moveaxis(kp, 2, 1)[~written] == 0).all() and (np.moveaxis(vp, 3, 1)[~written] == 0).all()
