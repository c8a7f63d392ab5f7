"""Seeded synthetic inputs for paged-KV attention.

This module only draws inputs: random bf16 queries and K/V pages, page
assignments, block tables and sequence lengths.  It holds none of the
attention arithmetic, so the CPU oracle (``oracle/``) and the CUDA library
(``paged_kv_decode_17_gb300``) can both be fed from it without sharing any
computation.

Shapes follow the serving workloads described on the pages:

* Ion blog ("Inside Ion", section "What That Buys"): Qwen2.5-7B at batch 32
  and 8k context -> ``qwen7b_decode`` (Hq=28, Hkv=4, D=128).
* "8. Kernels and Attention Backends" (section "Test the kernel at three
  levels"): ragged sequences, paged KV, one-token decode, long prefill,
  partially filled pages -> ``llama8b_ragged_decode``, ``varlen_prefill``,
  the awkward cases in ``awkward_cases``.
* "The Stack Below the Stack, Part 2" (section 2.2 Flash-Decoding): long
  contexts that need a split of the KV sequence -> the 131,072-token decode
  in ``mixed_step``.

Layout conventions (the pages leave them open; these are the library's):

* ``k_pool``/``v_pool``: bf16 ``[num_pages][Hkv][page_size][D]`` ("HND"),
  contiguous.
* ``q``: bf16 ``[total_q][Hq][D]``; rows of sequence ``b`` are
  ``cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1`` and sit at the LAST ``q_len``
  positions of the sequence (positions ``seq_len-q_len .. seq_len-1``).
* ``block_table``: int32 ``[B][max_pages_per_seq]``; entries past a
  sequence's last page are -1.
* Every pool slot that no sequence owns (unused pages, tail slots of a last
  partial page) holds bf16 NaN, so a kernel that reads memory it must not
  read produces a NaN that the tests see.
* ``k_new``/``v_new``: bf16 ``[total_q][Hkv][D]``: the K/V rows of the query
  positions.  With ``prewritten=True`` they are already in the pool (decode
  cases); with ``prewritten=False`` their pool slots are NaN until a
  writeback puts them there (prefill cases).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import torch

BF16_NAN_BITS = 0x7FC0


@dataclasses.dataclass
class PagedCase:
    """One batch of paged attention inputs (all tensors on ``device``)."""

    name: str
    q: torch.Tensor  # bf16 [total_q][Hq][D]
    k_pool: torch.Tensor  # bf16 [P][Hkv][ps][D]
    v_pool: torch.Tensor  # bf16 [P][Hkv][ps][D]
    k_new: torch.Tensor  # bf16 [total_q][Hkv][D]
    v_new: torch.Tensor  # bf16 [total_q][Hkv][D]
    block_table: torch.Tensor  # int32 [B][max_pages]
    seq_lens: torch.Tensor  # int32 [B]  (total KV length incl. the new rows)
    cu_seqlens_q: torch.Tensor  # int32 [B+1]
    page_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    softmax_scale: float
    prewritten: bool
    seq_lens_host: List[int]
    q_lens_host: List[int]

    @property
    def batch(self) -> int:
        return len(self.seq_lens_host)

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_seq_len(self) -> int:
        return max(self.seq_lens_host) if self.seq_lens_host else 0

    @property
    def max_q_len(self) -> int:
        return max(self.q_lens_host) if self.q_lens_host else 0

    def to(self, device) -> "PagedCase":
        fields = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            fields[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return PagedCase(**fields)


def _randn_bf16(shape, gen: torch.Generator, device, scale: float = 1.0) -> torch.Tensor:
    """N(0, 1) samples rounded to bf16 (round-to-nearest-even by torch)."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def _fill_randn_bf16_(t: torch.Tensor, gen: torch.Generator, rows_per_chunk: int = 1 << 14) -> None:
    """Fill a bf16 tensor with N(0,1) samples in chunks along dim 0 (bounded temporaries)."""
    n = t.shape[0]
    for s in range(0, n, rows_per_chunk):
        e = min(n, s + rows_per_chunk)
        t[s:e] = torch.randn(t[s:e].shape, generator=gen, device=t.device, dtype=torch.float32).to(torch.bfloat16)


def make_paged_case(
    name: str,
    seq_lens: Sequence[int],
    q_lens: Sequence[int],
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    page_size: int = 16,
    num_pages: Optional[int] = None,
    seed: int = 0,
    device="cpu",
    k_scale: float = 1.0,
    prewritten: bool = True,
    max_pages_per_seq: Optional[int] = None,
    softmax_scale: Optional[float] = None,
) -> PagedCase:
    """Draw one paged batch.

    Pages: each sequence needs ceil(seq_len/page_size) pages; the physical
    ids are taken, in order, from a seeded random permutation of the pool, so
    every sequence's pages are scattered and no page is shared.  Values: K, V
    and q are N(0,1) rounded to bf16 (K additionally multiplied by
    ``k_scale``, an exact power of two for the "sharp" variants); slots that
    no sequence owns are NaN.
    """
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    assert len(seq_lens) == len(q_lens)
    for s, ql in zip(seq_lens, q_lens):
        assert 0 <= ql <= s or (s == 0 and ql <= 1), (s, ql)
    B = len(seq_lens)
    ps = page_size
    pages_per_seq = [-(-s // ps) for s in seq_lens]
    need = sum(pages_per_seq)
    if num_pages is None:
        num_pages = max(1, need)
    assert num_pages >= need, (num_pages, need)
    if max_pages_per_seq is None:
        max_pages_per_seq = max([1] + pages_per_seq)
    gen = torch.Generator(device=device).manual_seed(seed)

    # page assignment: a seeded permutation of the pool, consumed in order
    perm = torch.randperm(num_pages, generator=gen, device=device).to(torch.int32)
    block_table = torch.full((B, max_pages_per_seq), -1, dtype=torch.int32, device=device)
    owner_rows = []  # (phys pages tensor, n_valid_tokens) per sequence
    off = 0
    for b in range(B):
        n = pages_per_seq[b]
        if n:
            block_table[b, :n] = perm[off : off + n]
        owner_rows.append(perm[off : off + n])
        off += n

    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    k_pool = torch.empty((num_pages, Hkv, ps, D), dtype=torch.bfloat16, device=device)
    v_pool = torch.empty((num_pages, Hkv, ps, D), dtype=torch.bfloat16, device=device)
    _fill_randn_bf16_(k_pool, gen, rows_per_chunk=max(1, (1 << 24) // (Hkv * ps * D)))
    _fill_randn_bf16_(v_pool, gen, rows_per_chunk=max(1, (1 << 24) // (Hkv * ps * D)))
    if k_scale != 1.0:
        k_pool.mul_(k_scale)

    # NaN-poison every slot that no sequence owns
    valid = torch.zeros((num_pages, ps), dtype=torch.bool, device=device)
    for b in range(B):
        n = pages_per_seq[b]
        if n == 0:
            continue
        phys = owner_rows[b].long()
        counts = torch.full((n,), ps, dtype=torch.int64, device=device)
        counts[-1] = seq_lens[b] - (n - 1) * ps
        slot_ok = torch.arange(ps, device=device)[None, :] < counts[:, None]
        valid[phys] = slot_ok
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=device)
    inval = (~valid)[:, None, :, None]
    k_pool.masked_fill_(inval, nan)
    v_pool.masked_fill_(inval, nan)

    total_q = sum(q_lens)
    q = _randn_bf16((total_q, Hq, D), gen, device)
    cu = [0]
    for ql in q_lens:
        cu.append(cu[-1] + ql)
    cu_seqlens_q = torch.tensor(cu, dtype=torch.int32, device=device)
    seq_lens_t = torch.tensor(seq_lens, dtype=torch.int32, device=device)

    # K/V rows of the query positions: taken from the pool for decode-style
    # cases (already written), drawn fresh (and NaN in the pool) otherwise.
    k_new = torch.empty((total_q, Hkv, D), dtype=torch.bfloat16, device=device)
    v_new = torch.empty((total_q, Hkv, D), dtype=torch.bfloat16, device=device)
    if prewritten:
        for b in range(B):
            if q_lens[b] == 0 or seq_lens[b] == 0:
                continue
            pos = torch.arange(seq_lens[b] - q_lens[b], seq_lens[b], device=device)
            phys = block_table[b].long()[pos // ps]
            slot = pos % ps
            k_new[cu[b] : cu[b + 1]] = k_pool[phys, :, slot, :]
            v_new[cu[b] : cu[b + 1]] = v_pool[phys, :, slot, :]
        if total_q and any(s == 0 for s in seq_lens):
            # q rows of empty sequences have no KV row; keep them finite
            for b in range(B):
                if seq_lens[b] == 0 and q_lens[b]:
                    k_new[cu[b] : cu[b + 1]] = 0
                    v_new[cu[b] : cu[b + 1]] = 0
    else:
        k_new.copy_(_randn_bf16((total_q, Hkv, D), gen, device, scale=k_scale))
        v_new.copy_(_randn_bf16((total_q, Hkv, D), gen, device))
        for b in range(B):
            if q_lens[b] == 0:
                continue
            pos = torch.arange(seq_lens[b] - q_lens[b], seq_lens[b], device=device)
            phys = block_table[b].long()[pos // ps]
            slot = pos % ps
            k_pool[phys, :, slot, :] = nan
            v_pool[phys, :, slot, :] = nan

    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    return PagedCase(
        name=name,
        q=q,
        k_pool=k_pool,
        v_pool=v_pool,
        k_new=k_new,
        v_new=v_new,
        block_table=block_table,
        seq_lens=seq_lens_t,
        cu_seqlens_q=cu_seqlens_q,
        page_size=ps,
        num_q_heads=Hq,
        num_kv_heads=Hkv,
        head_dim=D,
        softmax_scale=float(softmax_scale),
        prewritten=prewritten,
        seq_lens_host=seq_lens,
        q_lens_host=q_lens,
    )


def _uniform_ints(gen: torch.Generator, lo: int, hi: int, n: int) -> List[int]:
    """n integers uniform on [lo, hi] inclusive, drawn on the CPU."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


# ---------------------------------------------------------------------------
# The five workload shapes.  Each returns a PagedCase.
# ---------------------------------------------------------------------------

def tiny_decode(seed: int = 0, device="cpu", sharp: bool = False) -> PagedCase:
    """Batch 2, seq_lens {37, 100}, Hq=4, Hkv=2, D=64, 16-token pages in a
    shuffled pool of 16 pages (10 used); the sharp variant scales K by 4."""
    return make_paged_case(
        "tiny_decode_sharp" if sharp else "tiny_decode",
        seq_lens=[37, 100], q_lens=[1, 1], num_q_heads=4, num_kv_heads=2, head_dim=64,
        page_size=16, num_pages=16, seed=seed, device=device, k_scale=4.0 if sharp else 1.0,
    )


def qwen7b_decode(seed: int = 1, device="cpu", batch: int = 32, ctx: int = 8192) -> PagedCase:
    """Qwen2.5-7B-shaped decode: batch 32 at 8192 tokens, Hq=28, Hkv=4, D=128,
    16-token pages; the pool is exactly the 16,384 pages needed, assigned by a
    seeded permutation; one query per sequence."""
    return make_paged_case(
        "qwen7b_decode", seq_lens=[ctx] * batch, q_lens=[1] * batch, num_q_heads=28,
        num_kv_heads=4, head_dim=128, page_size=16, num_pages=batch * (-(-ctx // 16)),
        seed=seed, device=device,
    )


def qwen7b_multiquery(seed: int = 5, device="cpu", batch: int = 32, ctx: int = 8192, q_len: int = 4) -> PagedCase:
    """The qwen7b_decode shape with a block of q_len query rows per sequence
    (speculative-decode verification: the last q_len of the ctx tokens are
    the proposed ones, their K/V already in the pages)."""
    return make_paged_case(
        "qwen7b_multiquery", seq_lens=[ctx] * batch, q_lens=[q_len] * batch, num_q_heads=28,
        num_kv_heads=4, head_dim=128, page_size=16, num_pages=batch * (-(-ctx // 16)),
        seed=seed, device=device,
    )


def llama8b_ragged_lens(seed: int = 2, batch: int = 64, max_len: int = 32768) -> List[int]:
    gen = torch.Generator().manual_seed(seed)
    return _uniform_ints(gen, 1, max_len, batch)


def llama8b_ragged_decode(seed: int = 2, device="cpu", batch: int = 64, max_len: int = 32768,
                          num_pages: int = 131072) -> PagedCase:
    """Ragged Llama-3-8B-shaped decode: batch 64, seq_lens uniform on
    [1, 32768], Hq=32, Hkv=8, D=128, 16-token pages scattered over a
    131,072-page pool."""
    lens = llama8b_ragged_lens(seed, batch, max_len)
    return make_paged_case(
        "llama8b_ragged_decode", seq_lens=lens, q_lens=[1] * batch, num_q_heads=32,
        num_kv_heads=8, head_dim=128, page_size=16, num_pages=num_pages,
        max_pages_per_seq=-(-max_len // 16), seed=seed, device=device,
    )


def varlen_prefill_lens(seed: int = 3, nseq: int = 16, lo: int = 512, hi: int = 4096) -> List[int]:
    gen = torch.Generator().manual_seed(seed)
    return _uniform_ints(gen, lo, hi, nseq)


def varlen_prefill(seed: int = 3, device="cpu", nseq: int = 16, lo: int = 512, hi: int = 4096,
                   num_q_heads: int = 28, num_kv_heads: int = 4, head_dim: int = 128) -> PagedCase:
    """Varlen causal prefill with paged KV writeback: 16 sequences with
    lengths uniform on [512, 4096], no prior tokens, Hq=28, Hkv=4, D=128; the
    new K/V rows are not yet in the pool (their slots are NaN) and go to
    randomly assigned 16-token pages."""
    lens = varlen_prefill_lens(seed, nseq, lo, hi)
    need = sum(-(-s // 16) for s in lens)
    return make_paged_case(
        "varlen_prefill", seq_lens=lens, q_lens=lens, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=16,
        num_pages=need + need // 8 + 1, seed=seed, device=device, prewritten=False,
    )


def mixed_step_lens(seed: int = 4):
    gen = torch.Generator().manual_seed(seed)
    priors = _uniform_ints(gen, 0, 8192, 4)
    dec = _uniform_ints(gen, 1024, 65536, 60)
    seq_lens = [p + 2048 for p in priors] + dec + [131072]
    q_lens = [2048] * 4 + [1] * 61
    return seq_lens, q_lens


def mixed_step(seed: int = 4, device="cpu") -> PagedCase:
    """Mixed serving step: 4 prefill chunks of 2048 tokens, each after 0-8192
    prior cached tokens, plus 60 decodes with contexts uniform on
    [1024, 65536] and one 131,072-token decode; Hq=32, Hkv=8, D=128, 16-token
    pages; the pool is the pages needed plus 10% slack, shuffled.  The K/V of
    every query position is already in the pool (written by an earlier
    writeback in the same step)."""
    seq_lens, q_lens = mixed_step_lens(seed)
    need = sum(-(-s // 16) for s in seq_lens)
    return make_paged_case(
        "mixed_step", seq_lens=seq_lens, q_lens=q_lens, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, num_pages=need + need // 10, seed=seed, device=device,
    )


def mixed_step_small(seed: int = 4, device="cpu") -> PagedCase:
    """The mixed step at profiling size: the same 4 prefill chunks of 2048 tokens
    after 0-8192 prior tokens, 60 decodes with contexts uniform on [1024, 4096]
    and one 16,384-token decode (about 0.7 GB of KV, still above L2)."""
    gen = torch.Generator().manual_seed(seed)
    priors = _uniform_ints(gen, 0, 8192, 4)
    dec = _uniform_ints(gen, 1024, 4096, 60)
    seq_lens = [p + 2048 for p in priors] + dec + [16384]
    q_lens = [2048] * 4 + [1] * 61
    need = sum(-(-s // 16) for s in seq_lens)
    return make_paged_case(
        "mixed_step_small", seq_lens=seq_lens, q_lens=q_lens, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, num_pages=need + need // 10, seed=seed, device=device,
    )


def llama8b_ragged_small(seed: int = 2, device="cpu") -> PagedCase:
    """The ragged Llama-3-8B-shaped decode at profiling size: batch 16 with
    contexts uniform on [1, 32768] (the first 16 of the batch-64 draw), pool
    = the pages needed (about 1 GB of KV)."""
    lens = llama8b_ragged_lens(seed, 64, 32768)[:16]
    need = sum(-(-s // 16) for s in lens)
    return make_paged_case(
        "llama8b_ragged_small", seq_lens=lens, q_lens=[1] * 16, num_q_heads=32, num_kv_heads=8, head_dim=128,
        page_size=16, num_pages=need, max_pages_per_seq=32768 // 16, seed=seed, device=device,
    )


def awkward_cases(device="cpu", seed: int = 10) -> Dict[str, PagedCase]:
    """Small cases at the places fast paths skip work: one-token contexts,
    partially filled pages, contexts 127 and 4096, batch 1 and 32, extreme
    logits, an empty sequence, GQA groups 1..8, head_dim 64 and 128, pages of
    16, 64 and 256 tokens."""
    cases = {}
    cases["one_token"] = make_paged_case("one_token", [1, 1, 1], [1, 1, 1], 8, 2, 128, seed=seed, device=device)
    cases["ctx127_b1"] = make_paged_case("ctx127_b1", [127], [1], 8, 8, 128, num_pages=20, seed=seed + 1, device=device)
    cases["ctx4096_b32"] = make_paged_case("ctx4096_b32", [4096] * 32, [1] * 32, 8, 2, 64, seed=seed + 2, device=device)
    cases["partial_pages"] = make_paged_case("partial_pages", [15, 16, 17, 31, 33, 255], [1] * 6, 16, 4, 128,
                                             num_pages=40, seed=seed + 3, device=device)
    cases["extreme_logits"] = make_paged_case("extreme_logits", [300, 45], [1, 1], 4, 1, 128, k_scale=64.0,
                                              seed=seed + 4, device=device)
    cases["empty_seq"] = make_paged_case("empty_seq", [0, 50, 0, 7], [1, 1, 1, 1], 4, 2, 64, num_pages=12,
                                         seed=seed + 5, device=device)
    cases["mha_group1"] = make_paged_case("mha_group1", [200, 33], [1, 1], 4, 4, 128, seed=seed + 6, device=device)
    cases["group16"] = make_paged_case("group16", [513, 64], [1, 1], 32, 2, 128, seed=seed + 7, device=device)
    cases["group32_mqa"] = make_paged_case("group32_mqa", [129, 700], [1, 1], 32, 1, 64, seed=seed + 8, device=device)
    cases["page64"] = make_paged_case("page64", [100, 300], [1, 1], 8, 2, 128, page_size=64, seed=seed + 9,
                                      device=device)
    cases["page256"] = make_paged_case("page256", [600, 257, 1], [1, 1, 1], 8, 2, 128, page_size=256,
                                       seed=seed + 10, device=device)
    return cases
