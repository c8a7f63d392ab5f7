"""Algorithmic work of each call: the numerators of the roofline fractions.

* Decode KV bytes: every key and value row of every (sequence, KV head) is
  read once, ``sum_b seq_len_b * Hkv * D * 2 (K and V) * 2 bytes``.  Queries,
  outputs and block tables are not counted.  This is the byte count of
  "8. Kernels and Attention Backends", section "Counting attention's traffic"
  (decode reads about 2 x 4,096 x 128 x 2 bytes = 2 MiB per head at a
  4,096-token history).
* Prefill flops: ``4 * D * Hq * (visible query-key pairs)``; a query at
  absolute position ``t`` sees ``t + 1`` keys.  Masked pairs are not counted.
* Writeback bytes: each new K and V row is read once and written once.
"""

from __future__ import annotations

from typing import Sequence


def decode_kv_bytes(seq_lens: Sequence[int], num_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    return int(sum(int(x) for x in seq_lens)) * num_kv_heads * head_dim * 2 * elem_bytes


def visible_pairs(q_lens: Sequence[int], seq_lens: Sequence[int]) -> int:
    """Number of (query, key) pairs a causal, bottom-right aligned mask keeps."""
    total = 0
    for ql, L in zip(q_lens, seq_lens):
        ql, L = int(ql), int(L)
        prior = L - ql
        total += ql * prior + ql * (ql + 1) // 2
    return total


def prefill_flops(q_lens: Sequence[int], seq_lens: Sequence[int], num_q_heads: int, head_dim: int) -> int:
    return 4 * head_dim * num_q_heads * visible_pairs(q_lens, seq_lens)


def kv_write_bytes(total_new: int, num_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    return 2 * 2 * int(total_new) * num_kv_heads * head_dim * elem_bytes


def kv_write_rope_bytes(total_new: int, num_kv_heads: int, num_q_heads: int, head_dim: int,
                        elem_bytes: int = 2) -> int:
    """Fused writeback: K and V rows read and written, query rows read and
    written back in place (the norm weights, 2 x head_dim elements, are not counted)."""
    return kv_write_bytes(total_new, num_kv_heads, head_dim, elem_bytes) + \
        2 * int(total_new) * num_q_heads * head_dim * elem_bytes
