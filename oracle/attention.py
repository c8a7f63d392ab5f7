"""Reference definitions (numpy, float64) for paged-KV attention.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources
-------
* "8. Kernels and Attention Backends", section "Attention is an I/O
  problem": attention builds the query-key score matrix, applies a softmax
  and multiplies by the values; serving attention is ragged and its KV state
  may be paged.  This module is that plain computation: every score of a row
  is materialised at once, the softmax subtracts the row maximum (the
  stabilisation described in "The Stack Below the Stack, Part 2", section 2.1)
  and no tiling is used.
* "Inside Ion" (section "IonAttention in One Paragraph") and "8. Kernels and
  Attention Backends" (section "Kernels and Attention Backends" intro: KV
  blocks scattered through memory): K/V live in fixed-size pages reached
  through a per-sequence table of page ids; new K/V rows are written into
  their pages eagerly.

Readings where the pages are silent:

* pools are ``[num_pages][Hkv][page_size][D]``; query head ``h`` reads KV
  head ``h // (Hq // Hkv)``;
* query row ``i`` of a sequence with ``q_len`` new rows and ``seq_len`` total
  keys sits at absolute position ``seq_len - q_len + i`` and sees keys
  ``0 .. seq_len - q_len + i`` (bottom-right causal alignment; with
  ``q_len = 1`` this is ordinary decode);
* a row that sees no key (an empty sequence) has output 0 and lse = -inf,
  a defined value rather than NaN ("8. Kernels ...", section "Test the
  kernel at three levels": a fully masked row must give a defined result);
* ``lse`` is the natural-log log-sum-exp of the scaled scores.
"""

from __future__ import annotations

import math
from typing import Optional, Sequence, Tuple

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 numbers given as their uint16 bit patterns.

    A bf16 number is the upper half of an IEEE binary32 number; shifting the
    pattern into the top 16 bits of a uint32 and reading it as float32 gives
    the value exactly, and float32 -> float64 is exact.
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def gather_kv_rows(pool_bits: np.ndarray, table_row: np.ndarray, n_tokens: int, kv_head: int,
                   page_size: int) -> np.ndarray:
    """Logical K (or V) rows 0..n_tokens-1 of one sequence and KV head.

    Token ``j`` lives in physical page ``table_row[j // page_size]`` at slot
    ``j % page_size``; the loop visits tokens one by one, exactly as the
    definition reads.  Returns float64 ``[n_tokens][D]``.
    """
    D = pool_bits.shape[-1]
    out = np.empty((n_tokens, D), dtype=np.float64)
    for j in range(n_tokens):
        phys = int(table_row[j // page_size])
        slot = j % page_size
        out[j] = bf16_bits_to_f64(pool_bits[phys, kv_head, slot])
    return out


def attention_rows(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, positions: Sequence[int],
                   scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Materialised-score causal attention for a few query rows of one head.

    ``q_rows`` [R][D], ``keys``/``values`` [n][D] (float64), ``positions[r]``
    = absolute position of row r: it sees keys 0..positions[r].
    Returns (o [R][D], lse [R]).
    """
    R = q_rows.shape[0]
    D = values.shape[1] if values.ndim == 2 else q_rows.shape[1]
    o = np.zeros((R, D), dtype=np.float64)
    lse = np.full((R,), -np.inf, dtype=np.float64)
    for r in range(R):
        n_vis = min(int(positions[r]) + 1, keys.shape[0])
        if n_vis <= 0:
            continue  # no visible key: o = 0, lse = -inf
        s = scale * (keys[:n_vis] @ q_rows[r])  # all scores of the row at once
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        o[r] = (e @ values[:n_vis]) / l
        lse[r] = m + math.log(l)
    return o, lse


def paged_attention(q_bits: np.ndarray, k_pool_bits: np.ndarray, v_pool_bits: np.ndarray,
                    block_table: np.ndarray, seq_lens: Sequence[int], cu_seqlens_q: Sequence[int],
                    num_q_heads: int, num_kv_heads: int, page_size: int, scale: float,
                    seqs: Optional[Sequence[int]] = None, heads: Optional[Sequence[int]] = None,
                    ) -> Tuple[np.ndarray, np.ndarray]:
    """Causal attention of every query row against its sequence's paged K/V.

    ``q_bits`` bf16 bits [total_q][Hq][D]; pools bf16 bits [P][Hkv][ps][D];
    ``block_table`` int [B][max_pages]; ``seq_lens`` [B] total keys per
    sequence (including the query rows' own); ``cu_seqlens_q`` [B+1].
    ``seqs``/``heads`` restrict the work to a subset (other rows stay NaN).
    Returns float64 (out [total_q][Hq][D], lse [total_q][Hq]).
    """
    total_q, Hq, D = q_bits.shape
    assert Hq == num_q_heads and Hq % num_kv_heads == 0
    group = Hq // num_kv_heads
    out = np.full((total_q, Hq, D), np.nan)
    lse = np.full((total_q, Hq), np.nan)
    B = len(seq_lens)
    seqs = range(B) if seqs is None else seqs
    heads = range(Hq) if heads is None else heads
    for b in seqs:
        r0, r1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        L = int(seq_lens[b])
        q_len = r1 - r0
        positions = [L - q_len + i for i in range(q_len)]
        by_kv = {}
        for h in heads:
            g = h // group
            if g not in by_kv:
                by_kv[g] = (gather_kv_rows(k_pool_bits, block_table[b], L, g, page_size),
                            gather_kv_rows(v_pool_bits, block_table[b], L, g, page_size))
            K, V = by_kv[g]
            qr = bf16_bits_to_f64(q_bits[r0:r1, h, :])
            o, l = attention_rows(qr, K, V, positions, scale)
            out[r0:r1, h, :] = o
            lse[r0:r1, h] = l
    return out, lse


def kv_write_paged(k_pool_bits: np.ndarray, v_pool_bits: np.ndarray, k_new_bits: np.ndarray,
                   v_new_bits: np.ndarray, cu_seqlens_new: Sequence[int], seq_lens: Sequence[int],
                   block_table: np.ndarray, page_size: int) -> Tuple[np.ndarray, np.ndarray]:
    """Eager K/V writeback: copy each new row into its page slot.

    New row ``i`` of sequence ``b`` (``n_b`` new rows, ``seq_lens[b]`` keys
    after the write) is at position ``seq_lens[b] - n_b + i``, so it goes to
    page ``block_table[b][pos // page_size]``, slot ``pos % page_size``, for
    every KV head.  Returns new pools (copies); a pure bit copy, so the result
    must match the GPU bit for bit, untouched bytes included.
    """
    kp = np.array(k_pool_bits, copy=True)
    vp = np.array(v_pool_bits, copy=True)
    for b in range(len(seq_lens)):
        t0, t1 = int(cu_seqlens_new[b]), int(cu_seqlens_new[b + 1])
        n = t1 - t0
        for i in range(n):
            pos = int(seq_lens[b]) - n + i
            phys = int(block_table[b][pos // page_size])
            slot = pos % page_size
            kp[phys, :, slot, :] = k_new_bits[t0 + i]
            vp[phys, :, slot, :] = v_new_bits[t0 + i]
    return kp, vp
