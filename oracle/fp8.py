"""Reference definitions for an FP8 (e4m3) KV cache: the code table, the
quantising writeback and attention over the dequantised pages.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources
-------
* "The Stack Below the Stack, Part 2", closing recipe ("DP+EP + FP8 KV +
  chunked prefill"): the KV cache is stored in FP8.  The pages give no
  format details, so this module takes the plain reading:
* e4m3 as in the OCP 8-bit floating point specification (the format CUDA
  calls E4M3 / torch ``float8_e4m3fn``): 1 sign bit, 4 exponent bits with
  bias 7, 3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6;
  no infinities; the pattern S.1111.111 is NaN; the largest finite value is
  448;
* a K (or V) element x of KV head g is stored as the code nearest to
  ``x / scale[g]`` (round to nearest, ties to the even code, values beyond
  448 saturate to +-448), the quotient taken in float32 as the kernel
  takes it (a quantised code is an integer decision, so both sides make it
  in the same precision); it reads back as ``decode(code) * scale[g]``;
* attention then runs on the dequantised K/V exactly as in
  ``attention.paged_attention`` (float64, whole score row).

Readings where the pages are silent: one float32 scale per KV head for K and
one for V (a page is filled one token at a time by the eager writeback, so a
per-page scale would be fixed by its first token), and V stored transposed
inside each page block, ``[D][page_size]`` per (page, KV head), so that the
keys of one value column are contiguous.
"""

from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

from .attention import attention_rows, bf16_bits_to_f64

E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value (float64) of each e4m3 code (uint8)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


# magnitudes of the 127 finite non-negative codes, increasing with the code
_POS_VALUES = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code of each value (ties to the even code), saturating
    at +-448; NaN gives 0x7F.  ``x`` is taken as given (float32 or float64)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, 0x7E)  # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize(x_bits: np.ndarray, scale: float) -> np.ndarray:
    """Codes of bf16 values (given as bits) for one scale: encode(fp32(x) / fp32(scale))."""
    q = bf16_bits_to_f64(x_bits).astype(np.float32) / np.float32(scale)
    return e4m3_encode(q)


def kv_write_paged_fp8(k_pool: np.ndarray, v_pool_t: np.ndarray, k_new_bits: np.ndarray, v_new_bits: np.ndarray,
                       k_scale: Sequence[float], v_scale: Sequence[float], cu_seqlens_new: Sequence[int],
                       seq_lens: Sequence[int], block_table: np.ndarray, page_size: int
                       ) -> Tuple[np.ndarray, np.ndarray]:
    """Quantising writeback.  ``k_pool`` codes [P][Hkv][page_size][D];
    ``v_pool_t`` codes [P][Hkv][D][page_size] (V transposed per page block).
    New row i of sequence b goes to position seq_lens[b] - n_b + i, i.e. page
    block_table[b][pos // page_size], slot pos % page_size.  Returns copies."""
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool_t, copy=True)
    Hkv = kp.shape[1]
    for b in range(len(seq_lens)):
        t0, t1 = int(cu_seqlens_new[b]), int(cu_seqlens_new[b + 1])
        n = t1 - t0
        for i in range(n):
            pos = int(seq_lens[b]) - n + i
            phys = int(block_table[b][pos // page_size])
            slot = pos % page_size
            for g in range(Hkv):
                kp[phys, g, slot, :] = quantize(k_new_bits[t0 + i, g], k_scale[g])
                vp[phys, g, :, slot] = quantize(v_new_bits[t0 + i, g], v_scale[g])
    return kp, vp


def paged_attention_fp8(q_bits: np.ndarray, k_pool: np.ndarray, v_pool_t: np.ndarray, k_scale: Sequence[float],
                        v_scale: Sequence[float], block_table: np.ndarray, seq_lens: Sequence[int],
                        cu_seqlens_q: Sequence[int], num_q_heads: int, num_kv_heads: int, page_size: int,
                        scale: float, seqs: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Causal attention (bottom-right aligned) over the dequantised FP8 pages.

    Token j of sequence b, KV head g: K = decode(k_pool[phys][g][slot]) *
    k_scale[g], V = decode(v_pool_t[phys][g][:, slot]) * v_scale[g], with
    phys = block_table[b][j // page_size], slot = j % page_size.
    """
    total_q, Hq, D = q_bits.shape
    group = Hq // num_kv_heads
    out = np.full((total_q, Hq, D), np.nan)
    lse = np.full((total_q, Hq), np.nan)
    for b in (range(len(seq_lens)) if seqs is None else seqs):
        r0, r1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        L = int(seq_lens[b])
        q_len = r1 - r0
        positions = [L - q_len + i for i in range(q_len)]
        j = np.arange(L)
        phys = np.asarray(block_table[b], dtype=np.int64)[j // page_size]  # page of every token
        slot = j % page_size
        for g in range(num_kv_heads):
            K = e4m3_decode(k_pool[phys, g, slot, :]) * float(k_scale[g])    # [L][D]
            V = e4m3_decode(v_pool_t[phys, g, :, slot]) * float(v_scale[g])  # [L][D]
            for h in range(g * group, (g + 1) * group):
                o, l = attention_rows(bf16_bits_to_f64(q_bits[r0:r1, h, :]), K, V, positions, scale)
                out[r0:r1, h, :] = o
                lse[r0:r1, h] = l
    return out, lse


__all__ = ["E4M3_MAX", "e4m3_decode", "e4m3_encode", "quantize", "kv_write_paged_fp8", "paged_attention_fp8"]
