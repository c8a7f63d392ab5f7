"""Reference definitions (numpy, float64) for the rotary position embedding
and RMS normalisation fused into the K/V writeback.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources
-------
* "The Stack Below the Stack, Part 2", section 2.1 (kernel fusion): serving
  stacks fuse the normalisation of K (and Q), the rotary embedding and the
  KV-cache insertion into one kernel ("Fused Q-norm, KV-RoPE, and K-insert"),
  so the rotated K row is produced and written into its page in one pass.
  The pages name the fusion but do not restate the two operations, so this
  module writes out their standard definitions:
* rotary position embedding (RoFormer, Su et al. 2021), in the "rotate-half"
  pairing used by Llama- and Qwen-family models: dimension ``i`` (``i <
  D/2``) is paired with ``i + D/2``; the pair is rotated by the angle
  ``pos * base ** (-2 i / D)``;
* RMS normalisation (Zhang and Sennrich 2019): ``x / sqrt(mean(x**2) + eps)
  * weight``, applied per head before the rotation (as in models with
  per-head Q/K norms).

Readings where the pages are silent: the
rotate-half pairing, the frequency base as a parameter, normalisation before
rotation, and the row position ``seq_len - n_new + i`` (the slot the row is
written to) as the rotation position.
"""

from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

from .attention import bf16_bits_to_f64


def rms_norm(x: np.ndarray, weight: Optional[np.ndarray], eps: float) -> np.ndarray:
    """Normalise the last axis by its root mean square, then scale by ``weight``."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    y = x / np.sqrt(ms + eps)
    if weight is not None:
        y = y * np.asarray(weight, dtype=np.float64)
    return y


def rope_angles(pos: int, head_dim: int, base: float) -> np.ndarray:
    """Rotation angle of each of the D/2 pairs at position ``pos``."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return float(pos) * np.power(float(base), -2.0 * i / head_dim)


def rope_rotate_half(x: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotate pair (x[i], x[i + D/2]) by the angle of pair i, for every i < D/2.

    ``x`` is [..., D]; the same position applies to every leading index.
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    a = rope_angles(pos, D, base)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_writeback_rows(k_new_bits: np.ndarray, q_bits: Optional[np.ndarray], cu_seqlens_new: Sequence[int],
                        seq_lens: Sequence[int], base: float, k_norm_weight_bits: Optional[np.ndarray] = None,
                        q_norm_weight_bits: Optional[np.ndarray] = None, eps: float = 1e-6
                        ) -> Tuple[np.ndarray, Optional[np.ndarray], np.ndarray]:
    """The K rows (and Q rows) the fused writeback produces, before bf16 rounding.

    New row ``i`` of sequence ``b`` (``n_b`` new rows) sits at position
    ``seq_lens[b] - n_b + i``; its K heads (and Q heads) are RMS-normalised
    when a weight is given, then rotated at that position.  V rows are
    written unchanged (see ``attention.kv_write_paged`` for where every row
    goes).  Returns (k_rows [T][Hkv][D], q_rows [T][Hq][D] or None,
    positions [T]) in float64.
    """
    k = bf16_bits_to_f64(k_new_bits)
    q = None if q_bits is None else bf16_bits_to_f64(q_bits)
    kw = None if k_norm_weight_bits is None else bf16_bits_to_f64(k_norm_weight_bits)
    qw = None if q_norm_weight_bits is None else bf16_bits_to_f64(q_norm_weight_bits)
    T = k.shape[0]
    k_out = np.full(k.shape, np.nan)
    q_out = None if q is None else np.full(q.shape, np.nan)
    positions = np.full(T, -1, dtype=np.int64)
    for b in range(len(seq_lens)):
        t0, t1 = int(cu_seqlens_new[b]), int(cu_seqlens_new[b + 1])
        n = t1 - t0
        for i in range(n):
            t = t0 + i
            pos = int(seq_lens[b]) - n + i
            positions[t] = pos
            kr = rms_norm(k[t], kw, eps) if kw is not None else k[t]
            k_out[t] = rope_rotate_half(kr, pos, base)
            if q is not None:
                qr = rms_norm(q[t], qw, eps) if qw is not None else q[t]
                q_out[t] = rope_rotate_half(qr, pos, base)
    return k_out, q_out, positions


def round_to_bf16_f64(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), returned as float64.

    Two steps: float64 -> float32 (round to nearest even), then keep the top
    16 bits of the float32 pattern with round-to-nearest-even on the dropped
    16 bits.  The double rounding can differ from a direct float64 -> bf16
    rounding only when the float32 value lands exactly on a bf16 tie, which
    the tests treat as a one-ulp tolerance.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 7), 2.0 ** -133)


__all__ = ["rms_norm", "rope_angles", "rope_rotate_half", "rope_writeback_rows", "round_to_bf16_f64", "bf16_ulp"]
