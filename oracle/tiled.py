"""CPU model of tiled online softmax and of the split-KV log-sum-exp combine.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

This restates, in float64 and in the pages' order, the two identities the
CUDA kernels rely on, so that tests can check them against the materialised
definition in ``oracle.attention``:

* Online softmax ("The Stack Below the Stack, Part 2", section 2.1; "8.
  Kernels and Attention Backends", section "Attention is an I/O problem"):
  walk the scores one tile at a time carrying the largest score seen so far
  and the running sum of exponentials; when a tile raises the maximum,
  rescale the running sum (and the running weighted sum of values) by
  exp(old max - new max).  After the last tile the result equals the
  untiled softmax.
* Flash-Decoding (same page, section 2.2): split the keys into C chunks;
  each chunk yields its normalised partial output and its local log-sum-exp;
  the global log-sum-exp is log(sum_c exp(lse_c)) and the output is
  sum_c exp(lse_c - lse) * o_c.  A chunk that saw no key has lse_c = -inf
  and weight 0.
"""

from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np


def online_softmax_chunk(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float,
                         tile_sizes: Sequence[int]) -> Tuple[np.ndarray, float, float]:
    """Stream one chunk of keys tile by tile.

    Returns the running state after the last tile: (acc, m, l) with
    acc = sum_j exp(s_j - m) v_j (unnormalised), m = max_j s_j,
    l = sum_j exp(s_j - m).  An empty chunk returns (0, -inf, 0).
    """
    D = values.shape[1]
    acc = np.zeros(D)
    m = -math.inf
    l = 0.0
    start = 0
    ti = 0
    n = keys.shape[0]
    while start < n:
        size = max(1, int(tile_sizes[ti % len(tile_sizes)]))
        ti += 1
        stop = min(n, start + size)
        s = scale * (keys[start:stop] @ q)
        m_new = max(m, float(s.max()))
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        p = np.exp(s - m_new)
        l = l * alpha + float(p.sum())
        acc = acc * alpha + p @ values[start:stop]
        m = m_new
        start = stop
    return acc, m, l


def chunk_partial(q, keys, values, scale, tile_sizes) -> Tuple[np.ndarray, float]:
    """Normalised partial output o_c and local log-sum-exp lse_c of a chunk."""
    acc, m, l = online_softmax_chunk(q, keys, values, scale, tile_sizes)
    if l == 0.0:
        return np.zeros(values.shape[1]), -math.inf
    return acc / l, m + math.log(l)


def combine(partials: List[Tuple[np.ndarray, float]]) -> Tuple[np.ndarray, float]:
    """Merge chunk partials with the log-sum-exp identity."""
    lses = [lse for _, lse in partials if lse != -math.inf]
    if not lses:
        D = partials[0][0].shape[0] if partials else 0
        return np.zeros(D), -math.inf
    m = max(lses)
    total = sum(math.exp(x - m) for x in lses)
    lse = m + math.log(total)
    out = np.zeros_like(partials[0][0])
    for o_c, lse_c in partials:
        if lse_c == -math.inf:
            continue
        out = out + math.exp(lse_c - lse) * o_c
    return out, lse


def split_decode(q, keys, values, scale, chunk_bounds: Sequence[int], tile_sizes) -> Tuple[np.ndarray, float]:
    """Decode one query row by Flash-Decoding: chunks [b_i, b_{i+1}) of the
    keys, each streamed with ``online_softmax_chunk``, merged by ``combine``."""
    parts = []
    for c0, c1 in zip(chunk_bounds[:-1], chunk_bounds[1:]):
        parts.append(chunk_partial(q, keys[c0:c1], values[c0:c1], scale, tile_sizes))
    return combine(parts)
