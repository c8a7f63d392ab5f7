"""Scalar pure-Python restatement of paged causal attention, for tiny inputs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

It exists to pin ``oracle.attention`` against a second, independently written
computation: nested loops, ``math.exp``, its own bf16 decoding through
``struct``, and a softmax that runs max, exponentiate, sum, normalise in four
separate passes ("The Stack Below the Stack, Part 2", section 2.1: the
ordinary softmax needs the whole row, first for its maximum, then for the sum
of exponentials).
"""

from __future__ import annotations

import math
import struct
from typing import List, Sequence, Tuple


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def attention(q_bits, k_pool_bits, v_pool_bits, block_table, seq_lens: Sequence[int],
              cu_seqlens_q: Sequence[int], num_q_heads: int, num_kv_heads: int, page_size: int,
              scale: float) -> Tuple[List, List]:
    """Returns nested lists out[t][h][d] and lse[t][h] (floats)."""
    total_q = len(q_bits)
    D = len(q_bits[0][0]) if total_q else 0
    kv_of = [h * num_kv_heads // num_q_heads for h in range(num_q_heads)]
    out = [[[0.0] * D for _ in range(num_q_heads)] for _ in range(total_q)]
    lse = [[-math.inf] * num_q_heads for _ in range(total_q)]
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        r0, r1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        for t in range(r0, r1):
            pos = L - (r1 - r0) + (t - r0)
            for h in range(num_q_heads):
                g = kv_of[h]
                qv = [_bf16(x) for x in q_bits[t][h]]
                scores = []
                for j in range(0, min(pos + 1, L)):
                    page = int(block_table[b][j // page_size])
                    krow = k_pool_bits[page][g][j % page_size]
                    acc = 0.0
                    for d in range(D):
                        acc += qv[d] * _bf16(krow[d])
                    scores.append(scale * acc)
                if not scores:
                    continue
                mx = scores[0]
                for s in scores:
                    if s > mx:
                        mx = s
                w = [math.exp(s - mx) for s in scores]
                tot = 0.0
                for x in w:
                    tot += x
                for d in range(D):
                    acc = 0.0
                    for j in range(len(w)):
                        page = int(block_table[b][j // page_size])
                        acc += w[j] * _bf16(v_pool_bits[page][g][j % page_size][d])
                    out[t][h][d] = acc / tot
                lse[t][h] = mx + math.log(tot)
    return out, lse
