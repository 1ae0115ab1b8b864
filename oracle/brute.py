"""Pure-Python brute force for tiny inputs (no numpy in the arithmetic).

TEST INFRASTRUCTURE ONLY.  An independent second statement of what the
oracle computes, used to pin ``oracle.c``:

* storage bits are decoded with ``struct`` (binary16) or by widening to
  binary32 (bfloat16), not with the oracle's own bit routines;
* RoPE angles come straight from ``math.cos``/``math.sin`` of
  position * theta ** (-2 i / d) for the pair (i, i + d/2);
* keys and values are first placed into a dictionary "arena" keyed by
  (physical block, kv head, slot) through the block tables, then gathered
  back per sequence through the same tables (pages "Building Kshipra" part 3,
  section 1, fixed-size blocks reached through block tables);
* attention is the dense definition: scores q.k * scale for keys at
  positions <= the query's position (section 4, causal mask over the chunk),
  softmax with the row maximum subtracted, weighted sum of values.
"""

from __future__ import annotations

import math
import struct


def decode(bits: int, dtype: str) -> float:
    if dtype == "f16":
        return struct.unpack("<e", struct.pack("<H", bits))[0]
    return struct.unpack("<f", struct.pack("<I", bits << 16))[0]


def rotate(x, pos, theta):
    d = len(x)
    h = d // 2
    y = [0.0] * d
    for i in range(h):
        ang = pos * theta ** (-2.0 * i / d)
        c, s = math.cos(ang), math.sin(ang)
        y[i] = x[i] * c - x[i + h] * s
        y[i + h] = x[i + h] * c + x[i] * s
    return y


def attention(q, k_all, v_all, prefix_lens, query_lens, block_tables, block_size, num_kv_heads, theta, scale,
              dtype):
    """q: nested lists [T][Hq][d] of bits; k_all/v_all: [sum ctx][Hkv][d] bits.

    Returns nested lists [T][Hq][d] of floats.
    """
    S = len(prefix_lens)
    Hq = len(q[0]) if q else 0
    G = Hq // num_kv_heads
    # place every row into a dict arena through the block tables
    arena_k, arena_v = {}, {}
    row = 0
    for s in range(S):
        ctx = prefix_lens[s] + query_lens[s]
        for j in range(ctx):
            blk = block_tables[s][j // block_size]
            for h in range(num_kv_heads):
                arena_k[(blk, h, j % block_size)] = k_all[row][h]
                arena_v[(blk, h, j % block_size)] = v_all[row][h]
            row += 1
    out = []
    t = 0
    for s in range(S):
        ctx = prefix_lens[s] + query_lens[s]
        # gather back through the block tables
        keys = {}
        vals = {}
        for h in range(num_kv_heads):
            keys[h] = [rotate([decode(b, dtype) for b in arena_k[(block_tables[s][j // block_size], h,
                                                                   j % block_size)]], j, theta)
                       for j in range(ctx)]
            vals[h] = [[decode(b, dtype) for b in arena_v[(block_tables[s][j // block_size], h, j % block_size)]]
                       for j in range(ctx)]
        for i in range(query_lens[s]):
            pos = prefix_lens[s] + i
            heads = []
            for hq in range(Hq):
                g = hq // G
                qr = rotate([decode(b, dtype) for b in q[t][hq]], pos, theta)
                scores = []
                for j in range(pos + 1):
                    scores.append(scale * sum(a * b for a, b in zip(qr, keys[g][j])))
                m = max(scores)
                e = [math.exp(x - m) for x in scores]
                z = sum(e)
                d = len(qr)
                heads.append([sum(e[j] * vals[g][j][c] for j in range(pos + 1)) / z for c in range(d)])
            out.append(heads)
            t += 1
    return out
