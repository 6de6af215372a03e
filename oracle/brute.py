"""Pure-Python brute force for tiny paged-attention cases (test infrastructure).

A second, independent spelling of the oracle's definition, with Python lists
and ``math.exp``, used on inputs of a few keys and a few dims to cross-check
the C oracle's indexing, marshalling and threading.  It walks the request's
pages one by one (instead of computing slot = page*ps + offset per key), so
an indexing slip on either side shows up as a mismatch.  It shares no code
with the C oracle or the CUDA library.
"""
from __future__ import annotations

import math
import struct


def bf16_bits_to_float(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def attention_row(q_row, k_pool, v_pool, page_size, pages, pos, head, hq, hkv, scale):
    """q_row: [Hq][D] floats; pools: [S][Hkv][D] floats; pages: page ids of the request.

    Returns (o: list[float] of length D, lse: float) for keys 0..pos.
    """
    group = hq // hkv
    g = head // group
    keys, vals = [], []
    for page in pages:
        for off in range(page_size):
            if len(keys) == pos + 1:
                break
            slot = page * page_size + off
            keys.append(k_pool[slot][g])
            vals.append(v_pool[slot][g])
    assert len(keys) == pos + 1, "page table too short for this position"
    q = q_row[head]
    scores = [scale * sum(a * b for a, b in zip(q, k)) for k in keys]
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    z = math.fsum(w)
    d = len(q)
    o = [math.fsum(w[j] * vals[j][x] for j in range(len(vals))) / z for x in range(d)]
    return o, m + math.log(z)
