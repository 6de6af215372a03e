"""Algorithmic work of one call, for throughput and roofline figures.

These count the work the method must do, not what a kernel happens to
move: decode reads every cached K and V element of every request once;
extend does 4*D*Hq FLOP (two D-long dot products, multiply+add) per
causally valid (query, key) pair; store reads and writes each new row once.
"""
from __future__ import annotations

from .workloads import Workload


def decode_kv_bytes(w: Workload) -> int:
    """Algorithmic bytes of one decode call: every cached K and V element read once."""
    if w.decode is None:
        return 0
    return int(w.decode.seq_lens.sum().item()) * w.hkv * w.d * 2 * 2


def extend_flops(w: Workload) -> int:
    """Algorithmic FLOP of one extend call: 4*D*Hq per causally valid (query, key) pair."""
    if w.extend is None:
        return 0
    pre = w.extend.prefix_lens.long().cpu()
    ext = w.extend.ext_lens.long().cpu()
    pairs = int((ext * pre + ext * (ext + 1) // 2).sum().item())
    return 4 * w.d * w.hq * pairs


def store_bytes(w: Workload) -> int:
    """Algorithmic bytes of one store call: new K/V read + written, plus out_loc."""
    n = 0
    if w.extend is not None:
        n += w.extend.total_tokens
    if w.decode is not None:
        n += w.decode.num_reqs
    return n * w.hkv * w.d * 2 * 2 * 2 + 4 * n
