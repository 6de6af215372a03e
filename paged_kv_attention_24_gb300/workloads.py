"""Seeded synthetic inputs for paged-KV attention.

This module serves both the CUDA library's tests/bench and the CPU oracle,
so it holds none of the method's arithmetic: it draws lengths, allocates
pages, fills the pool with N(0,1) bf16 values (unused slots hold NaN, so a
stray read poisons the result) and lays out the metadata.  Attention itself
is computed elsewhere (kernels on one side, the oracle on the other).

The shapes follow the pages' workloads: the offline benchmark of
"Mini-SGLang 实战指南" §9.1 (256 requests, input and output lengths drawn
uniformly from 100-1024 tokens, Qwen3-0.6B / Qwen3-14B) and the Qwen3-32B
online setup of §9.2, with the head shapes of those models (0.6B: 16 q
heads / 8 kv heads; 14B: 40/8; 32B: 64/8; head_dim 128).  The Qwen trace
itself is not available, so seeded uniform lengths stand in for it.

Layout of a pool: K and V are separate bf16 tensors [num_slots, Hkv, D];
slot = page_id * page_size + offset.  Page tables are int32 [B, W] of page
ids; entries past a request's last page hold -1 and are never read.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0


@dataclasses.dataclass
class DecodeBatch:
    q: torch.Tensor            # bf16 [B, Hq, D]
    seq_lens: torch.Tensor     # int32 [B]   (includes the current token)
    page_table: torch.Tensor   # int32 [B, W] page ids
    new_loc: torch.Tensor      # int32 [B]   slot of each request's current token
    max_seq_len: int

    @property
    def num_reqs(self) -> int:
        return int(self.q.shape[0])


@dataclasses.dataclass
class ExtendBatch:
    q: torch.Tensor            # bf16 [T, Hq, D], request-major
    prefix_lens: torch.Tensor  # int32 [B]  cached tokens before the chunk
    ext_lens: torch.Tensor     # int32 [B]  tokens in the chunk
    cu_ext: torch.Tensor       # int32 [B+1]
    positions: torch.Tensor    # int32 [T]  absolute position of each chunk token
    page_table: torch.Tensor   # int32 [B, W]
    out_loc: torch.Tensor      # int32 [T]  slot of each chunk token
    max_ext_len: int
    max_seq_len: int

    @property
    def num_reqs(self) -> int:
        return int(self.prefix_lens.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])


@dataclasses.dataclass
class Workload:
    name: str
    hq: int
    hkv: int
    d: int
    page_size: int
    scale: float
    k_pool: torch.Tensor       # bf16 [S, Hkv, D]
    v_pool: torch.Tensor
    decode: Optional[DecodeBatch] = None
    extend: Optional[ExtendBatch] = None
    seed: int = 0

    @property
    def num_slots(self) -> int:
        return int(self.k_pool.shape[0])

    def new_tokens(self):
        """(k_new, v_new, out_loc) for every token this step stores: chunk tokens, then decode tokens."""
        locs = []
        if self.extend is not None:
            locs.append(self.extend.out_loc)
        if self.decode is not None:
            locs.append(self.decode.new_loc)
        loc = torch.cat(locs) if locs else torch.zeros(0, dtype=torch.int32, device=self.k_pool.device)
        idx = loc.long()
        return self.k_pool[idx].contiguous(), self.v_pool[idx].contiguous(), loc.contiguous()

    def to(self, device) -> "Workload":
        def mv(x):
            return x.to(device) if isinstance(x, torch.Tensor) else x
        dec = None if self.decode is None else DecodeBatch(
            **{f.name: mv(getattr(self.decode, f.name)) for f in dataclasses.fields(DecodeBatch)})
        ext = None if self.extend is None else ExtendBatch(
            **{f.name: mv(getattr(self.extend, f.name)) for f in dataclasses.fields(ExtendBatch)})
        return dataclasses.replace(self, k_pool=mv(self.k_pool), v_pool=mv(self.v_pool),
                                   decode=dec, extend=ext)


class PageAllocator:
    """Hands out page ids in a seeded random order (so slots are scattered)."""

    def __init__(self, num_pages: int, rng: np.random.Generator):
        self.order = rng.permutation(num_pages).astype(np.int64)
        self.next = 0

    def take(self, n: int) -> np.ndarray:
        if self.next + n > self.order.shape[0]:
            raise ValueError("KV pool too small for the requested sequences")
        out = self.order[self.next:self.next + n]
        self.next += n
        return out


def _pages(n_tokens: int, ps: int) -> int:
    return (n_tokens + ps - 1) // ps


def make_workload(name: str, hq: int, hkv: int, d: int, page_size: int, seed: int,
                  decode_seq_lens=None, extend_prefix_lens=None, extend_ext_lens=None,
                  shared_prefix_len: int = 0, num_slots: Optional[int] = None,
                  device="cpu", value_dist: str = "normal") -> Workload:
    """Build a pool plus optional decode and extend batches.

    ``shared_prefix_len`` > 0 makes every extend request's prefix the same
    page ids (a radix-cache hit shared by all of them); it must be a multiple
    of the page size and equal each extend_prefix_lens entry.
    """
    rng = np.random.default_rng(seed)
    ps = int(page_size)
    dec_seq = None if decode_seq_lens is None else np.asarray(decode_seq_lens, dtype=np.int64)
    pre = None if extend_prefix_lens is None else np.asarray(extend_prefix_lens, dtype=np.int64)
    ext = None if extend_ext_lens is None else np.asarray(extend_ext_lens, dtype=np.int64)

    pages_needed = 0
    if dec_seq is not None:
        pages_needed += int(sum(_pages(int(s), ps) for s in dec_seq))
    if ext is not None:
        if shared_prefix_len:
            assert shared_prefix_len % ps == 0 and np.all(pre == shared_prefix_len)
            pages_needed += shared_prefix_len // ps
            pages_needed += int(sum(_pages(int(e), ps) for e in ext))
        else:
            pages_needed += int(sum(_pages(int(p + e), ps) for p, e in zip(pre, ext)))
    if num_slots is None:
        num_slots = max(4096, int(math.ceil(pages_needed * ps / 4096)) * 4096)
    num_pages = num_slots // ps
    assert num_pages * ps == num_slots, "pool size must be a whole number of pages"
    alloc = PageAllocator(num_pages, rng)
    used = np.zeros(num_slots, dtype=bool)

    def mark(page_ids: np.ndarray, n_tokens: int):
        pos = np.arange(n_tokens)
        used[page_ids[pos // ps] * ps + pos % ps] = True

    def slots_of(page_ids: np.ndarray, positions: np.ndarray) -> np.ndarray:
        return page_ids[positions // ps] * ps + positions % ps

    # --- decode requests
    dec_tables = []
    if dec_seq is not None:
        for s in dec_seq:
            pg = alloc.take(_pages(int(s), ps))
            mark(pg, int(s))
            dec_tables.append(pg)
    # --- extend requests
    ext_tables = []
    if ext is not None:
        shared = alloc.take(shared_prefix_len // ps) if shared_prefix_len else None
        if shared is not None:
            mark(shared, shared_prefix_len)
        for p, e in zip(pre, ext):
            if shared is not None:
                own = alloc.take(_pages(int(e), ps))
                mark(own, int(e))
                pg = np.concatenate([shared, own])
            else:
                pg = alloc.take(_pages(int(p + e), ps))
                mark(pg, int(p + e))
            ext_tables.append(pg)

    gen = torch.Generator(device=device).manual_seed(seed)

    def randn(*shape):
        if value_dist == "normal":
            x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
        elif value_dist == "uniform":
            x = torch.rand(*shape, generator=gen, device=device, dtype=torch.float32) * 2 - 1
        else:
            raise ValueError(value_dist)
        return x.to(torch.bfloat16)

    k_pool = randn(num_slots, hkv, d)
    v_pool = randn(num_slots, hkv, d)
    unused = torch.from_numpy(~used).to(device)
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=device)
    k_pool[unused] = nan
    v_pool[unused] = nan

    def table(rows):
        w = max(1, max(len(r) for r in rows))
        t = np.full((len(rows), w), -1, dtype=np.int32)
        for i, r in enumerate(rows):
            t[i, :len(r)] = r
        return torch.from_numpy(t).to(device)

    decode = None
    if dec_seq is not None:
        B = len(dec_seq)
        new_loc = np.array([slots_of(dec_tables[i], np.array([dec_seq[i] - 1]))[0] for i in range(B)],
                           dtype=np.int32)
        decode = DecodeBatch(
            q=randn(B, hq, d),
            seq_lens=torch.tensor(dec_seq, dtype=torch.int32, device=device),
            page_table=table(dec_tables) if B else torch.zeros((0, 1), dtype=torch.int32, device=device),
            new_loc=torch.from_numpy(new_loc).to(device),
            max_seq_len=int(dec_seq.max()) if B else 0)
    extend = None
    if ext is not None:
        B = len(ext)
        T = int(ext.sum())
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(ext)
        positions = np.concatenate([np.arange(p, p + e) for p, e in zip(pre, ext)]).astype(np.int32) \
            if T else np.zeros(0, dtype=np.int32)
        out_loc = np.concatenate([slots_of(ext_tables[i], np.arange(pre[i], pre[i] + ext[i]))
                                  for i in range(B)]).astype(np.int32) if T else np.zeros(0, np.int32)
        extend = ExtendBatch(
            q=randn(T, hq, d),
            prefix_lens=torch.tensor(pre, dtype=torch.int32, device=device),
            ext_lens=torch.tensor(ext, dtype=torch.int32, device=device),
            cu_ext=torch.from_numpy(cu).to(device),
            positions=torch.from_numpy(positions).to(device),
            page_table=table(ext_tables),
            out_loc=torch.from_numpy(out_loc).to(device),
            max_ext_len=int(ext.max()) if B else 0,
            max_seq_len=int((pre + ext).max()) if B else 0)
    return Workload(name=name, hq=hq, hkv=hkv, d=d, page_size=ps, scale=1.0 / math.sqrt(d),
                    k_pool=k_pool, v_pool=v_pool, decode=decode, extend=extend, seed=seed)


# ------------------------------------------------------------- the configs

CONFIG_NAMES = {
    1: "decode-tiny-qwen3-0.6b-b4-ps1",
    2: "extend-radix-qwen3-0.6b-b8-ps1",
    3: "decode-offline-qwen3-0.6b-b256-ps1",
    4: "mixed-qwen3-14b-decode-b128-extend-8192-over-4096-ps16",
    5: "mixed-qwen3-32b-extend-8x1024-shared-2048-decode-b64-ps64",
}


def config(i: int, device="cpu", seed: Optional[int] = None, part: str = "all",
           page_size: Optional[int] = None) -> Workload:
    """The five workloads (seed defaults to 1000 + i).

    ``part`` = "decode" / "extend" keeps only that batch of a mixed config;
    ``page_size`` overrides the config's page size (same lengths and seeds).
    """
    seed = 1000 + i if seed is None else seed
    rng = np.random.default_rng(seed + 7919)  # lengths; pool layout uses ``seed``
    dec = pre = ext = None
    shared = 0
    ps = 1
    num_slots = None
    if i == 1:
        hq, hkv = 16, 8
        dec = rng.integers(17, 200, size=4, endpoint=True)
        num_slots = 4096
    elif i == 2:
        hq, hkv = 16, 8
        pre = rng.integers(0, 1024, size=8, endpoint=True)
        ext = rng.integers(100, 1024, size=8, endpoint=True)
        assert ext.sum() <= 8192
    elif i == 3:
        hq, hkv = 16, 8
        dec = rng.integers(100, 1024, size=256, endpoint=True) + rng.integers(0, 1024, size=256, endpoint=True)
    elif i == 4:
        hq, hkv, ps = 40, 8, 16
        dec = rng.integers(512, 4096, size=128, endpoint=True)
        pre, ext = np.array([4096]), np.array([8192])
    elif i == 5:
        hq, hkv, ps = 64, 8, 64
        dec = rng.integers(1024, 8192, size=64, endpoint=True)
        pre, ext = np.full(8, 2048), np.full(8, 1024)
        shared = 2048
    else:
        raise ValueError(f"no config {i}")
    if page_size is not None:
        ps = int(page_size)
        if shared and shared % ps:
            raise ValueError("the shared prefix must be a whole number of pages")
        if num_slots is not None and num_slots % ps:
            num_slots = None
    if part == "decode":
        pre = ext = None
        shared = 0
    elif part == "extend":
        dec = None
    name = CONFIG_NAMES[i] + ("" if part == "all" else f"-{part}")
    if page_size is not None:
        name += f"-page{ps}"
    return make_workload(name, hq, hkv, 128, ps,
                         seed, decode_seq_lens=dec, extend_prefix_lens=pre, extend_ext_lens=ext,
                         shared_prefix_len=shared, num_slots=num_slots, device=device)
