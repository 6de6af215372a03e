"""Host radix prefix cache (libmsgl_attn, include/msgl_radix.h) — CPU only.

* unit cases: matching, partial pages, duplicates, pins, LRU eviction, leases;
* a randomized comparison with a small Python model of the same rules
  (page-aligned chunks, LIFO free list, eviction by (stamp, page id));
* an end-to-end check: page tables built by the cache for requests that
  share prefixes give the same attention (fp64 oracle) as private pages.
"""
import math
import random

import numpy as np
import pytest
import torch

from paged_kv_attention_24_gb300 import build as cuda_build
from paged_kv_attention_24_gb300.radix import RadixCache, RadixError


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cuda_build.build()


def test_match_insert_and_reuse():
    c = RadixCache(page_size=4, num_pages=16)
    toks = list(range(10))                         # 2 full pages + 2 tokens
    n, pages, lease = c.match(toks)
    assert n == 0 and len(pages) == 0
    own = c.alloc(3)
    assert c.insert(toks, own, lease) == 2         # the partial page is not cached
    assert c.stats() == {"free": 14, "cached": 2, "pinned": 0}
    n, pages, lease2 = c.match(toks + [99, 98])
    assert n == 8 and list(pages) == list(own[:2])
    assert c.stats()["pinned"] == 2
    c.release(lease2, [])
    assert c.stats()["pinned"] == 0
    n, pages, lease3 = c.match([0, 1, 2, 3, 7, 7, 7, 7])   # diverges in the second page
    assert n == 4 and list(pages) == [own[0]]
    c.release(lease3, [])


def test_duplicate_pages_are_freed():
    c = RadixCache(page_size=2, num_pages=8)
    toks = [5, 6, 7, 8]
    _, _, l1 = c.match(toks)
    p1 = c.alloc(2)
    _, _, l2 = c.match(toks)                       # a second request computed the same prefix
    p2 = c.alloc(2)
    assert c.insert(toks, p1, l1) == 2
    assert c.insert(toks, p2, l2) == 0             # already cached: p2 returns to the free list
    assert c.stats() == {"free": 6, "cached": 2, "pinned": 0}


def test_pinned_pages_survive_eviction_and_lru_order():
    c = RadixCache(page_size=1, num_pages=4)
    for t in ([1], [2], [3]):
        _, _, l = c.match(t)
        c.insert(t, c.alloc(1), l)                 # three cached single-page prefixes
    n, pin_pages, lease = c.match([1])             # [1] is now pinned and most recent
    assert n == 1
    got = c.alloc(3)                               # 1 free page + evicts [2] then [3] (oldest first)
    assert len(got) == 3
    assert c.stats() == {"free": 0, "cached": 1, "pinned": 1}
    with pytest.raises(RadixError):
        c.alloc(1)                                 # only the pinned page is left
    assert c.match([2])[0] == 0 and c.match([3])[0] == 0
    c.release(lease, [])
    assert len(c.alloc(1)) == 1                    # now [1] can be evicted


def test_errors():
    c = RadixCache(page_size=2, num_pages=4)
    with pytest.raises(RadixError):
        c.insert([1, 2], [0], 12345)               # unknown lease
    _, _, l = c.match([1, 2])
    with pytest.raises(RadixError):
        c.insert([1, 2], [7], l)                   # page id outside the pool
    c.release(l, [])
    with pytest.raises(RadixError):
        c.release(l, [])                           # lease already ended
    with pytest.raises(RadixError):
        RadixCache(0, 4)


class Model:
    """The cache's rules, restated in Python for the randomized comparison."""

    def __init__(self, ps, n):
        self.ps, self.n = ps, n
        self.free = list(range(n - 1, -1, -1))
        self.state = ["free"] * n
        self.root = {"children": {}, "page": -1, "pins": 0, "stamp": 0, "parent": None}
        self.clock, self.next_lease, self.leases = 0, 1, {}

    def chunks(self, toks):
        return [tuple(toks[i * self.ps:(i + 1) * self.ps]) for i in range(len(toks) // self.ps)]

    def match(self, toks):
        self.clock += 1
        cur, path = self.root, []
        for ch in self.chunks(toks):
            if ch not in cur["children"]:
                break
            cur = cur["children"][ch]
            cur["stamp"] = self.clock
            path.append(cur)
        for nd in path:
            nd["pins"] += 1
        lid = self.next_lease
        self.next_lease += 1
        self.leases[lid] = path
        return len(path) * self.ps, [nd["page"] for nd in path], lid

    def leaves(self):
        out = []

        def walk(nd):
            for ch in nd["children"].values():
                walk(ch)
            if nd is not self.root and not nd["children"] and nd["pins"] == 0:
                out.append(nd)
        walk(self.root)
        return out

    def alloc(self, k):
        while len(self.free) < k:
            cand = self.leaves()
            if not cand:
                return None
            nd = min(cand, key=lambda x: (x["stamp"], x["page"]))
            par = nd["parent"]
            del par["children"][nd["key"]]
            self.state[nd["page"]] = "free"
            self.free.append(nd["page"])
        out = [self.free.pop() for _ in range(k)]
        for p in out:
            self.state[p] = "held"
        return out

    def end(self, lid):
        for nd in self.leases.pop(lid):
            nd["pins"] -= 1

    def insert(self, toks, pages, lid):
        self.clock += 1
        ps = self.ps
        npg = -(-len(toks) // ps)
        cur, added = self.root, 0
        for i in range(npg):
            p = pages[i]
            if (i + 1) * ps > len(toks):
                if self.state[p] == "held":
                    self.state[p] = "free"; self.free.append(p)
                continue
            ch = tuple(toks[i * ps:(i + 1) * ps])
            if ch in cur["children"]:
                nd = cur["children"][ch]
                if nd["page"] != p and self.state[p] == "held":
                    self.state[p] = "free"; self.free.append(p)
                nd["stamp"] = self.clock
                cur = nd
                continue
            nd = {"children": {}, "page": p, "pins": 0, "stamp": self.clock, "parent": cur, "key": ch}
            cur["children"][ch] = nd
            self.state[p] = "cached"
            cur = nd
            added += 1
        self.end(lid)
        return added

    def release(self, lid, pages):
        self.end(lid)
        for p in pages:
            if self.state[p] == "held":
                self.state[p] = "free"; self.free.append(p)

    def stats(self):
        cached = sum(1 for s in self.state if s == "cached")
        pinned = 0

        def walk(nd):
            nonlocal pinned
            for ch in nd["children"].values():
                pinned += ch["pins"] > 0
                walk(ch)
        walk(self.root)
        return {"free": len(self.free), "cached": cached, "pinned": pinned}


@pytest.mark.parametrize("seed", range(6))
def test_random_ops_match_model(seed):
    rng = random.Random(seed)
    ps, npages = rng.choice([1, 2, 4]), rng.choice([6, 12, 40])
    c, m = RadixCache(ps, npages), Model(ps, npages)
    running = []                                   # (tokens, pages, lease_c, lease_m)
    for _ in range(300):
        op = rng.random()
        if op < 0.5 and len(running) < 4:
            toks = [rng.randrange(3) for _ in range(rng.randrange(0, 5 * ps + 2))]
            nc, pc, lc = c.match(toks)
            nm, pm, lm = m.match(toks)
            assert (nc, list(pc)) == (nm, pm)
            need = -(-len(toks) // ps) - len(pm)
            got_m = m.alloc(need)
            if got_m is None:
                with pytest.raises(RadixError):
                    c.alloc(need)
                c.release(lc, []); m.release(lm, [])
            else:
                got_c = c.alloc(need)
                assert list(got_c) == got_m
                running.append((toks, list(pc) + got_m, lc, lm))
        elif running:
            toks, pages, lc, lm = running.pop(rng.randrange(len(running)))
            if rng.random() < 0.7:
                assert c.insert(toks, pages, lc) == m.insert(toks, pages, lm)
            else:
                c.release(lc, pages); m.release(lm, pages)
        assert c.stats() == m.stats()
        held = sum(len(p) - sum(1 for x in p if m.state[x] == "cached") for _, p, _, _ in running)
        s = c.stats()
        assert s["free"] + s["cached"] + held == npages


def _kv_for(tokens, pos, hkv, d):
    """Deterministic K/V of a token at `pos`: a function of the prefix tokens[0..pos] only."""
    g = torch.Generator().manual_seed(hash(tuple(tokens[:pos + 1])) & 0x7FFFFFFF)
    return (torch.randn(2, hkv, d, generator=g)).to(torch.bfloat16)


def test_shared_prefix_page_tables_match_private_pages():
    """Requests admitted through the cache read their shared prefix from earlier requests' pages.

    Each request is checked while it runs (after admission and storing its own tokens, before
    its pages are inserted and possibly reused), against the same request on private pages.
    """
    import oracle
    ps, hq, hkv, d = 4, 4, 2, 16
    rng = random.Random(5)
    base = [rng.randrange(50) for _ in range(22)]
    reqs = [base, base[:13] + [rng.randrange(50) for _ in range(7)], base[:9] + [7, 7, 7],
            base[:13] + [rng.randrange(50) for _ in range(9)]]
    c = RadixCache(ps, 64)
    kp = torch.full((64 * ps, hkv, d), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    prefixes = []
    for toks in reqs:
        n, pages, lease = c.admit(toks)
        prefixes.append(n)
        for pos in range(n, len(toks)):            # compute (store) only the non-cached tokens
            slot = int(pages[pos // ps]) * ps + pos % ps
            kv = _kv_for(toks, pos, hkv, d)
            kp[slot], vp[slot] = kv[0], kv[1]
        ext = len(toks) - n
        q = torch.randn(ext, hq, d).to(torch.bfloat16)
        o, lse = oracle.extend(q, kp, vp, ps, pages[None, :], np.array([n], np.int32),
                               np.array([ext], np.int32), 0.25)
        # the same request on private pages holding all of its tokens
        npg = math.ceil(len(toks) / ps)
        kp2 = torch.zeros(npg * ps, hkv, d, dtype=torch.bfloat16)
        vp2 = torch.zeros_like(kp2)
        for pos in range(len(toks)):
            kv = _kv_for(toks, pos, hkv, d)
            kp2[pos], vp2[pos] = kv[0], kv[1]
        o2, lse2 = oracle.extend(q, kp2, vp2, ps, np.arange(npg, dtype=np.int32)[None, :],
                                 np.array([n], np.int32), np.array([ext], np.int32), 0.25)
        np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)
        c.insert(toks, pages, lease)               # finished: cache its full pages
    assert prefixes == [0, 12, 8, 12]


def test_eviction_cost_follows_pages_freed_not_tree_size():
    """A full 1M-page pool: evicting allocations cost per page freed, not per cached page.

    1024 cached chains of 1024 single-token pages fill the pool.  Two hundred 1-page
    allocations (each evicts one leaf) and then one 100k-page allocation must be fast;
    a walk of the whole tree per allocation would take seconds for the first part alone.
    Eviction order stays oldest-first: the first chains inserted lose their tails first.
    """
    import time
    n_chain, chain = 1024, 1024
    c = RadixCache(page_size=1, num_pages=n_chain * chain)
    for i in range(n_chain):
        toks = np.arange(chain, dtype=np.int32) + i * chain
        _, _, lease = c.match(toks)
        c.insert(toks, c.alloc(chain), lease)
    assert c.stats() == {"free": 0, "cached": n_chain * chain, "pinned": 0}
    t0 = time.perf_counter()
    for _ in range(200):
        c.alloc(1)
    t_small = time.perf_counter() - t0
    t0 = time.perf_counter()
    c.alloc(100_000)
    t_big = time.perf_counter() - t0
    assert t_small < 0.5, f"200 one-page evictions took {t_small:.2f} s"
    assert t_big < 2.0, f"a 100k-page eviction took {t_big:.2f} s"
    assert c.stats()["cached"] == n_chain * chain - 100_200
    # 100,200 = 97 * 1024 + 872: chains 0..96 (the oldest) are gone, chain 97 lost its
    # last 872 pages, chain 98 is whole
    n, _, lease = c.match(np.arange(chain, dtype=np.int32) + 97 * chain)
    assert n == chain - 872
    c.release(lease, [])
    n, _, lease = c.match(np.arange(chain, dtype=np.int32) + 98 * chain)
    assert n == chain
    c.release(lease, [])
    n, _, lease = c.match(np.arange(chain, dtype=np.int32))
    assert n == 0
    c.release(lease, [])
