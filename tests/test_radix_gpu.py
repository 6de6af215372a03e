"""The radix cache feeding the GPU kernels: page tables of shared prefixes -> store -> extend.

A first request runs and is cached.  A batch of four requests that share
parts of its prefix is then admitted together: each gets the cached pages of
its longest page-aligned match plus fresh pages, msgl_store_kv writes the
new tokens' K/V, and one msgl_attn_extend call runs the batch over those
page tables.  The result must match the fp64 oracle on the same pool.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300.radix import RadixCache
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def test_radix_batch_extend_on_gpu():
    ps, hq, hkv, d, num_pages = 16, 40, 8, 128, 512
    g = torch.Generator().manual_seed(77)
    rng = np.random.default_rng(77)
    c = RadixCache(ps, num_pages)
    kp = torch.full((num_pages * ps, hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = kp.clone()
    pool = ops.KVPool(kp, vp, ps)

    def store(pages, lo, hi):
        n = hi - lo
        if n == 0:
            return
        k = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16).cuda()
        v = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16).cuda()
        pos = np.arange(lo, hi)
        loc = torch.from_numpy((pages[pos // ps] * ps + pos % ps).astype(np.int32)).cuda()
        ops.store_kv(pool, k, v, loc)

    warm = rng.integers(0, 1000, size=700).tolist()
    n0, pages0, lease0 = c.admit(warm)
    store(pages0, n0, len(warm))
    c.insert(warm, pages0, lease0)

    reqs = [warm[:300] + rng.integers(0, 1000, size=200).tolist(),
            warm[:650] + rng.integers(0, 1000, size=5).tolist(),
            rng.integers(0, 1000, size=129).tolist(),
            warm[:16] + rng.integers(0, 1000, size=33).tolist()]
    admitted = [c.admit(t) for t in reqs]
    for (n, pages, _), toks in zip(admitted, reqs):
        store(pages, n, len(toks))
    prefix = np.array([a[0] for a in admitted], dtype=np.int32)
    ext = np.array([len(t) - a[0] for t, a in zip(reqs, admitted)], dtype=np.int32)
    assert list(prefix) == [288, 640, 0, 16]
    width = max(len(a[1]) for a in admitted)
    pt = np.full((len(reqs), width), -1, dtype=np.int32)
    for i, a in enumerate(admitted):
        pt[i, :len(a[1])] = a[1]
    cu = np.concatenate([[0], np.cumsum(ext)]).astype(np.int32)
    T = int(cu[-1])
    q = torch.randn(T, hq, d, generator=g).to(torch.bfloat16).cuda()
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    status = ops.new_status()
    o, lse = ops.attn_extend(pool, q, dev(pt), dev(prefix), dev(ext), dev(cu), int(ext.max()),
                             int((prefix + ext).max()), d ** -0.5, status=status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = oracle.extend(q.cpu(), kp.cpu(), vp.cpu(), ps, pt, prefix, ext, d ** -0.5)
    a, _ = oracle.extend(q.cpu(), kp.cpu(), vp.cpu().abs(), ps, pt, prefix, ext, d ** -0.5)
    assert_o_close(o, ref_o, abs_ref=a)
    assert_lse_close(lse, ref_l)
    for (n, pages, lease), toks in zip(admitted, reqs):
        c.insert(toks, pages, lease)
    assert c.stats()["pinned"] == 0
