"""Pins for the fp64 oracle, independent of the oracle's own code.

Every check here compares the oracle with something other than itself:

* a library routine the definition reduces to: PyTorch's fp64 scaled-dot-
  product attention (``enable_gqa``: consecutive q heads share a kv head)
  for O, and PyTorch's CPU flash-attention op, which also returns the
  natural-log LSE, on the gathered, contiguous K/V with an explicit mask;
* closed forms: one key; q = 0; all keys equal; V constant; two keys;
* invariants the method fixes: the same result for page sizes 1/16/64 and
  under any permutation of pool pages; a prefill split into chunks equals
  the unsplit prefill; extend over a cached prefix equals recomputing the
  whole sequence; decode equals the last row of the extend; attention over
  a key range splits into two ranges merged by their LSEs;
* a pure-Python brute force that walks the pages one by one;
* the store step against NumPy fancy-index assignment.

Each pin takes ``mutant``; ``test_oracle_mutants.py`` builds oracles with
one planted mistake each and checks that every such mistake fails a pin.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from paged_kv_attention_24_gb300 import workloads as W

TOL = 1e-11


def tiny(hq=4, hkv=2, d=8, ps=1, dec=None, pre=None, ext=None, shared=0, seed=0, slots=None):
    if slots is None:
        need = 0
        if dec is not None:
            need += sum(-(-s // ps) for s in dec)
        if ext is not None:
            need += sum(-(-(p + e) // ps) for p, e in zip(pre, ext))
        slots = (need + 8) * ps
    return W.make_workload("tiny", hq, hkv, d, ps, seed, decode_seq_lens=dec, extend_prefix_lens=pre,
                           extend_ext_lens=ext, shared_prefix_len=shared, num_slots=slots)


def gather(w, table_row, n):
    """Contiguous [n, Hkv, D] fp64 K and V of one request (a plain gather, no attention math)."""
    ps = w.page_size
    pos = np.arange(n)
    tr = table_row.numpy()
    slots = tr[pos // ps].astype(np.int64) * ps + pos % ps
    return (w.k_pool[torch.from_numpy(slots)].double(), w.v_pool[torch.from_numpy(slots)].double())


def run_extend(w, mutant=0):
    e = w.extend
    return oracle.extend(e.q, w.k_pool, w.v_pool, w.page_size, e.page_table, e.prefix_lens,
                         e.ext_lens, w.scale, mutant=mutant)


def run_decode(w, mutant=0):
    d = w.decode
    return oracle.decode(d.q, w.k_pool, w.v_pool, w.page_size, d.page_table, d.seq_lens, w.scale,
                         mutant=mutant)


# ----------------------------------------------------------------- pins

def pin_sdpa_extend(mutant=0, ps=4, seed=1):
    """O against torch SDPA (fp64, enable_gqa) and LSE against the CPU flash op."""
    w = tiny(hq=6, hkv=2, d=16, ps=ps, pre=[0, 5, 9], ext=[7, 3, 6], seed=seed)
    o, lse = run_extend(w, mutant)
    e = w.extend
    for b in range(3):
        p, n = int(e.prefix_lens[b]), int(e.ext_lens[b])
        k, v = gather(w, e.page_table[b], p + n)
        lo, hi = int(e.cu_ext[b]), int(e.cu_ext[b + 1])
        q = e.q[lo:hi].double().permute(1, 0, 2).unsqueeze(0)        # [1, Hq, n, D]
        kk = k.permute(1, 0, 2).unsqueeze(0)                           # [1, Hkv, S, D]
        vv = v.permute(1, 0, 2).unsqueeze(0)
        allowed = torch.arange(p + n)[None, :] <= (p + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=allowed,
                                                               scale=w.scale, enable_gqa=True)
        np.testing.assert_allclose(o[lo:hi], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=TOL)
        rep = w.hq // w.hkv
        fmask = torch.zeros(n, p + n, dtype=torch.float64).masked_fill(~allowed, -math.inf)
        _, ref_lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
            q, kk.repeat_interleave(rep, 1), vv.repeat_interleave(rep, 1), 0.0, False,
            attn_mask=fmask, scale=w.scale)
        np.testing.assert_allclose(lse[lo:hi], ref_lse[0].permute(1, 0).numpy(), rtol=0, atol=TOL)


def pin_sdpa_decode(mutant=0, ps=16, seed=2):
    w = tiny(hq=8, hkv=2, d=8, ps=ps, dec=[1, 17, 40, 33], seed=seed)
    o, lse = run_decode(w, mutant)
    dd = w.decode
    for b in range(dd.num_reqs):
        n = int(dd.seq_lens[b])
        k, v = gather(w, dd.page_table[b], n)
        q = dd.q[b:b + 1].double().permute(1, 0, 2).unsqueeze(0)       # [1, Hq, 1, D]
        kk = k.permute(1, 0, 2).unsqueeze(0)
        vv = v.permute(1, 0, 2).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, scale=w.scale, enable_gqa=True)
        np.testing.assert_allclose(o[b], ref[0, :, 0].numpy(), rtol=0, atol=TOL)
        rep = w.hq // w.hkv
        _, ref_lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
            q, kk.repeat_interleave(rep, 1), vv.repeat_interleave(rep, 1), 0.0, False, scale=w.scale)
        np.testing.assert_allclose(lse[b], ref_lse[0, :, 0].numpy(), rtol=0, atol=TOL)


def pin_closed_forms(mutant=0):
    # one key: o = v0, lse = scale * <q, k0>
    w = tiny(hq=4, hkv=2, d=8, ps=1, dec=[1, 1], seed=3)
    o, lse = run_decode(w, mutant)
    dd = w.decode
    for b in range(2):
        slot = int(dd.page_table[b, 0])
        for h in range(4):
            g = h // 2
            kv = w.k_pool[slot, g].double()
            np.testing.assert_allclose(o[b, h], w.v_pool[slot, g].double().numpy(), rtol=0, atol=TOL)
            s0 = w.scale * float((dd.q[b, h].double() * kv).sum())
            assert abs(lse[b, h] - s0) < TOL
    # q = 0: uniform weights -> o = mean of v, lse = ln(n)
    w = tiny(hq=2, hkv=1, d=4, ps=2, dec=[5, 9], seed=4)
    w.decode.q.zero_()
    o, lse = run_decode(w, mutant)
    for b, n in enumerate([5, 9]):
        k, v = gather(w, w.decode.page_table[b], n)
        np.testing.assert_allclose(o[b, 0], v[:, 0].mean(0).numpy(), rtol=0, atol=TOL)
        assert abs(lse[b, 0] - math.log(n)) < TOL
    # V constant per kv head -> o equals that constant for every q head of the group
    w = tiny(hq=4, hkv=2, d=4, ps=1, dec=[6], seed=5)
    w.v_pool[:, 0, :] = 0.75
    w.v_pool[:, 1, :] = -2.5
    o, _ = run_decode(w, mutant)
    np.testing.assert_allclose(o[0, :2], 0.75, atol=TOL)
    np.testing.assert_allclose(o[0, 2:], -2.5, atol=TOL)
    # all keys equal: lse = s + ln(n), o = mean v
    w = tiny(hq=2, hkv=1, d=4, ps=1, dec=[7], seed=6)
    w.k_pool[:] = torch.tensor([0.5, -1.0, 2.0, 0.25], dtype=torch.bfloat16)
    o, lse = run_decode(w, mutant)
    k, v = gather(w, w.decode.page_table[0], 7)
    s = w.scale * float((w.decode.q[0, 0].double() * k[0, 0]).sum())
    assert abs(lse[0, 0] - (s + math.log(7))) < TOL
    np.testing.assert_allclose(o[0, 0], v[:, 0].mean(0).numpy(), atol=TOL)
    # two keys: o = sigma(s0 - s1) v0 + sigma(s1 - s0) v1, lse = logaddexp(s0, s1)
    w = tiny(hq=2, hkv=2, d=4, ps=1, dec=[2], seed=7)
    o, lse = run_decode(w, mutant)
    k, v = gather(w, w.decode.page_table[0], 2)
    for h in range(2):
        s = [w.scale * float((w.decode.q[0, h].double() * k[j, h]).sum()) for j in range(2)]
        a = 1.0 / (1.0 + math.exp(s[1] - s[0]))
        np.testing.assert_allclose(o[0, h], (a * v[0, h] + (1 - a) * v[1, h]).numpy(), atol=TOL)
        assert abs(lse[0, h] - np.logaddexp(s[0], s[1])) < TOL


def pin_page_size_and_permutation(mutant=0):
    """Same logical K/V laid out with page sizes 1, 16, 64 and shuffled pages: same result."""
    rng = np.random.default_rng(11)
    hq, hkv, d = 4, 2, 8
    seqs = [70, 129, 3]
    kv = [(torch.randn(n, hkv, d).to(torch.bfloat16), torch.randn(n, hkv, d).to(torch.bfloat16)) for n in seqs]
    q = torch.randn(len(seqs), hq, d).to(torch.bfloat16)
    results = []
    for ps in (1, 16, 64):
        for shuffle in (False, True):
            pages_per = [-(-n // ps) for n in seqs]
            n_pages = sum(pages_per) + 3
            order = rng.permutation(n_pages) if shuffle else np.arange(n_pages)
            kp = torch.full((n_pages * ps, hkv, d), float("nan"), dtype=torch.bfloat16)
            vp = kp.clone()
            table = np.full((len(seqs), max(pages_per)), -1, dtype=np.int32)
            nxt = 0
            for b, n in enumerate(seqs):
                for i in range(pages_per[b]):
                    table[b, i] = order[nxt]; nxt += 1
                pos = np.arange(n)
                slots = table[b][pos // ps].astype(np.int64) * ps + pos % ps
                kp[torch.from_numpy(slots)] = kv[b][0]
                vp[torch.from_numpy(slots)] = kv[b][1]
            o, lse = oracle.decode(q, kp, vp, ps, table, np.array(seqs, dtype=np.int32), 0.3, mutant=mutant)
            results.append((o, lse))
    for o, lse in results[1:]:
        np.testing.assert_allclose(o, results[0][0], rtol=0, atol=TOL)
        np.testing.assert_allclose(lse, results[0][1], rtol=0, atol=TOL)


def pin_chunked_equals_unchunked(mutant=0):
    """A 40-token prefill run as chunks 11 + 13 + 16 over the growing prefix equals one pass."""
    w = tiny(hq=4, hkv=2, d=8, ps=4, pre=[0], ext=[40], seed=8)
    o_full, lse_full = run_extend(w, mutant)
    e = w.extend
    row = 0
    for lo, hi in ((0, 11), (11, 24), (24, 40)):
        o, lse = oracle.extend(e.q[lo:hi], w.k_pool, w.v_pool, w.page_size, e.page_table,
                               np.array([lo], np.int32), np.array([hi - lo], np.int32), w.scale,
                               mutant=mutant)
        np.testing.assert_allclose(o, o_full[lo:hi], rtol=0, atol=TOL)
        np.testing.assert_allclose(lse, lse_full[lo:hi], rtol=0, atol=TOL)
        row += hi - lo
    assert row == 40


def pin_prefix_and_decode_consistency(mutant=0):
    """Extend over a cached prefix equals full recompute; decode equals the extend's last row."""
    w = tiny(hq=6, hkv=3, d=8, ps=2, pre=[13], ext=[9], seed=9)
    e = w.extend
    o_ext, lse_ext = run_extend(w, mutant)
    # full recompute: the same sequence as a 22-token prefill with no prefix; q for the first
    # 13 rows is arbitrary (only the last 9 rows are compared)
    q_full = torch.cat([torch.randn(13, 6, 8).to(torch.bfloat16), e.q])
    o_all, lse_all = oracle.extend(q_full, w.k_pool, w.v_pool, w.page_size, e.page_table,
                                   np.array([0], np.int32), np.array([22], np.int32), w.scale,
                                   mutant=mutant)
    np.testing.assert_allclose(o_ext, o_all[13:], rtol=0, atol=TOL)
    np.testing.assert_allclose(lse_ext, lse_all[13:], rtol=0, atol=TOL)
    o_dec, lse_dec = oracle.decode(e.q[-1:], w.k_pool, w.v_pool, w.page_size, e.page_table,
                                   np.array([22], np.int32), w.scale, mutant=mutant)
    np.testing.assert_allclose(o_dec[0], o_ext[-1], rtol=0, atol=TOL)
    np.testing.assert_allclose(lse_dec[0], lse_ext[-1], rtol=0, atol=TOL)


def pin_split_merge(mutant=0):
    """Keys [0, n) = keys [0, a) merged with keys [a, n) through their LSEs."""
    w = tiny(hq=4, hkv=2, d=8, ps=1, dec=[30], seed=10)
    dd = w.decode
    o, lse = run_decode(w, mutant)
    a = 12
    table = dd.page_table[0].numpy()
    o1, l1 = oracle.decode(dd.q, w.k_pool, w.v_pool, 1, table[None, :a], np.array([a], np.int32),
                           w.scale, mutant=mutant)
    o2, l2 = oracle.decode(dd.q, w.k_pool, w.v_pool, 1, table[None, a:30], np.array([30 - a], np.int32),
                           w.scale, mutant=mutant)
    m = np.logaddexp(l1, l2)
    np.testing.assert_allclose(lse, m, rtol=0, atol=TOL)
    merged = (np.exp(l1 - m)[..., None] * o1 + np.exp(l2 - m)[..., None] * o2)
    np.testing.assert_allclose(o, merged, rtol=0, atol=TOL)


def pin_brute_force(mutant=0):
    for ps, d, seed in ((1, 4, 12), (2, 8, 13), (4, 4, 14)):
        w = tiny(hq=4, hkv=2, d=d, ps=ps, pre=[0, 3], ext=[4, 2], seed=seed)
        e = w.extend
        o, lse = run_extend(w, mutant)
        kp = w.k_pool.float().tolist()
        vp = w.v_pool.float().tolist()
        t = 0
        for b in range(2):
            pages = [int(x) for x in e.page_table[b] if int(x) >= 0]
            for i in range(int(e.ext_lens[b])):
                qrow = e.q[t].float().tolist()
                for h in range(4):
                    ob, lb = brute.attention_row(qrow, kp, vp, ps, pages, int(e.prefix_lens[b]) + i, h,
                                                 4, 2, w.scale)
                    np.testing.assert_allclose(o[t, h], ob, rtol=0, atol=1e-12)
                    assert abs(lse[t, h] - lb) < 1e-12
                t += 1


def pin_store(mutant=0):
    rng = np.random.default_rng(15)
    S, hkv, d, n = 64, 2, 8, 20
    kp = torch.randn(S, hkv, d).to(torch.bfloat16)
    vp = torch.randn(S, hkv, d).to(torch.bfloat16)
    kn = torch.randn(n, hkv, d).to(torch.bfloat16)
    vn = torch.randn(n, hkv, d).to(torch.bfloat16)
    loc = rng.permutation(S)[:n].astype(np.int32)
    ko, vo = oracle.store_kv(kp, vp, kn, vn, loc, mutant=mutant)
    kr = kp.clone(); vr = vp.clone()
    kr[torch.from_numpy(loc).long()] = kn
    vr[torch.from_numpy(loc).long()] = vn
    assert np.array_equal(ko, oracle._bits(kr)) and np.array_equal(vo, oracle._bits(vr))


PINS = [pin_sdpa_extend, pin_sdpa_decode, pin_closed_forms, pin_page_size_and_permutation,
        pin_chunked_equals_unchunked, pin_prefix_and_decode_consistency, pin_split_merge,
        pin_brute_force, pin_store]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("ps", [1, 16, 64])
def test_sdpa_page_sizes(ps):
    pin_sdpa_extend(0, ps=ps, seed=20 + ps)
    pin_sdpa_decode(0, ps=ps, seed=30 + ps)


def test_out_of_range_page_is_an_error():
    w = tiny(hq=2, hkv=1, d=4, ps=1, dec=[5], seed=16)
    bad = w.decode.page_table.clone()
    bad[0, 2] = 10_000
    with pytest.raises(oracle.OracleError):
        oracle.decode(w.decode.q, w.k_pool, w.v_pool, 1, bad, w.decode.seq_lens, w.scale)


def test_nan_poison_untouched():
    """Unused slots are NaN; a correct gather never reads them."""
    w = tiny(hq=4, hkv=2, d=8, ps=16, dec=[5, 33], seed=17)
    assert torch.isnan(w.k_pool.float()).any()
    o, lse = run_decode(w)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
