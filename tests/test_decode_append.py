"""msgl_attn_decode_append: store the current token's K/V and decode in one launch.

Compared with the fp64 oracle run on the pool that already holds the new
rows, while the GPU pool starts with those rows poisoned (NaN): the kernel
must attend the new key from k_new/v_new and leave the rows, bit-exact, in
the pool.
"""
import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def _run(w, poison=True, loc=None, status=None):
    d = w.decode
    full_k, full_v = w.k_pool.clone(), w.v_pool.clone()
    idx = d.new_loc.long()
    k_new, v_new = full_k[idx].contiguous(), full_v[idx].contiguous()
    if poison:
        w.k_pool[idx] = float("nan")
        w.v_pool[idx] = float("nan")
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    o, lse = ops.attn_decode_append(pool, d.q, k_new, v_new, d.new_loc if loc is None else loc,
                                    d.page_table, d.seq_lens, d.max_seq_len, w.scale, status=status)
    return o, lse, full_k, full_v


@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_append_matches_oracle_and_writes_pool(cfg):
    w = W.config(cfg, device="cuda", part="decode")
    status = ops.new_status()
    o, lse, full_k, full_v = _run(w, status=status)
    assert ops.read_status(status) == 0
    d = w.decode
    ref_o, ref_l = oracle.decode(d.q.cpu(), full_k.cpu(), full_v.cpu(), w.page_size, d.page_table.cpu(),
                                 d.seq_lens.cpu(), w.scale)
    assert_o_close(o, ref_o, f"config {cfg}")
    assert_lse_close(lse, ref_l)
    assert torch.equal(w.k_pool.view(torch.int16), full_k.view(torch.int16))
    assert torch.equal(w.v_pool.view(torch.int16), full_v.view(torch.int16))


@pytest.mark.parametrize("ps", [1, 16, 64])
def test_append_short_and_page_boundary_lengths(ps):
    seqs = [1, 2, ps, ps + 1, 17, 300, 2049]
    w = W.make_workload("app", 40, 8, 128, ps, seed=60 + ps, decode_seq_lens=seqs, device="cuda")
    o, lse, full_k, full_v = _run(w)
    d = w.decode
    ref_o, ref_l = oracle.decode(d.q.cpu(), full_k.cpu(), full_v.cpu(), w.page_size, d.page_table.cpu(),
                                 d.seq_lens.cpu(), w.scale)
    a, _ = oracle.decode(d.q.cpu(), full_k.cpu(), full_v.cpu().abs(), w.page_size, d.page_table.cpu(),
                         d.seq_lens.cpu(), w.scale)
    assert_o_close(o, ref_o, abs_ref=a)
    assert_lse_close(lse, ref_l)
    assert torch.equal(w.k_pool.view(torch.int16), full_k.view(torch.int16))


@pytest.mark.parametrize("ps", [1, 64])
def test_append_wrong_slot_is_flagged(ps):
    w = W.make_workload("appbad", 16, 8, 128, ps, seed=70, decode_seq_lens=[40, 50], device="cuda")
    loc = w.decode.new_loc.clone()
    loc[1] = (int(loc[1]) + 1) % w.num_slots
    status = ops.new_status()
    _run(w, poison=False, loc=loc, status=status)
    assert ops.read_status(status) & ops.DEVERR_APPEND_SLOT


def test_append_two_head_groups_and_split_requests():
    """16 kv heads (two head groups per key) and requests long enough to span several CTA
    ranges: only the range holding the current token writes it."""
    w = W.make_workload("app16", 32, 16, 128, 64, seed=71, decode_seq_lens=[9000, 7000, 65, 3000],
                        device="cuda")
    o, lse, full_k, full_v = _run(w)
    d = w.decode
    ref_o, ref_l = oracle.decode(d.q.cpu(), full_k.cpu(), full_v.cpu(), w.page_size, d.page_table.cpu(),
                                 d.seq_lens.cpu(), w.scale)
    a, _ = oracle.decode(d.q.cpu(), full_k.cpu(), full_v.cpu().abs(), w.page_size, d.page_table.cpu(),
                         d.seq_lens.cpu(), w.scale)
    assert_o_close(o, ref_o, abs_ref=a)
    assert_lse_close(lse, ref_l)
    assert torch.equal(w.k_pool.view(torch.int16), full_k.view(torch.int16))
    assert torch.equal(w.v_pool.view(torch.int16), full_v.view(torch.int16))
