"""Error behaviour: host validation codes and device status bits (no traps, no faults).

Device-side cases use in-bounds buffers only; the bad value is an index the
kernel range-checks before any access, so nothing out of bounds is read.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def test_bad_page_id_sets_status_and_zeroes_only_that_row():
    w = W.make_workload("badpage", 16, 8, 128, 16, seed=1, decode_seq_lens=[300, 200, 50], device="cuda")
    d = w.decode
    good_o, good_l = ops.attn_decode(ops.KVPool(w.k_pool, w.v_pool, 16), d.q, d.page_table, d.seq_lens,
                                     d.max_seq_len, w.scale)
    pt = d.page_table.clone()
    pt[1, 3] = w.num_slots // 16 + 5          # page id past the pool
    status = ops.new_status()
    o, lse = ops.attn_decode(ops.KVPool(w.k_pool, w.v_pool, 16), d.q, pt, d.seq_lens, d.max_seq_len,
                             w.scale, status=status)
    flags = ops.read_status(status)
    assert flags & ops.DEVERR_PAGE_RANGE
    assert torch.all(o[1] == 0) and torch.all(lse[1] == float("-inf"))
    assert torch.equal(o[0], good_o[0]) and torch.equal(o[2], good_o[2])


@pytest.mark.parametrize("ps", [1, 64])
def test_bad_page_inside_a_long_request(ps):
    """A bad page id deep inside a long request (page size 64 takes the TMA box copies, 1 the
    per-key copies): only that request's row is zeroed; the others match the clean run."""
    seqs = [3000, 2500, 700, 4100]
    w = W.make_workload("badmid", 32, 8, 128, ps, seed=11, decode_seq_lens=seqs, device="cuda")
    d = w.decode
    pool = ops.KVPool(w.k_pool, w.v_pool, ps)
    good_o, good_l = ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, d.max_seq_len, w.scale)
    pt = d.page_table.clone()
    pt[1, 1337 // ps] = -3
    status = ops.new_status()
    o, lse = ops.attn_decode(pool, d.q, pt, d.seq_lens, d.max_seq_len, w.scale, status=status)
    assert ops.read_status(status) & ops.DEVERR_PAGE_RANGE
    assert torch.all(o[1] == 0) and torch.all(lse[1] == float("-inf"))
    for b in (0, 2, 3):
        assert torch.equal(o[b], good_o[b]) and torch.equal(lse[b], good_l[b])


def test_short_page_table_is_a_range_error():
    w = W.make_workload("short", 16, 8, 128, 16, seed=2, decode_seq_lens=[100], device="cuda")
    d = w.decode
    status = ops.new_status()
    narrow = d.page_table[:, :3].contiguous()   # 3 pages = 48 keys < 100
    o, lse = ops.attn_decode(ops.KVPool(w.k_pool, w.v_pool, 16), d.q, narrow, d.seq_lens, 100, w.scale,
                             status=status)
    assert ops.read_status(status) & ops.DEVERR_PAGE_RANGE
    assert torch.all(o == 0)


def test_zero_seq_len_is_a_length_error():
    w = W.make_workload("zero", 16, 8, 128, 1, seed=3, decode_seq_lens=[10, 20], device="cuda")
    d = w.decode
    d.seq_lens[0] = 0
    status = ops.new_status()
    o, lse = ops.attn_decode(ops.KVPool(w.k_pool, w.v_pool, 1), d.q, d.page_table, d.seq_lens, 20,
                             w.scale, status=status)
    assert ops.read_status(status) & ops.DEVERR_LENGTH
    assert torch.all(o[0] == 0) and torch.isfinite(lse[1]).all()


def test_seq_len_over_max_is_a_length_error():
    w = W.make_workload("over", 16, 8, 128, 1, seed=4, decode_seq_lens=[10, 20], device="cuda")
    d = w.decode
    status = ops.new_status()
    o, lse = ops.attn_decode(ops.KVPool(w.k_pool, w.v_pool, 1), d.q, d.page_table, d.seq_lens, 15,
                             w.scale, status=status)
    assert ops.read_status(status) & ops.DEVERR_LENGTH
    assert torch.all(o[1] == 0)


def test_bad_out_loc_skips_row_and_sets_status():
    S = 256
    kp = torch.zeros(S, 8, 128, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    kn = torch.ones(3, 8, 128, dtype=torch.bfloat16, device="cuda")
    loc = torch.tensor([5, S + 3, 7], dtype=torch.int32, device="cuda")
    status = ops.new_status()
    ops.store_kv(ops.KVPool(kp, vp, 1), kn, kn, loc, status=status)
    assert ops.read_status(status) == ops.DEVERR_SLOT_RANGE
    assert torch.all(kp[5] == 1) and torch.all(kp[7] == 1)
    assert int((kp != 0).any(dim=(1, 2)).sum()) == 2


def test_wrong_positions_flagged():
    w = W.make_workload("pos", 16, 8, 128, 1, seed=5, extend_prefix_lens=[4], extend_ext_lens=[30],
                        device="cuda")
    e = w.extend
    pos = e.positions.clone()
    pos[7] += 1
    status = ops.new_status()
    ops.attn_extend(ops.KVPool(w.k_pool, w.v_pool, 1), e.q, e.page_table, e.prefix_lens, e.ext_lens,
                    e.cu_ext, e.max_ext_len, e.max_seq_len, w.scale, positions=pos, status=status)
    assert ops.read_status(status) & ops.DEVERR_POSITION


def test_host_validation_errors():
    w = W.make_workload("host", 16, 8, 128, 1, seed=6, decode_seq_lens=[50], device="cuda")
    d = w.decode
    pool = ops.KVPool(w.k_pool, w.v_pool, 1)
    with pytest.raises(ops.MsglError) as ei:
        ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, 50, 0.0)
    assert ei.value.status == 1
    bad_pool = ops.KVPool(w.k_pool, w.v_pool, 3)
    with pytest.raises(ops.MsglError) as ei:
        ops.attn_decode(bad_pool, d.q, d.page_table, d.seq_lens, 50, w.scale)
    assert ei.value.status == 2
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.MsglError) as ei:
        ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, 100000, w.scale, workspace=small)
    assert ei.value.status == 6
    with pytest.raises(ValueError):
        ops.attn_decode(pool, d.q.float(), d.page_table, d.seq_lens, 50, w.scale)


def test_status_word_accumulates_and_calls_continue():
    """After an error the context stays usable and later good calls are exact."""
    w = W.make_workload("after", 16, 8, 128, 1, seed=7, decode_seq_lens=[64], device="cuda")
    d = w.decode
    pool = ops.KVPool(w.k_pool, w.v_pool, 1)
    pt = d.page_table.clone()
    pt[0, 0] = -3
    status = ops.new_status()
    ops.attn_decode(pool, d.q, pt, d.seq_lens, 64, w.scale, status=status)
    assert ops.read_status(status) & ops.DEVERR_PAGE_RANGE
    import oracle
    o, lse = ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, 64, w.scale)
    ref_o, _ = oracle.decode(d.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(), 1, d.page_table.cpu(),
                             d.seq_lens.cpu(), w.scale)
    assert_o_close(o, ref_o)


def test_bounded_wait_times_out_into_status_and_context_survives():
    """A wait that nothing satisfies gives up (about 5 ms here), sets the timeout bit, and later
    calls still run and are exact."""
    import time
    status = ops.new_status()
    t0 = time.time()
    ops.selftest_wait_timeout(status, budget_cycles=10_000_000)
    flags = ops.read_status(status)
    assert flags == ops.DEVERR_TIMEOUT
    assert time.time() - t0 < 5.0
    w = W.make_workload("after_timeout", 16, 8, 128, 16, seed=9, decode_seq_lens=[200, 33], device="cuda")
    d = w.decode
    import oracle
    o, lse = ops.attn_decode(ops.KVPool(w.k_pool, w.v_pool, 16), d.q, d.page_table, d.seq_lens, 200, w.scale)
    ref_o, _ = oracle.decode(d.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(), 16, d.page_table.cpu(),
                             d.seq_lens.cpu(), w.scale)
    assert_o_close(o, ref_o)


def test_extend_chunk_longer_than_max_ext_len_is_a_length_error():
    """A chunk longer than the max_ext_len bound: status bit set; the other request's rows exact."""
    from tests.test_extend import run_oracle
    w = W.make_workload("ext_over", 16, 8, 128, 16, seed=8, extend_prefix_lens=[100, 40],
                        extend_ext_lens=[50, 300], device="cuda")
    e = w.extend
    status = ops.new_status()
    o, lse = ops.attn_extend(ops.KVPool(w.k_pool, w.v_pool, w.page_size), e.q, e.page_table, e.prefix_lens,
                             e.ext_lens, e.cu_ext, 60, e.max_seq_len, w.scale, status=status)
    assert ops.read_status(status) & ops.DEVERR_LENGTH
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o[:50], ref_o[:50], "in-bound request")
    assert_lse_close(lse[:50], ref_l[:50], "in-bound request")
