"""msgl_attn_mixed: the extend and decode batches of one forward in one call.

The mixed step runs the same kernels as msgl_attn_extend and msgl_attn_decode, in
another order (decode key ranges, then the extend behind them with programmatic
dependent launch, then the decode merge), so its outputs must equal the two
separate calls bit for bit.  The separate calls are checked against the oracle in
test_extend.py and test_decode.py; the decode half is checked against it here too.
"""
import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def separate(w, pool, status=None):
    e, d = w.extend, w.decode
    oe, le = ops.attn_extend(pool, e.q, e.page_table, e.prefix_lens, e.ext_lens, e.cu_ext, e.max_ext_len,
                             e.max_seq_len, w.scale, positions=e.positions, status=status)
    od, ld = ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, d.max_seq_len, w.scale, status=status)
    return oe, le, od, ld


def mixed(w, pool, status=None, **kw):
    e, d = w.extend, w.decode
    (oe, le), (od, ld) = ops.attn_mixed(pool, w.scale, e.q, e.page_table, e.prefix_lens, e.ext_lens, e.cu_ext,
                                        e.max_ext_len, e.max_seq_len, d.q, d.page_table, d.seq_lens,
                                        d.max_seq_len, positions=e.positions, status=status, **kw)
    return oe, le, od, ld


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def assert_same(a, b):
    for x, y, name in zip(a, b, ("extend o", "extend lse", "decode o", "decode lse")):
        assert torch.equal(bits(x), bits(y)), f"{name} differs from the separate calls"


@pytest.mark.parametrize("cfg", [4, 5])
def test_mixed_step_configs_match_separate_calls_and_oracle(cfg):
    w = W.config(cfg, device="cuda")
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    status = ops.new_status()
    ref = separate(w, pool, status)
    got = mixed(w, pool, status)
    assert ops.read_status(status) == 0
    assert_same(got, ref)
    d = w.decode
    ref_o, ref_l = oracle.decode(d.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(), w.page_size, d.page_table.cpu(),
                                 d.seq_lens.cpu(), w.scale)
    assert_o_close(got[2], ref_o, f"config {cfg} mixed decode")
    assert_lse_close(got[3], ref_l, f"config {cfg} mixed decode")


@pytest.mark.parametrize("ps", [1, 16, 64])
def test_mixed_small_batches(ps):
    w = W.make_workload("mix", 40, 8, 128, ps, seed=80 + ps, decode_seq_lens=[1, 17, 300, 2049, 4096],
                        extend_prefix_lens=[0, 64, 1000], extend_ext_lens=[5, 300, 129], device="cuda")
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    status = ops.new_status()
    ref = separate(w, pool, status)
    for _ in range(2):   # the workspace is reused: a second call gives the same bits
        got = mixed(w, pool, status)
        assert_same(got, ref)
    assert ops.read_status(status) == 0
    e = w.extend
    ref_o, ref_l = oracle.extend(e.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(), ps, e.page_table.cpu(),
                                 e.prefix_lens.cpu(), e.ext_lens.cpu(), w.scale)
    a, _ = oracle.extend(e.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu().abs(), ps, e.page_table.cpu(),
                         e.prefix_lens.cpu(), e.ext_lens.cpu(), w.scale)
    assert_o_close(got[0], ref_o, f"ps {ps} mixed extend", abs_ref=a)
    assert_lse_close(got[1], ref_l)


def test_mixed_with_one_batch_empty():
    w = W.make_workload("mix1", 16, 8, 128, 16, seed=90, decode_seq_lens=[700, 33],
                        extend_prefix_lens=[48], extend_ext_lens=[200], device="cuda")
    pool = ops.KVPool(w.k_pool, w.v_pool, 16)
    e, d = w.extend, w.decode
    ref = separate(w, pool)
    empty_q = torch.empty(0, 16, 128, dtype=torch.bfloat16, device="cuda")
    empty_i = torch.empty(0, dtype=torch.int32, device="cuda")
    (oe, le), _ = ops.attn_mixed(pool, w.scale, e.q, e.page_table, e.prefix_lens, e.ext_lens, e.cu_ext,
                                 e.max_ext_len, e.max_seq_len, empty_q, d.page_table[:0], empty_i, 1)
    assert torch.equal(bits(oe), bits(ref[0])) and torch.equal(bits(le), bits(ref[1]))
    _, (od, ld) = ops.attn_mixed(pool, w.scale, empty_q, e.page_table[:0], empty_i, empty_i,
                                 torch.zeros(1, dtype=torch.int32, device="cuda"), 0, 0, d.q, d.page_table,
                                 d.seq_lens, d.max_seq_len)
    assert torch.equal(bits(od), bits(ref[2])) and torch.equal(bits(ld), bits(ref[3]))


def test_mixed_graph_capture_replay():
    """Captured once, replayed with new queries and new decode lengths."""
    w = W.make_workload("mixg", 64, 8, 128, 64, seed=91, decode_seq_lens=[4000, 1500, 8192, 64] * 4,
                        extend_prefix_lens=[2048, 0], extend_ext_lens=[512, 700], device="cuda")
    pool = ops.KVPool(w.k_pool, w.v_pool, 64)
    e, d = w.extend, w.decode
    outs = [torch.empty_like(e.q), torch.empty(e.q.shape[:2], dtype=torch.float32, device="cuda"),
            torch.empty_like(d.q), torch.empty(d.q.shape[:2], dtype=torch.float32, device="cuda")]
    ws = torch.empty(ops.mixed_workspace_size(d.num_reqs, e.total_tokens, e.num_reqs, 64, 8, e.max_seq_len,
                                              d.max_seq_len), dtype=torch.uint8, device="cuda")
    kw = dict(ext_out=outs[0], ext_lse=outs[1], dec_out=outs[2], dec_lse=outs[3], workspace=ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mixed(w, pool, **kw)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mixed(w, pool, **kw)
    e.q.copy_(torch.randn_like(e.q.float()).to(torch.bfloat16))
    d.q.copy_(torch.randn_like(d.q.float()).to(torch.bfloat16))
    d.seq_lens.copy_(torch.clamp(d.seq_lens // 3, min=1))
    for t in outs:
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert_same(outs, separate(w, pool))


def test_mixed_validation_failure_launches_nothing():
    w = W.make_workload("mixbad", 16, 8, 128, 16, seed=92, decode_seq_lens=[100],
                        extend_prefix_lens=[0], extend_ext_lens=[50], device="cuda")
    pool = ops.KVPool(w.k_pool, w.v_pool, 16)
    e, d = w.extend, w.decode
    oe = torch.full_like(e.q, 3.0)
    od = torch.full_like(d.q, 3.0)
    with pytest.raises(ops.MsglError):
        # max_ext_len above max_seq_len is a host validation error of the extend batch
        ops.attn_mixed(pool, w.scale, e.q, e.page_table, e.prefix_lens, e.ext_lens, e.cu_ext, 50, 10,
                       d.q, d.page_table, d.seq_lens, d.max_seq_len, ext_out=oe, dec_out=od)
    with pytest.raises(ops.MsglError):
        # too small a workspace for the decode batch
        ops.attn_mixed(pool, w.scale, e.q, e.page_table, e.prefix_lens, e.ext_lens, e.cu_ext, e.max_ext_len,
                       e.max_seq_len, d.q, d.page_table, d.seq_lens, d.max_seq_len, ext_out=oe, dec_out=od,
                       workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert (oe == 3.0).all() and (od == 3.0).all()
