"""msgl_attn_extend against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def run_gpu(w, status=None, q=None, prefix=None, ext=None, cu=None, positions=None):
    e = w.extend
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    return ops.attn_extend(pool, e.q if q is None else q, e.page_table,
                           e.prefix_lens if prefix is None else prefix,
                           e.ext_lens if ext is None else ext, e.cu_ext if cu is None else cu,
                           e.max_ext_len, e.max_seq_len, w.scale,
                           positions=e.positions if positions is None else positions, status=status)


def run_oracle(w, v_abs=False):
    """The oracle's (o, lse); with v_abs, o over |V| (the rounding allowance's A)."""
    e = w.extend
    vp = w.v_pool.cpu()
    return oracle.extend(e.q.cpu(), w.k_pool.cpu(), vp.abs() if v_abs else vp, w.page_size,
                         e.page_table.cpu(), e.prefix_lens.cpu(), e.ext_lens.cpu(), w.scale)


def abs_ref(w):
    return run_oracle(w, v_abs=True)[0]


def test_extend_config2_full():
    w = W.config(2, device="cuda", part="extend")
    status = ops.new_status()
    o, lse = run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, "config 2")
    assert_lse_close(lse, ref_l, "config 2")


@pytest.mark.parametrize("cfg", [4, 5])
def test_extend_large_configs_full(cfg):
    """Every row and every q head of the Qwen3-14B and Qwen3-32B extends against the oracle.

    Qwen3-14B: one 8192-token chunk over a 4096-token cached prefix (40/8 heads, page
    size 16).  Qwen3-32B: 8 chunks of 1024 tokens over one shared 2048-token prefix
    (64/8 heads, page size 64).  The oracle takes about 35 s and 18 s of fp64 work on
    16 host cores.
    """
    w = W.config(cfg, device="cuda", part="extend")
    status = ops.new_status()
    o, lse = run_gpu(w, status)
    assert ops.read_status(status) == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    ref_o, ref_l = run_oracle(w)
    assert ref_o.shape == tuple(o.shape) and ref_l.shape == tuple(lse.shape)
    assert_o_close(o, ref_o, f"config {cfg}")
    assert_lse_close(lse, ref_l, f"config {cfg}")


@pytest.mark.parametrize("ps", [1, 16, 64, 256])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (40, 8), (64, 8), (8, 8), (4, 1)])
def test_extend_ragged_shapes(ps, hq, hkv):
    pre = [0, 5, 130, 0, 1000, 64, 255]
    ext = [1, 127, 128, 129, 33, 300, 2]
    w = W.make_workload("ragged", hq, hkv, 128, ps, seed=ps + hq, extend_prefix_lens=pre,
                        extend_ext_lens=ext, device="cuda")
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, f"ps={ps} hq={hq}", abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_extend_shared_prefix_pages():
    """Requests whose page tables point at the same prefix pages (radix hit)."""
    w = W.make_workload("shared", 64, 8, 128, 64, seed=9, extend_prefix_lens=[512] * 4,
                        extend_ext_lens=[200, 64, 1, 333], shared_prefix_len=512, device="cuda")
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_chunked_equals_unchunked_on_gpu():
    """A 700-token prefill run as chunks 300 + 250 + 150 matches the single pass (both vs oracle)."""
    w = W.make_workload("chunks", 16, 8, 128, 16, seed=10, extend_prefix_lens=[0], extend_ext_lens=[700],
                        device="cuda")
    o_full, l_full = run_gpu(w)
    e = w.extend
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    for lo, hi in ((0, 300), (300, 550), (550, 700)):
        n = hi - lo
        o, l = ops.attn_extend(pool, e.q[lo:hi].contiguous(), e.page_table,
                               torch.tensor([lo], dtype=torch.int32, device="cuda"),
                               torch.tensor([n], dtype=torch.int32, device="cuda"),
                               torch.tensor([0, n], dtype=torch.int32, device="cuda"), n, hi, w.scale)
        assert (o.float() - o_full[lo:hi].float()).abs().max().item() <= 1e-2
        assert (l - l_full[lo:hi]).abs().max().item() <= 1e-3
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o_full, ref_o, abs_ref=abs_ref(w))


def test_decode_equals_last_extend_row():
    w = W.make_workload("last", 40, 8, 128, 16, seed=11, extend_prefix_lens=[100, 0],
                        extend_ext_lens=[57, 300], device="cuda")
    o_e, l_e = run_gpu(w)
    e = w.extend
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    last = (e.cu_ext[1:] - 1).long()
    seq = (e.prefix_lens + e.ext_lens).int()
    o_d, l_d = ops.attn_decode(pool, e.q[last].contiguous(), e.page_table, seq, int(seq.max()), w.scale)
    assert (o_d.float() - o_e[last].float()).abs().max().item() <= 1e-2
    assert (l_d - l_e[last]).abs().max().item() <= 1e-3


def test_extend_without_positions():
    w = W.make_workload("nopos", 16, 8, 128, 1, seed=12, extend_prefix_lens=[3], extend_ext_lens=[40],
                        device="cuda")
    e = w.extend
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    o, lse = ops.attn_extend(pool, e.q, e.page_table, e.prefix_lens, e.ext_lens, e.cu_ext,
                             e.max_ext_len, e.max_seq_len, w.scale, positions=None)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("ps", [2, 4, 8, 32, 128])
@pytest.mark.parametrize("hq,hkv", [(24, 8), (48, 8), (56, 8), (12, 4)])
def test_extend_group_and_page_variants(ps, hq, hkv):
    """G = 3, 6, 7 (GQA padding rows in every Q tile) with gathered and tiled page paths."""
    pre = [0, 129, 63, 300]
    ext = [5, 250, 77, 131]
    w = W.make_workload("variants", hq, hkv, 128, ps, seed=ps * 7 + hq, extend_prefix_lens=pre,
                        extend_ext_lens=ext, device="cuda")
    status = ops.new_status()
    o, lse = run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, f"ps={ps} hq={hq}", abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("hq,hkv,ps", [(128, 8, 16), (64, 2, 1), (64, 1, 64), (48, 3, 16)])
def test_extend_more_than_eight_q_heads_per_kv_head(hq, hkv, ps):
    """G = 16, 32, 64 (a 128-row Q tile holds 8, 4 or 2 tokens) and an odd kv head count."""
    w = W.make_workload("wideg", hq, hkv, 128, ps, seed=hq + hkv + ps, extend_prefix_lens=[0, 37, 300],
                        extend_ext_lens=[19, 130, 64], device="cuda")
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, f"hq={hq} hkv={hkv} ps={ps}", abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("ext", [1, 2, 3, 7])
def test_extend_chunk_smaller_than_tile(ext):
    """Fewer tokens than one Q tile holds (the TMA box is clipped to the tokens that exist)."""
    w = W.make_workload("tiny", 16, 8, 128, 16, seed=40 + ext, extend_prefix_lens=[37],
                        extend_ext_lens=[ext], device="cuda")
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_extend_long_prefix_many_tiles():
    """A 16k-token cached prefix with a short chunk: many K/V tiles, ring wrap-around."""
    w = W.make_workload("longpre", 64, 8, 128, 64, seed=50, extend_prefix_lens=[16384, 3],
                        extend_ext_lens=[40, 200], device="cuda")
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("ps", [1, 4, 16, 32, 64])
def test_extend_bad_page_zeroes_affected_rows(ps):
    """A page id past the pool: status bit set; rows that would read it are zero, earlier rows exact.

    Page sizes below 16 take the cp.async copy path, 16 and up the TMA path; at 16 and 32
    the key tile holds whole pages copied as boxes and the bad page's rows gathered."""
    w = W.make_workload("badpage", 16, 8, 128, ps, seed=51, extend_prefix_lens=[64], extend_ext_lens=[100],
                        device="cuda")
    e = w.extend
    good_o, good_l = run_gpu(w)
    pt = e.page_table.clone()
    bad_page_idx = 112 // ps                           # first bad key 112 -> chunk rows i >= 48
    pt[0, bad_page_idx] = w.num_slots // ps + 3
    pool = ops.KVPool(w.k_pool, w.v_pool, ps)
    status = ops.new_status()
    o, lse = ops.attn_extend(pool, e.q, pt, e.prefix_lens, e.ext_lens, e.cu_ext, e.max_ext_len,
                             e.max_seq_len, w.scale, positions=e.positions, status=status)
    assert ops.read_status(status) & ops.DEVERR_PAGE_RANGE
    first_bad_row = bad_page_idx * ps - 64
    assert torch.all(o[first_bad_row:] == 0)
    assert torch.all(lse[first_bad_row:] == float("-inf"))
    assert torch.equal(o[:first_bad_row], good_o[:first_bad_row])


@pytest.mark.parametrize("ps", [1, 16])
def test_extend_zero_length_requests_and_graph_replay(ps):
    """Requests with no chunk tokens write nothing; a captured extend replays with new inputs."""
    w = W.make_workload("zero", 40, 8, 128, ps, seed=52, extend_prefix_lens=[10, 500, 0],
                        extend_ext_lens=[0, 70, 33], device="cuda")
    e = w.extend
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    o = torch.empty_like(e.q)
    lse = torch.empty(e.q.shape[:2], dtype=torch.float32, device="cuda")
    args = (pool, e.q, e.page_table, e.prefix_lens, e.ext_lens, e.cu_ext, e.max_ext_len, e.max_seq_len,
            w.scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.attn_extend(*args, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ops.attn_extend(*args, out=o, lse=lse)
    e.q.copy_(torch.randn_like(e.q.float()).to(torch.bfloat16))
    o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)
