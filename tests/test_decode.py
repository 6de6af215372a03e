"""msgl_attn_decode against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def run_gpu(w, status=None):
    d = w.decode
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    return ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, d.max_seq_len, w.scale, status=status)


def run_oracle(w, rows=None, v_abs=False):
    """The oracle's (o, lse); with v_abs, o over |V| (the rounding allowance's A)."""
    d = w.decode
    kp, vp = w.k_pool.cpu(), w.v_pool.cpu()
    if v_abs:
        vp = vp.abs()
    if rows is None:
        return oracle.decode(d.q.cpu(), kp, vp, w.page_size, d.page_table.cpu(), d.seq_lens.cpu(), w.scale)
    # only the sampled requests, every q head
    rows = np.asarray(rows, dtype=np.int32)
    req = np.repeat(rows, w.hq)
    head = np.tile(np.arange(w.hq, dtype=np.int32), len(rows))
    pos = d.seq_lens.cpu().numpy()[req] - 1
    o, lse = oracle.attention_items(d.q.cpu(), kp, vp, w.page_size, d.page_table.cpu(), w.scale,
                                    req, req, pos, head)
    return o.reshape(len(rows), w.hq, w.d), lse.reshape(len(rows), w.hq)


def abs_ref(w, rows=None):
    return run_oracle(w, rows, v_abs=True)[0]


@pytest.mark.parametrize("cfg", [1, 3, 4, 5])
def test_decode_configs(cfg):
    w = W.config(cfg, device="cuda", part="decode")
    status = ops.new_status()
    o, lse = run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, f"config {cfg}")
    assert_lse_close(lse, ref_l, f"config {cfg}")


@pytest.mark.parametrize("ps", [1, 2, 8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (40, 8), (64, 8), (4, 1), (10, 2), (32, 16), (48, 24)])
def test_decode_shapes(ps, hq, hkv):
    seqs = [1, 2, ps - 1 if ps > 1 else 3, ps, ps + 1, 2 * ps + 3, 77, 1000, 4099]
    w = W.make_workload("shapes", hq, hkv, 128, ps, seed=ps * 100 + hq, decode_seq_lens=seqs, device="cuda")
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, f"ps={ps} hq={hq} hkv={hkv}", abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("hq,hkv,ps", [(128, 8, 16), (32, 2, 1), (48, 2, 64), (64, 1, 16), (24, 12, 16), (12, 3, 1)])
def test_decode_more_than_eight_q_heads_per_kv_head(hq, hkv, ps):
    """G > 8 (several consumer warps per kv head, smaller head groups) and kv head counts that
    are neither <= 8 nor multiples of 8."""
    seqs = [1, 40, 333, 1500, 2049]
    w = W.make_workload("wideg", hq, hkv, 128, ps, seed=hq * 7 + hkv + ps, decode_seq_lens=seqs, device="cuda")
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, f"hq={hq} hkv={hkv} ps={ps}", abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_decode_large_batch_graph_replay():
    """A 192-request batch (split and merge under programmatic dependent launch) captured in a
    CUDA graph and replayed with new lengths."""
    seqs = [4000, 3500, 2900, 4096, 1200, 3900, 4096, 2500] * 24
    w = W.make_workload("poolgraph", 40, 8, 128, 16, seed=23, decode_seq_lens=seqs, device="cuda")
    d = w.decode
    pool = ops.KVPool(w.k_pool, w.v_pool, 16)
    ws = torch.empty(ops.decode_workspace_size(d.num_reqs, w.hq, w.hkv, 4096), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(d.q)
    lse = torch.empty(d.q.shape[:2], dtype=torch.float32, device="cuda")
    status = ops.new_status()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, 4096, w.scale, out=o, lse=lse, workspace=ws,
                        status=status)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, 4096, w.scale, out=o, lse=lse, workspace=ws,
                        status=status)
    full = d.seq_lens.clone()
    for trial in range(2):
        # new lengths within each request's pages
        frac = torch.rand(full.shape, device="cuda")
        d.seq_lens.copy_(torch.clamp((full.float() * frac).to(torch.int32), min=1))
        o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert ops.read_status(status) == 0
        rows = list(range(0, d.num_reqs, 17)) + [d.num_reqs - 1]
        ref_o, ref_l = run_oracle(w, rows)
        assert_o_close(o[rows], ref_o, f"replay {trial}")
        assert_lse_close(lse[rows], ref_l)


def test_decode_long_single_request():
    """One 65k-token request: many key chunks merged by LSE."""
    w = W.make_workload("long", 16, 8, 128, 16, seed=3, decode_seq_lens=[65536], device="cuda")
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_decode_uniform_values_and_large_scores():
    """Inputs with larger magnitudes (scores of tens) still match."""
    w = W.make_workload("big", 16, 8, 128, 1, seed=4, decode_seq_lens=[300, 17, 2000], device="cuda")
    w.decode.q.mul_(4)
    o, lse = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_decode_batch_equals_single():
    """A request's result does not depend on the other requests in the batch."""
    w = W.make_workload("batch", 40, 8, 128, 16, seed=6, decode_seq_lens=[500, 3000, 45, 1200],
                        device="cuda")
    o, lse = run_gpu(w)
    d = w.decode
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    for b in range(4):
        o1, l1 = ops.attn_decode(pool, d.q[b:b + 1].contiguous(), d.page_table[b:b + 1].contiguous(),
                                 d.seq_lens[b:b + 1].contiguous(), int(d.seq_lens[b]), w.scale)
        ref_o, ref_l = run_oracle(w, rows=[b])
        a = abs_ref(w, rows=[b])
        assert_o_close(o1, ref_o, abs_ref=a)
        assert_o_close(o[b:b + 1], ref_o, abs_ref=a)


def test_decode_graph_capture_replay():
    """The launch shape depends only on host scalars, so a captured decode replays correctly."""
    w = W.make_workload("graph", 16, 8, 128, 16, seed=8, decode_seq_lens=[1000, 900, 512], device="cuda")
    d = w.decode
    d.seq_lens.copy_(torch.tensor([100, 900, 33], dtype=torch.int32))
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    o = torch.empty_like(d.q)
    lse = torch.empty(d.q.shape[:2], dtype=torch.float32, device="cuda")
    ws_n = ops.decode_workspace_size(3, 16, 8, 1024)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, 1024, w.scale, out=o, lse=lse, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, 1024, w.scale, out=o, lse=lse, workspace=ws)
    o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    # new lengths, same graph: the kernels read seq_lens from device memory
    d.seq_lens.copy_(torch.tensor([1000, 1, 512], dtype=torch.int32))
    graph.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = run_oracle(w)
    assert_o_close(o, ref_o, abs_ref=abs_ref(w))
    assert_lse_close(lse, ref_l)
