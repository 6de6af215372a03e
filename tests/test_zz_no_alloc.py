"""The allocation-free decode entry point matches the workspace one.

msgl_attn_decode_noalloc serves callers that cannot allocate device memory
(engines whose device memory is all planned by a host pool, plugin-style
interfaces that only hand over input and output pointers, loops that cannot
pay for cudaMalloc's implicit synchronisation).  It takes its split scratch
from a static array inside the library.  Here it is called through the C
ABI twice in a row, on two different batches, and each result is compared
with msgl_attn_decode's on the same inputs, within the parity tolerances
used by every other test.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3

pytestmark = pytest.mark.gpu


def _compare(w):
    d = w.decode
    assert ops.decode_workspace_size(d.num_reqs, w.hq, w.hkv, d.max_seq_len) > 0, \
        "the case must need split scratch"
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    ref_o, ref_l = ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, d.max_seq_len, w.scale)
    out = torch.full_like(d.q, float("nan"))
    lse = torch.full(d.q.shape[:2], float("nan"), dtype=torch.float32, device=d.q.device)
    status = ops.new_status()
    pc, pt = pool.c(), ops._pages(d.page_table)
    rc = ops.load().msgl_attn_decode_noalloc(
        ctypes.byref(pc), ctypes.byref(pt), ctypes.c_void_p(d.q.data_ptr()), w.hq,
        ctypes.c_void_p(d.seq_lens.data_ptr()), d.num_reqs, d.max_seq_len, w.scale,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, ops.load().msgl_last_error()
    assert ops.read_status(status) == 0
    err = (out.float() - ref_o.float()).abs()
    assert torch.isfinite(out.float()).all()
    assert err.max().item() <= O_MAX and err.mean().item() <= O_MEAN
    assert (lse - ref_l).abs().max().item() <= LSE_MAX


def test_noalloc_matches_workspace_decode_twice():
    # first call: many long requests (large scratch use); second: a different, smaller batch,
    # so leftovers from the first call would show up in the second
    w1 = W.make_workload("na1", 64, 8, 128, 64, seed=21, decode_seq_lens=[8192, 1024, 5000, 7777] * 4,
                         device="cuda")
    w2 = W.make_workload("na2", 16, 8, 128, 1, seed=22, decode_seq_lens=[3000, 17, 1500], device="cuda")
    _compare(w1)
    _compare(w2)
