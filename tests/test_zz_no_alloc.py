"""The allocation-free decode entry point: same results, no allocation, clear rejection.

msgl_attn_decode_noalloc serves callers that cannot allocate device memory
(engines whose device memory is all planned by a host pool, plugin-style
interfaces that only hand over input and output pointers, loops that cannot
pay for cudaMalloc's implicit synchronisation).  It takes its split scratch
from a static array inside the library.  Here it is called twice in a row,
on two different batches (once through the raw C ABI, once through the
Python binding), and each result is compared with the fp64 oracle and with
msgl_attn_decode's on the same inputs, within the parity tolerances used by
every other test.  A batch too large for the built-in scratch must be
refused before anything is launched.  This file is named to be collected
last.
"""
import ctypes

import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_o_close

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3
MSGL_ERR_WORKSPACE = 6

pytestmark = pytest.mark.gpu


def _raw_noalloc(pool, w, out, lse, status):
    d = w.decode
    pc, pt = pool.c(), ops._pages(d.page_table)
    return ops.load().msgl_attn_decode_noalloc(
        ctypes.byref(pc), ctypes.byref(pt), ctypes.c_void_p(d.q.data_ptr()), w.hq,
        ctypes.c_void_p(d.seq_lens.data_ptr()), d.num_reqs, d.max_seq_len, w.scale,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _compare(w, through_binding):
    d = w.decode
    assert ops.decode_workspace_size(d.num_reqs, w.hq, w.hkv, d.max_seq_len) <= ops.NOALLOC_SCRATCH_BYTES
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    ws_o, ws_l = ops.attn_decode(pool, d.q, d.page_table, d.seq_lens, d.max_seq_len, w.scale)
    out = torch.full_like(d.q, float("nan"))
    lse = torch.full(d.q.shape[:2], float("nan"), dtype=torch.float32, device=d.q.device)
    status = ops.new_status()
    if through_binding:
        ops.attn_decode_noalloc(pool, d.q, d.page_table, d.seq_lens, d.max_seq_len, w.scale,
                                out=out, lse=lse, status=status)
    else:
        rc = _raw_noalloc(pool, w, out, lse, status)
        assert rc == 0, ops.load().msgl_last_error()
    assert ops.read_status(status) == 0
    assert torch.isfinite(out.float()).all()
    err = (out.float() - ws_o.float()).abs()
    assert err.max().item() <= O_MAX and err.mean().item() <= O_MEAN
    assert (lse - ws_l).abs().max().item() <= LSE_MAX
    ref_o, ref_l = oracle.decode(d.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(), w.page_size,
                                 d.page_table.cpu(), d.seq_lens.cpu(), w.scale)
    assert_o_close(out, ref_o, f"{w.name} no-alloc")
    assert_lse_close(lse, ref_l, f"{w.name} no-alloc")


def test_noalloc_matches_oracle_and_workspace_decode_twice():
    # first call: many long requests (large scratch use); second: a different, smaller batch,
    # so leftovers from the first call would show up in the second
    w1 = W.make_workload("na1", 64, 8, 128, 64, seed=21, decode_seq_lens=[8192, 1024, 5000, 7777] * 4,
                         device="cuda")
    w2 = W.make_workload("na2", 16, 8, 128, 1, seed=22, decode_seq_lens=[3000, 17, 1500], device="cuda")
    _compare(w1, through_binding=False)
    _compare(w2, through_binding=True)


def test_noalloc_allocates_nothing_after_first_call():
    """After the first call on the device (which may load the module), a call changes neither
    torch's allocator counters nor the device's free memory."""
    w = W.make_workload("na3", 40, 8, 128, 16, seed=23, decode_seq_lens=[700, 2000, 31], device="cuda")
    d = w.decode
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    out = torch.empty_like(d.q)
    lse = torch.empty(d.q.shape[:2], dtype=torch.float32, device=d.q.device)
    status = ops.new_status()
    ops.attn_decode_noalloc(pool, d.q, d.page_table, d.seq_lens, d.max_seq_len, w.scale, out=out, lse=lse,
                            status=status)
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0])
    for _ in range(3):
        ops.attn_decode_noalloc(pool, d.q, d.page_table, d.seq_lens, d.max_seq_len, w.scale, out=out,
                                lse=lse, status=status)
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0])
    assert after == before
    assert ops.read_status(status) == 0


def test_noalloc_rejects_batch_beyond_scratch():
    """600 requests x 64 q heads need (600 + 512) * 64 * 516 bytes > 32 MiB: refused with
    MSGL_ERR_WORKSPACE, both sizes in the message, nothing launched."""
    B, hq, hkv = 600, 64, 8
    need = ops.decode_workspace_size(B, hq, hkv, 4096)
    assert need == (B + 512) * hq * 516 and need > ops.NOALLOC_SCRATCH_BYTES
    w = W.make_workload("na4", hq, hkv, 128, 64, seed=24, decode_seq_lens=[64] * B, device="cuda")
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    out = torch.full_like(w.decode.q, 7.0)
    lse = torch.full(w.decode.q.shape[:2], 7.0, dtype=torch.float32, device="cuda")
    status = ops.new_status()
    d = w.decode
    pc, pt = pool.c(), ops._pages(d.page_table)
    rc = ops.load().msgl_attn_decode_noalloc(
        ctypes.byref(pc), ctypes.byref(pt), ctypes.c_void_p(d.q.data_ptr()), hq,
        ctypes.c_void_p(d.seq_lens.data_ptr()), B, 4096, w.scale, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == MSGL_ERR_WORKSPACE
    msg = ops.load().msgl_last_error().decode()
    assert str(need) in msg and str(ops.NOALLOC_SCRATCH_BYTES) in msg, msg
    with pytest.raises(ops.MsglError):
        ops.attn_decode_noalloc(pool, d.q, d.page_table, d.seq_lens, 4096, w.scale, out=out, lse=lse,
                                status=status)
    torch.cuda.synchronize()
    assert (out == 7.0).all() and (lse == 7.0).all()
    assert ops.read_status(status) == 0
