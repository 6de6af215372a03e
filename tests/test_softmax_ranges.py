"""Softmax ranges on the GPU against the oracle.

* Scores that keep growing along the sequence: every few K/V tiles a row's running
  maximum rises by more than the extend kernel's lazy-rescale threshold (2^8), so the
  accumulated O is rescaled again and again; in the decode the online softmax moves its
  maximum on every tile.
* Scores that only fall: the maximum is set by the first keys and never moves.
* Softmax scales other than 1/sqrt(head_dim) (the scale is a call argument).

Both ramps come from one workload: key j's K row gets u_g * slope * (j + 1) added, with
u_g a random unit vector per kv head, so rows whose query points along u_g see rising
scores and the others falling ones.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W
from tests import test_decode as TD
from tests import test_extend as TE
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu

# about 2.4 (in log2 units) of score growth per 128 keys for a query with <q, u> = 1,
# so a rising row passes the 2^8 rescale threshold every three to four tiles
SLOPE = 0.15


def add_key_ramp(w, page_table, seq_lens, seed):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    u = torch.randn(w.hkv, w.d, generator=gen, dtype=torch.float64)
    u /= u.norm(dim=1, keepdim=True)
    pt = page_table.cpu().numpy()
    ps = w.page_size
    for b, n in enumerate(seq_lens):
        j = np.arange(int(n))
        slots = torch.from_numpy(pt[b][j // ps] * ps + j % ps).long().to(w.k_pool.device)
        ramp = torch.from_numpy(SLOPE * (j + 1.0)).to(w.k_pool.device)
        k = w.k_pool[slots].double() + ramp[:, None, None] * u.to(w.k_pool.device)[None]
        w.k_pool[slots] = k.to(torch.bfloat16)


def rising_and_falling_rows(q, w, u_seed):
    """Count (row, head) pairs whose query has a positive / negative component along u."""
    gen = torch.Generator(device="cpu").manual_seed(u_seed)
    u = torch.randn(w.hkv, w.d, generator=gen, dtype=torch.float64)
    u /= u.norm(dim=1, keepdim=True)
    G = w.hq // w.hkv
    proj = torch.einsum("thd,hd->th", q.cpu().double(), u.repeat_interleave(G, 0))
    return int((proj > 0.5).sum()), int((proj < -0.5).sum())


@pytest.mark.parametrize("ps", [1, 16, 64])
def test_extend_rising_and_falling_scores(ps):
    w = W.make_workload("ramp", 64, 8, 128, ps, seed=71, extend_prefix_lens=[704, 0, 1536],
                        extend_ext_lens=[320, 900, 192], device="cuda")
    e = w.extend
    seq = (e.prefix_lens + e.ext_lens).cpu().numpy()
    add_key_ramp(w, e.page_table, seq, seed=5)
    up, down = rising_and_falling_rows(e.q, w, 5)
    assert up > 1000 and down > 1000
    status = ops.new_status()
    o, lse = TE.run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = TE.run_oracle(w)
    # rising rows end far above where they started
    assert ref_l.max() - ref_l.min() > 30
    assert_o_close(o, ref_o, f"ramp ps {ps}", abs_ref=TE.abs_ref(w))
    assert_lse_close(lse, ref_l, f"ramp ps {ps}")


@pytest.mark.parametrize("ps", [1, 64])
def test_decode_rising_and_falling_scores(ps):
    w = W.make_workload("ramp", 40, 8, 128, ps, seed=72, decode_seq_lens=[2100, 300, 2500, 17],
                        device="cuda")
    d = w.decode
    add_key_ramp(w, d.page_table, d.seq_lens.cpu().numpy(), seed=6)
    status = ops.new_status()
    o, lse = TD.run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = TD.run_oracle(w)
    assert ref_l.max() - ref_l.min() > 30
    assert_o_close(o, ref_o, f"decode ramp ps {ps}", abs_ref=TD.abs_ref(w))
    assert_lse_close(lse, ref_l, f"decode ramp ps {ps}")


@pytest.mark.parametrize("scale", [0.03, 0.3, 1.0])
def test_scales_other_than_inverse_sqrt_head_dim(scale):
    w = W.make_workload("scale", 16, 8, 128, 16, seed=73, extend_prefix_lens=[200, 0],
                        extend_ext_lens=[150, 260], decode_seq_lens=[333, 1000], device="cuda")
    w.scale = scale
    o, lse = TE.run_gpu(w)
    ref_o, ref_l = TE.run_oracle(w)
    assert_o_close(o, ref_o, f"extend scale {scale}", abs_ref=TE.abs_ref(w))
    assert_lse_close(lse, ref_l, f"extend scale {scale}")
    o, lse = TD.run_gpu(w)
    ref_o, ref_l = TD.run_oracle(w)
    assert_o_close(o, ref_o, f"decode scale {scale}", abs_ref=TD.abs_ref(w))
    assert_lse_close(lse, ref_l, f"decode scale {scale}")
