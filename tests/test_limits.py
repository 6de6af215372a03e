"""The largest shapes the boundary accepts, against the oracle.

* 64 kv heads (a pool row of 16 KiB per slot, the most `num_kv_heads` may be), with one
  and with two q heads per kv head, on the store, the decode and the extend;
* 64 q heads per kv head (the largest G) at the largest page size, 256;
* a 2048-request decode batch (two thousand partial rows for the merge) and a decode
  over 131,072 keys (one request spread over every split CTA);
* a batch whose requests have one key each next to long ones.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_o_close
from tests import test_decode as TD
from tests import test_extend as TE

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hkv,ps", [(64, 64, 16), (128, 64, 1)])
def test_sixty_four_kv_heads(hq, hkv, ps):
    w = W.make_workload("hkv64", hq, hkv, 128, ps, seed=hq + ps, decode_seq_lens=[1, 300, 2049],
                        extend_prefix_lens=[0, 200], extend_ext_lens=[130, 77], device="cuda")
    # store: the new tokens' rows, written over zeros
    k_new, v_new, loc = w.new_tokens()
    ref_k = w.k_pool.clone()
    w.k_pool[loc.long()] = 0
    w.v_pool[loc.long()] = 0
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    status = ops.new_status()
    ops.store_kv(pool, k_new, v_new, loc, status=status)
    assert ops.read_status(status) == 0
    assert torch.equal(w.k_pool.view(torch.int16), ref_k.view(torch.int16))
    o, lse = TD.run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = TD.run_oracle(w)
    assert_o_close(o, ref_o, f"decode hq={hq} hkv={hkv}", abs_ref=TD.abs_ref(w))
    assert_lse_close(lse, ref_l)
    o, lse = TE.run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = TE.run_oracle(w)
    assert_o_close(o, ref_o, f"extend hq={hq} hkv={hkv}", abs_ref=TE.abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_largest_group_at_largest_page_size():
    w = W.make_workload("g64", 64, 1, 128, 256, seed=77, decode_seq_lens=[5, 256, 257, 3000],
                        extend_prefix_lens=[0, 512], extend_ext_lens=[300, 33], device="cuda")
    o, lse = TD.run_gpu(w)
    ref_o, ref_l = TD.run_oracle(w)
    assert_o_close(o, ref_o, "decode G=64 ps=256", abs_ref=TD.abs_ref(w))
    assert_lse_close(lse, ref_l)
    o, lse = TE.run_gpu(w)
    ref_o, ref_l = TE.run_oracle(w)
    assert_o_close(o, ref_o, "extend G=64 ps=256", abs_ref=TE.abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_decode_two_thousand_requests_with_one_key_neighbours():
    rng = np.random.default_rng(78)
    seqs = rng.integers(1, 300, size=2048)
    seqs[::9] = 1
    w = W.make_workload("b2048", 16, 8, 128, 1, seed=78, decode_seq_lens=seqs, device="cuda")
    status = ops.new_status()
    o, lse = TD.run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = TD.run_oracle(w)
    assert_o_close(o, ref_o, "B=2048", abs_ref=TD.abs_ref(w))
    assert_lse_close(lse, ref_l)


def test_decode_over_131072_keys():
    w = W.make_workload("k131k", 40, 8, 128, 64, seed=79, decode_seq_lens=[131072, 7], device="cuda")
    status = ops.new_status()
    o, lse = TD.run_gpu(w, status)
    assert ops.read_status(status) == 0
    ref_o, ref_l = TD.run_oracle(w)
    assert_o_close(o, ref_o, "131072 keys", abs_ref=TD.abs_ref(w))
    assert_lse_close(lse, ref_l)
