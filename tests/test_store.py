"""msgl_store_kv against the oracle's scatter: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import ops

pytestmark = pytest.mark.gpu


def _case(S, hkv, n, seed):
    g = torch.Generator().manual_seed(seed)
    kp = torch.randn(S, hkv, 128, generator=g).to(torch.bfloat16)
    vp = torch.randn(S, hkv, 128, generator=g).to(torch.bfloat16)
    kp[::7] = float("nan")                      # poison: stored bits must pass through unchanged
    kn = torch.randn(n, hkv, 128, generator=g).to(torch.bfloat16)
    vn = torch.randn(n, hkv, 128, generator=g).to(torch.bfloat16)
    kn[::5, 0, :3] = float("inf")
    loc = torch.from_numpy(np.random.default_rng(seed).permutation(S)[:n].astype(np.int32))
    return kp, vp, kn, vn, loc


@pytest.mark.parametrize("S,hkv,n", [(4096, 8, 0), (4096, 8, 1), (4096, 8, 4), (16384, 8, 8192 + 64),
                                     (1024, 1, 1000), (2048, 2, 333), (512, 4, 17), (4096, 16, 2048)])
def test_store_bit_exact(S, hkv, n):
    kp, vp, kn, vn, loc = _case(S, hkv, n, seed=S + hkv + n)
    ko, vo = oracle.store_kv(kp, vp, kn, vn, loc)
    gk, gv = kp.cuda(), vp.cuda()
    pool = ops.KVPool(gk, gv, 1)
    status = ops.new_status()
    ops.store_kv(pool, kn.cuda(), vn.cuda(), loc.cuda(), status=status)
    assert ops.read_status(status) == 0
    assert np.array_equal(oracle._bits(gk.cpu()), ko)
    assert np.array_equal(oracle._bits(gv.cpu()), vo)


def test_store_config5_step():
    """The full mixed step of the Qwen3-32B workload: 8192 chunk tokens + 64 decode tokens, ps 64."""
    from paged_kv_attention_24_gb300 import workloads as W
    w = W.config(5, device="cuda")
    k_new, v_new, loc = w.new_tokens()
    before_k = w.k_pool.clone()
    w.k_pool[loc.long()] = 0
    w.v_pool[loc.long()] = 0
    pool = ops.KVPool(w.k_pool, w.v_pool, w.page_size)
    ops.store_kv(pool, k_new, v_new, loc)
    torch.cuda.synchronize()
    assert torch.equal(w.k_pool.view(torch.int16), before_k.view(torch.int16))
