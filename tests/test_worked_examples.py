"""Hand-solvable worked examples (tests/golden/worked_examples.json).

The pages print no numeric example, so these fixtures are built so that the
softmax has a closed form: every score is an integer multiple of ln 2 and
every weight an exact power of two (tests/golden/make_worked_examples.py
explains the construction and computes the answers with exact fractions,
without the oracle or the CUDA library).  They pin the paged lookup (keys on
non-contiguous pages, a page shared by two requests), the grouped-query head
mapping (4 q heads on 2 kv heads), causal extend rows, and the decode row.

The oracle must reproduce them to fp64 rounding; the CUDA path must meet the
usual parity bar.  The CUDA kernels take head_dim 128, so the 4-wide vectors
are zero-padded; zero components change neither score nor output.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.parity import assert_lse_close, assert_o_close

_FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")


def _cases():
    with open(_FIXTURE) as f:
        return json.load(f)["cases"]


CASES = _cases()
IDS = [c["name"] for c in CASES]


def materialise(c, d):
    """Pool, queries and expected values of one case, vectors padded to width d."""
    ps, npages, hq, hkv = c["page_size"], c["num_pages"], c["hq"], c["hkv"]
    reqs = c["requests"]
    k_pool = torch.full((npages * ps, hkv, d), float("nan"), dtype=torch.float64)
    v_pool = torch.full((npages * ps, hkv, d), float("nan"), dtype=torch.float64)
    width = max(len(r["pages"]) for r in reqs)
    table = torch.zeros((len(reqs), width), dtype=torch.int32)
    q_rows, o_rows, l_rows = [], [], []
    for b, r in enumerate(reqs):
        table[b, :len(r["pages"])] = torch.tensor(r["pages"], dtype=torch.int32)
        for j in range(r["seq_len"]):
            slot = r["pages"][j // ps] * ps + j % ps
            for g in range(hkv):
                k_pool[slot, g] = 0.0
                k_pool[slot, g, 0] = r["a"][g][j]
                v_pool[slot, g] = 0.0
                v_pool[slot, g, :len(r["v"][g][j])] = torch.tensor(r["v"][g][j], dtype=torch.float64)
        for i in range(r["seq_len"] - r["prefix_len"]):
            q = torch.zeros((hq, d), dtype=torch.float64)
            q[:, 0] = torch.tensor(c["c"], dtype=torch.float64)
            q_rows.append(q)
            o = np.zeros((hq, d))
            o[:, :4] = np.asarray(r["expected_o"][i])
            o_rows.append(o)
            l_rows.append(np.asarray(r["expected_lse"][i]))
    return dict(
        k_pool=k_pool.to(torch.bfloat16), v_pool=v_pool.to(torch.bfloat16),
        q=torch.stack(q_rows).to(torch.bfloat16), page_table=table,
        prefix=torch.tensor([r["prefix_len"] for r in reqs], dtype=torch.int32),
        ext=torch.tensor([r["seq_len"] - r["prefix_len"] for r in reqs], dtype=torch.int32),
        o=np.stack(o_rows), lse=np.stack(l_rows), scale=math.log(2.0), page_size=ps)


def test_fixture_first_case_by_hand():
    """Weights 1, 2, 4 over three keys: o = (1, 2, 4, 0) / 7 and lse = ln 7, worked by hand."""
    r = CASES[0]["requests"][0]
    np.testing.assert_allclose(r["expected_o"][0][0], [1 / 7, 2 / 7, 4 / 7, 0.0], rtol=0, atol=1e-15)
    assert abs(r["expected_lse"][0][0] - math.log(7.0)) < 1e-15


@pytest.mark.parametrize("d", [4, 128])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_oracle_extend_reproduces_worked_examples(case, d):
    m = materialise(case, d)
    o, lse = oracle.extend(m["q"], m["k_pool"], m["v_pool"], m["page_size"], m["page_table"],
                           m["prefix"], m["ext"], m["scale"])
    np.testing.assert_allclose(o, m["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, m["lse"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_oracle_decode_reproduces_last_rows(case):
    """The decode row of each request is its extend row at position seq_len - 1."""
    m = materialise(case, 4)
    last = np.cumsum(m["ext"].numpy()) - 1
    seq = m["prefix"] + m["ext"]
    o, lse = oracle.decode(m["q"][last], m["k_pool"], m["v_pool"], m["page_size"], m["page_table"],
                           seq, m["scale"])
    np.testing.assert_allclose(o, m["o"][last], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, m["lse"][last], rtol=0, atol=1e-12)


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_cuda_extend_and_decode_worked_examples(case):
    from paged_kv_attention_24_gb300 import ops
    m = materialise(case, 128)
    dev = "cuda"
    pool = ops.KVPool(m["k_pool"].to(dev), m["v_pool"].to(dev), m["page_size"])
    table = m["page_table"].to(dev)
    ext = m["ext"]
    cu = torch.zeros(len(ext) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(ext, 0)
    positions = torch.cat([torch.arange(int(p), int(p) + int(e), dtype=torch.int32)
                           for p, e in zip(m["prefix"], ext)])
    seq = m["prefix"] + ext
    status = ops.new_status()
    o, lse = ops.attn_extend(pool, m["q"].to(dev), table, m["prefix"].to(dev), ext.to(dev), cu.to(dev),
                             int(ext.max()), int(seq.max()), m["scale"], positions=positions.to(dev),
                             status=status)
    assert ops.read_status(status) == 0
    assert_o_close(o, m["o"], f"{case['name']} extend", rounding_aware=True)
    assert_lse_close(lse, m["lse"], f"{case['name']} extend")
    last = (cu[1:] - 1).long()
    o, lse = ops.attn_decode(pool, m["q"][last].to(dev), table, seq.to(dev), int(seq.max()), m["scale"],
                             status=status)
    assert ops.read_status(status) == 0
    assert_o_close(o, m["o"][last.numpy()], f"{case['name']} decode", rounding_aware=True)
    assert_lse_close(lse, m["lse"][last.numpy()], f"{case['name']} decode")


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 7, 8])
def test_planted_oracle_mistakes_miss_worked_examples(mutant):
    """Each planted oracle mistake (see test_oracle_mutants) misses at least one worked example."""
    missed = False
    for c in CASES:
        m = materialise(c, 4)
        try:
            o, lse = oracle.extend(m["q"], m["k_pool"], m["v_pool"], m["page_size"], m["page_table"],
                                   m["prefix"], m["ext"], m["scale"], mutant=mutant)
        except oracle.OracleError:
            missed = True
            continue
        if not (np.allclose(o, m["o"], rtol=0, atol=1e-9) and np.allclose(lse, m["lse"], rtol=0, atol=1e-9)):
            missed = True
    assert missed, f"planted mistake {mutant} reproduces every worked example"
