"""Writes tests/golden/worked_examples.json: small paged-attention cases with exact answers.

The pages describe the computation in words and print no worked example.  A
query row at absolute position p attends keys 0..p of its request.  Those
keys are the pool history plus the chunk's new tokens, found through the
request's page table ("不懂SGLang？从miniSGLang开始" §1.3; "Mini-SGLang
实战指南" §6.1, §6.2).  The cases are built so that the softmax has a closed
form:

* every q head h has q = (c_h, 0, ..., 0) with c_h an integer;
* key j of kv head g has k = (a_j, 0, ..., 0) with a_j an integer;
* scale = ln 2.

So the score is c_h a_j ln 2 and the weight is exactly 2^(c_h a_j).  Then
o = sum_j 2^(c_h a_j) v_j / sum_j 2^(c_h a_j) and lse = ln sum_j 2^(c_h a_j).
Every input is exactly representable in bf16.  Expected values are exact
fractions (Python ``fractions``) rounded once to float.  This script imports
neither the oracle nor the CUDA library, and its inputs are fixed literals,
not random.  Rerun it to regenerate the fixture.
"""
import json
import math
import os
from fractions import Fraction


def solve(seq_len, prefix_len, hq, hkv, c, a, v):
    """Exact o/lse for rows at positions prefix_len..seq_len-1 of one request."""
    G = hq // hkv
    o_rows, lse_rows = [], []
    for pos in range(prefix_len, seq_len):
        o_h, l_h = [], []
        for h in range(hq):
            g = h // G
            w = [Fraction(2) ** (c[h] * a[g][j]) for j in range(pos + 1)]
            z = sum(w)
            d = len(v[g][0])
            o_h.append([float(sum(w[j] * Fraction(v[g][j][e]) for j in range(pos + 1)) / z)
                        for e in range(d)])
            l_h.append(math.log(z.numerator) - math.log(z.denominator))
        o_rows.append(o_h)
        lse_rows.append(l_h)
    return o_rows, lse_rows


def case(name, page_size, num_pages, hq, hkv, c, requests):
    """requests: list of dicts with seq_len, prefix_len, pages, a [Hkv][seq], v [Hkv][seq][d]."""
    out = {"name": name, "page_size": page_size, "num_pages": num_pages, "hq": hq, "hkv": hkv,
           "c": c, "scale": "ln2", "requests": []}
    for r in requests:
        o, lse = solve(r["seq_len"], r["prefix_len"], hq, hkv, c, r["a"], r["v"])
        out["requests"].append(dict(r, expected_o=o, expected_lse=lse))
    return out


def main():
    cases = []
    # One request, one head, three keys on pages 3 then 1 (page size 2); a = 0, 1, 2 gives
    # weights 1, 2, 4, so o = (1, 2, 4, 2 - 4 + 2) / 7 and lse = ln 7.
    cases.append(case("three_keys_paged", 2, 4, 1, 1, [1], [
        dict(seq_len=3, prefix_len=2, pages=[3, 1], a=[[0, 1, 2]],
             v=[[[1, 0, 0, 2], [0, 1, 0, -2], [0, 0, 1, 0.5]]])]))
    # Two requests, 4 q heads on 2 kv heads, page size 4.  Both start with the same page 6
    # (a shared cached prefix); request 0 decodes one row, request 1 extends three rows
    # causally.  c = 1, 2, 0, -1 gives sharp, sharper, uniform and reversed weights.
    k0 = [3, 0, 1, 0]
    k1 = [1, 1, 1, 1]
    v0 = [[j - 1.5, 0.25 * j, 1.0, -1.0] for j in range(4)]
    v1 = [[0.5, j, -j, 2.0] for j in range(4)]
    cases.append(case("gqa_shared_page", 4, 8, 4, 2, [1, 2, 0, -1], [
        dict(seq_len=5, prefix_len=4, pages=[6, 2],
             a=[k0 + [2], k1 + [1]],
             v=[v0 + [[4.0, -4.0, 0.5, 0.0]], v1 + [[1.0, 1.0, 1.0, 1.0]]]),
        dict(seq_len=7, prefix_len=4, pages=[6, 5],
             a=[k0 + [0, 5, -2], k1 + [0, 0, 3]],
             v=[v0 + [[2.0, 2.0, 2.0, 2.0], [-1.0, 0.0, 1.0, 0.0], [0.0, 8.0, 0.0, -8.0]],
                v1 + [[0.0, 0.0, 0.0, 0.0], [4.0, 4.0, -4.0, 1.0], [-0.5, 0.5, 3.0, -3.0]]])]))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "worked_examples.json")
    with open(path, "w") as f:
        json.dump({"source": "closed forms of softmax attention with power-of-two weights, "
                             "written by make_worked_examples.py",
                   "cases": cases}, f, indent=1)
    print(path)


if __name__ == "__main__":
    main()
