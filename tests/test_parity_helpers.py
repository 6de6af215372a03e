"""The rounding-aware O bound equals half the bf16 spacing at the rounded exact value.

Checked against torch.nextafter in bfloat16 (a library routine independent of the
helper's frexp arithmetic), over values spanning many binades, signs, exact powers
of two and zero.
"""
import numpy as np
import torch

from tests.parity import O_MAX, bf16_half_ulp, o_bound


def _spacing_above(x):
    r = torch.from_numpy(x).to(torch.bfloat16)
    mag = r.abs()
    up = torch.nextafter(mag, torch.full_like(mag, float("inf")))
    return ((up.double() - mag.double()) / 2).numpy()


def test_half_ulp_matches_nextafter():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.uniform(-6, 4, 5000),
                        [0.0, 1.0, 2.0, 4.0, -4.0, 8.0, 3.99, 4.01, 1e-30, -7.999]])
    np.testing.assert_array_equal(bf16_half_ulp(x), _spacing_above(x))


def test_bound_only_widens_at_four_and_above():
    x = np.array([0.0, 1.0, 1.999, 2.0, 3.98, 3.999, 4.0, 5.0, 8.0, -6.0])
    b = o_bound(x, rounding_aware=True)
    assert (b[np.abs(x) < 3.99] == O_MAX).all()   # half ulp <= 2^-8 < 1e-2 below 4
    assert b[6] == 2.0 ** -6 and b[8] == 2.0 ** -5 and b[9] == 2.0 ** -6
    assert o_bound(x) == O_MAX


def test_bound_with_p_rounding_term():
    """With A (the oracle's o over |V|), the allowance adds 2^-8 (1 + 2^-10) A to the
    output half ulp taken at |o| + that term, and never drops below 1e-2."""
    from tests.parity import P_REL
    o = np.array([0.1, 2.9, 3.99, -5.0, 0.0])
    a = np.array([0.2, 3.0, 3.99, 5.0, 9.0])
    b = o_bound(o, abs_ref=a)
    pre = P_REL * a
    np.testing.assert_array_equal(b, np.maximum(O_MAX, bf16_half_ulp(np.abs(o) + pre) + pre))
    assert b[0] == O_MAX
    assert b[1] == 2.0 ** -7 + pre[1]            # 2.9 + 0.0117 stays in [2, 4)
    assert b[2] == 2.0 ** -6 + pre[2]            # 3.99 + 0.0156 crosses into [4, 8)
    assert P_REL == 2.0 ** -8 * (1 + 2.0 ** -10)


def test_bf16_relative_rounding_error_is_two_to_minus_eight():
    """The P term's constant: RNE to bf16 moves a value by at most 2^-8 of itself, and
    values just above a power of two come within a hair of it."""
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(1, 2, 200000), [1.0 + 2.0 ** -8 + 1e-9, 128.5 + 1e-6]])
    r = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    rel = np.abs(r - x) / x
    assert rel.max() <= 2.0 ** -8
    assert rel.max() > 0.99 * 2.0 ** -8
