"""Shared parity helpers: GPU results against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output).  On the five
workloads the bar is the stated one: O max absolute error <= 1e-2, O mean
absolute error <= 1e-3, LSE max absolute error <= 1e-3.

Synthetic edge cases include rows that see only one to three keys, where
|o| can reach 4 or more, and peaked softmaxes (scales up to 1, rows that see
few keys), where one or two weights carry the row.  There the two roundings
the kernels make are larger than 1e-2 together, whatever the internal
precision:

* P is rounded to bf16 before the PV product (8 significant bits: relative
  error <= 2^-8 per weight), which moves o by at most 2^-8 * A,
  A = sum_j softmax_j |v_j| (the oracle's o with every V element replaced by
  its absolute value);
* o is rounded to bf16 once at the end: half a bf16 ulp at |o| + 2^-8 A.
  A bf16 number in [4, 8) has an ulp of 2^-5, so even the correctly rounded
  exact value can sit 2^-6 = 0.0156 away from it.

Tests of such cases pass ``abs_ref`` (= A) and allow, per element, the
larger of 1e-2 and half_ulp(|o| + pre) + pre with pre = 2^-8 (1 + 2^-10) A
(the 2^-10 covers fp32 accumulation and the approximate exp2).  The
worked examples, whose softmax weights are exact powers of two (so P rounds
exactly), pass ``rounding_aware=True`` for the output rounding alone
(pre = 0).  Wherever that sum is below 1e-2 (|o| < 2 with a spread-out
softmax, the usual case) the plain bound applies.  The mean bound of 1e-3
always holds.
"""
import numpy as np
import torch

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3
P_REL = 2.0 ** -8 * (1.0 + 2.0 ** -10)   # bf16 rounding of P, plus fp32 / exp2 slack


def bf16_half_ulp(x):
    """Half the spacing of bf16 numbers at RNE(x), elementwise (x float64)."""
    r = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()
    mant, exp = np.frexp(np.abs(r))          # |r| = mant * 2^exp, mant in [0.5, 1)
    # bf16 keeps 8 significant bits: ulp = 2^(exp - 8); subnormals and zero get the smallest spacing
    half = np.ldexp(1.0, np.maximum(exp, -125) - 9)
    return np.where(r == 0, np.ldexp(1.0, -134), half)


def o_bound(o_ref, rounding_aware=False, abs_ref=None):
    """Per-element bound on |o_gpu - o_ref|."""
    if abs_ref is None and not rounding_aware:
        return np.float64(O_MAX)
    pre = 0.0 if abs_ref is None else P_REL * np.asarray(abs_ref, np.float64)
    return np.maximum(O_MAX, bf16_half_ulp(np.abs(o_ref) + pre) + pre)


def assert_o_close(o_gpu, o_ref, what="", rounding_aware=False, abs_ref=None):
    o = o_gpu.double().cpu().numpy() if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu, np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    bound = o_bound(o_ref, rounding_aware, abs_ref)
    excess = err - bound
    i = np.unravel_index(excess.argmax(), err.shape)
    a = "" if abs_ref is None else f", A {np.asarray(abs_ref)[i]:.6g}"
    assert excess.max() <= 0, (f"{what}: O abs err {err[i]:.3e} above bound "
                               f"{np.broadcast_to(bound, err.shape)[i]:.3e} at {i} "
                               f"(gpu {o[i]:.6g}, exact {o_ref[i]:.6g}{a})")
    assert err.mean() <= O_MEAN, f"{what}: O mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def assert_lse_close(l_gpu, l_ref, what=""):
    l = l_gpu.double().cpu().numpy() if isinstance(l_gpu, torch.Tensor) else np.asarray(l_gpu, np.float64)
    err = np.abs(l - l_ref)
    assert np.isfinite(l).all(), f"{what}: non-finite lse"
    assert err.max() <= LSE_MAX, f"{what}: LSE max abs err {err.max():.3e}"
    return float(err.max())
