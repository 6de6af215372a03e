"""Shared parity helpers: GPU results against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output): on O the max
absolute error is at most 1e-2 and the mean absolute error at most 1e-3;
on the natural-log LSE the max absolute error is at most 1e-3.
"""
import numpy as np
import torch

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3


def assert_o_close(o_gpu, o_ref, what=""):
    o = o_gpu.double().cpu().numpy() if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu, np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX, f"{what}: O max abs err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert err.mean() <= O_MEAN, f"{what}: O mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def assert_lse_close(l_gpu, l_ref, what=""):
    l = l_gpu.double().cpu().numpy() if isinstance(l_gpu, torch.Tensor) else np.asarray(l_gpu, np.float64)
    err = np.abs(l - l_ref)
    assert np.isfinite(l).all(), f"{what}: non-finite lse"
    assert err.max() <= LSE_MAX, f"{what}: LSE max abs err {err.max():.3e}"
    return float(err.max())
