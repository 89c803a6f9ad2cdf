"""Tolerances and comparison helpers for CUDA-vs-oracle parity.

The bounds are the ones the target states for this library:
fp32 outputs max |dO| <= 1e-5; bf16 outputs max |dO| <= 2e-2 and mean
|dO| <= 2e-3; the log-sum-exp within 1e-3.  The oracle always reads the same
stored (rounded) inputs as the kernel, upcast to float64.
"""
import numpy as np
import torch

TOL_F32_MAX = 1e-5
TOL_BF16_MAX = 2e-2
TOL_BF16_MEAN = 2e-3
TOL_LSE = 1e-3


def f64(t):
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu")
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.float()
        return t.double().numpy()
    return np.asarray(t, dtype=np.float64)


def check_o(o_gpu, o_ref, dtype, what=""):
    a, b = f64(o_gpu), f64(o_ref)
    assert a.shape == b.shape, (a.shape, b.shape)
    assert np.isfinite(a).all(), f"{what}: non-finite output"
    err = np.abs(a - b)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    if dtype == torch.float32 or dtype == "f32":
        assert mx <= TOL_F32_MAX, f"{what}: fp32 max |dO| = {mx:.3e} > {TOL_F32_MAX}"
    else:
        assert mx <= TOL_BF16_MAX, f"{what}: bf16 max |dO| = {mx:.3e} > {TOL_BF16_MAX}"
        assert mean <= TOL_BF16_MEAN, f"{what}: bf16 mean |dO| = {mean:.3e} > {TOL_BF16_MEAN}"
    return mx, mean


def check_lse(lse_gpu, lse_ref, what=""):
    a, b = f64(lse_gpu), f64(lse_ref)
    both_inf = np.isneginf(a) & np.isneginf(b)
    assert (np.isneginf(a) == np.isneginf(b)).all(), f"{what}: -inf LSE pattern differs"
    d = np.abs(np.where(both_inf, 0.0, a) - np.where(both_inf, 0.0, b))
    mx = float(d.max()) if d.size else 0.0
    assert mx <= TOL_LSE, f"{what}: max |dLSE| = {mx:.3e} > {TOL_LSE}"
    return mx
