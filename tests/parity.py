"""Tolerances and comparison helpers for CUDA-vs-oracle parity.

The bounds are the ones the target states for this library:
fp32 outputs max |dO| <= 1e-5; bf16 outputs max |dO| <= 2e-2 and mean
|dO| <= 2e-3; the log-sum-exp within 1e-3.  The oracle always reads the same
stored (rounded) inputs as the kernel, upcast to float64.
"""
import math

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


def fp8_bound(P, O_ref, q_hat_rows, k_hat, v_hat, v_scale, *, scale, block=128):
    """Bound on |O_fp8 - O_ref| per element for FP8 attention over dequantised blocks.

    Inputs come from the oracle: P [n, Nk] the softmax weights of n query rows
    (oracle.attention_weights) and O_ref [n, d] = P V^ (oracle.attention_rows) of
    the dequantised blocks q^, k^, v^ (q_hat_rows [n, d], k_hat/v_hat [Nk, d]),
    v_scale [ceil(Nk / block)] the V block scales as stored (fp32).  Nothing here
    computes a softmax or an attention output.

    The kernel computes x_j = s_j - m + log2 r_j (log2 units, m its reference
    maximum, r_j = max(v_scale_j / max v_scale, 2^-20), 1 for a zero block),
    p_j = 2^x_j, rounds p_j to e4m3 for the P V product, keeps the unrounded p_j
    in the row sum l, and writes bf16(o~ * max v_scale / l).  Terms (derived
    term by term in the design notes, "FP8 error bound"):

    * t_round: e4m3 moves p by at most max(2^-4 p, 2^-10); scaled back by
      1 / (r_j l) with 1 / l <= P_max (the lazy reference lies at most 2^8 below
      the row maximum and never above it), key j moves O by at most
      b_j = max(2^-4 P_j, 2^-10 P_max / r_j) |v^_j|.  t_round = sum_j b_j.
    * t_w: every weight carries a relative error eta from the fp32 scores (128
      products summed in fp32 in the tensor core, three fp32 scale products,
      one FMA), ex2.approx, __log2f of r_j and the fp32 row sum and rescales;
      normalisation turns it into |W_j - P_j| <= 2 eta / (1 - eta) P_j.
    * t_acc: o~ sums Nk products in fp32 in the tensor core, (32 + Nk/32 + 1)
      roundings deep.
    * t_floor: blocks with v_scale_j below 2^-20 max v_scale use r_j = 2^-20.
    * the fp32 epilogue (two roundings) and bf16 RN of O: 2^-8 of the value.

    Returns (tol [n, d], sigma2 [n, d]); sigma2 is the mean square error the
    rounding model predicts (each rounding error uniform within its bound):
    sum_j b_j^2 / 3 + (2^-8 |O|)^2 / 3 + (t_w + t_acc + t_floor)^2.
    """
    P = np.asarray(P, dtype=np.float64)
    O = np.asarray(O_ref, dtype=np.float64)
    q = np.asarray(q_hat_rows, dtype=np.float64)
    kk = np.asarray(k_hat, dtype=np.float64)
    av = np.abs(np.asarray(v_hat, dtype=np.float64))
    n, Nk = P.shape
    d = q.shape[1]
    if Nk == 0 or n == 0:
        z = np.zeros(O.shape)
        return z + 2.0 ** -8 * np.abs(O), z
    vs = np.asarray(v_scale, dtype=np.float64)
    vmax = vs.max() if vs.size else 0.0
    ratio = vs / (vmax if vmax > 0 else 1.0)
    r_blk = np.where(vs > 0, np.maximum(ratio, 2.0 ** -20), 1.0)
    r = np.repeat(r_blk, block)[:Nk]
    floored = np.repeat((vs > 0) & (ratio < 2.0 ** -20), block)[:Nk]
    live = P > 0
    pmax = P.max(axis=1, keepdims=True)
    n_tiles = -(-Nk // block)
    # eta: relative error of each weight before normalisation
    A = np.abs(q) @ np.abs(kk).T                          # sum_k |q_k k_jk|, bounds |S_j| / scale
    log2e = 1.0 / math.log(2.0)
    m_abs = log2e * scale * A.max(axis=1, keepdims=True) + 30.0
    dx = log2e * scale * (d * 2.0 ** -23) * A + 2.0 ** -21 * m_abs + 2.0 ** -17
    eta_key = np.where(live, np.expm1(math.log(2.0) * dx) + 2.0 ** -21, 0.0).max(axis=1, keepdims=True)
    eta = eta_key + (24 + 4 * n_tiles) * 2.0 ** -24
    w = 2 * eta / (1 - eta)
    A1 = P @ av                                           # sum_j P_j |v^_j|
    bj = np.where(live, np.maximum(2.0 ** -4 * P, 2.0 ** -10 * pmax / r[None, :]), 0.0)
    t_round = (1 + w) * (bj @ av)
    t_w = w * A1
    t_acc = (32 + Nk / 32 + 1) * 2.0 ** -23 * ((1 + 2.0 ** -4) * (1 + w) * A1 + t_round)
    vs_key = np.repeat(vs, block)[:Nk]
    fl = np.where(floored, 2.0 ** -20 * vmax / np.where(vs_key > 0, vs_key, 1.0) - 1.0, 0.0)
    t_floor = (P * fl[None, :]) @ av
    pre = t_round + t_w + t_acc + t_floor
    tol = pre + (2.0 ** -8 + 2.0 ** -22) * (np.abs(O) + pre)
    sigma2 = (bj ** 2) @ (av ** 2) / 3 + (2.0 ** -8 * O) ** 2 / 3 + (t_w + t_acc + t_floor) ** 2
    return tol, sigma2


def check_fp8(o_gpu, O_ref, tol, sigma2, what=""):
    """The FP8 parity checks: every element within its bound, and the errors as a whole
    no larger than the rounding model predicts (mean square <= the predicted mean
    square, against an expected ratio of at most 1/3 ... 1) and unbiased (the
    least-squares slope of the error on O within 2^-5; rounding P toward zero
    instead of to nearest gives -0.02 to -0.045, correct rounding within 0.012
    in the float64 emulation of tests/test_fp8_bound_cpu.py)."""
    a = f64(o_gpu)
    assert np.isfinite(a).all(), f"{what}: non-finite output"
    err = a - np.asarray(O_ref, dtype=np.float64)
    worst = float((np.abs(err) / np.maximum(tol, 1e-300)).max()) if err.size else 0.0
    assert worst <= 1.0, f"{what}: max |dO| / bound = {worst:.3f} (max |dO| {np.abs(err).max():.3e})"
    ms, ms_model = float((err ** 2).mean()), float(np.asarray(sigma2).mean())
    assert ms <= ms_model + 1e-30, f"{what}: mean square error {ms:.3e} > rounding model {ms_model:.3e}"
    oo = float((np.asarray(O_ref) ** 2).sum())
    slope = float((err * O_ref).sum()) / oo if oo > 0 else 0.0
    assert abs(slope) <= 2.0 ** -5, f"{what}: error correlates with O (slope {slope:.4f})"
    return worst, ms / ms_model if ms_model > 0 else 0.0, slope
