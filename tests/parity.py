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


def fp8_tolerance_rows(q_rows, k, v, v_scale, rows, Nq, *, causal, scale, block=128):
    """fp8_tolerance for selected query rows of one head: q_rows [len(rows), d] (the
    dequantised query rows), k, v [Nk, d] (the head's dequantised keys and values),
    v_scale [ceil(Nk / block)], rows their indices among Nq query rows."""
    q = np.asarray(q_rows, dtype=np.float64)
    kk = np.asarray(k, dtype=np.float64)
    vv = np.asarray(v, dtype=np.float64)
    Nk = kk.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    S = scale * q @ kk.T
    if causal:
        keep = np.arange(Nk)[None, :] <= rows[:, None] + (Nk - Nq)
        S = np.where(keep, S, -np.inf)
    smax = S.max(axis=1, keepdims=True) if Nk else np.full((len(rows), 1), -np.inf)
    live = np.isfinite(smax[:, 0])
    E = np.where(live[:, None], np.exp(S - np.where(live[:, None], smax, 0.0)), 0.0)
    L = E.sum(axis=1, keepdims=True)
    P = np.where(live[:, None], E / np.where(L > 0, L, 1.0), 0.0)
    O = P @ vv
    LSE = np.where(live, smax[:, 0] + np.log(np.where(L[:, 0] > 0, L[:, 0], 1.0)), -np.inf)
    vs = np.asarray(v_scale, dtype=np.float64)
    vmax = vs.max() if vs.size else 0.0
    r = np.where(vs > 0, np.maximum(vs / (vmax if vmax > 0 else 1.0), 2.0 ** -20), 1.0)
    r_key = np.repeat(r, block)[:Nk]
    pmax = P.max(axis=1, keepdims=True) if Nk else np.zeros((len(rows), 1))
    bj = np.maximum(2.0 ** -4 * P, 2.0 ** -10 * pmax / r_key[None, :]) * (P > 0)
    av = np.abs(vv)
    lin = bj @ av
    quad = np.sqrt((bj ** 2) @ (av ** 2))
    tol = np.minimum(lin, 7 * quad) + 2.0 ** -8 * np.abs(O) + 1e-3 * (P @ av) + 1e-6
    return O, LSE, tol


def fp8_tolerance(q_hat, k_hat, v_hat, v_scale, *, causal, scale, block=128):
    """Per-element bound on |O_fp8 - O_oracle| for attention over dequantised FP8 blocks.

    The FP8 kernel rounds p' = p * r_j to e4m3 before P V (r_j = v_scale_j /
    max v_scale <= 1, p = 2^(s - m_ref) with the reference max m_ref within 8
    (log2) of the row max, so l >= 1 * L where L = sum exp(S - S_max)).  e4m3
    rounding moves x by at most max(2^-4 x, 2^-10), so key j moves the output
    by at most b_j = max(2^-4 P_j, 2^-10 P_max / r_j) |v_j| (P the oracle's
    softmax weights).  The errors of different keys are bounded, independent
    roundings, so the bound is min(sum b_j, 7 sqrt(sum b_j^2)) (Hoeffding at
    7 sigma), plus the bf16 rounding of O (2^-8 |O|), plus 1e-3 sum P_j |v_j|
    for fp32 accumulation inside the tensor core.  Returns (O, LSE, tol)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q_hat, k_hat, v_hat))
    B, H, Nq, d = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    O = np.zeros((B, H, Nq, d))
    LSE = np.full((B, H, Nq), -np.inf)
    tol = np.zeros((B, H, Nq, d))
    vs = np.asarray(v_scale, dtype=np.float64)
    rows = np.arange(Nq)
    for b in range(B):
        for h in range(H):
            kv = h // g
            O[b, h], LSE[b, h], tol[b, h] = fp8_tolerance_rows(q[b, h], k[b, kv], v[b, kv], vs[b, kv], rows, Nq,
                                                               causal=causal, scale=scale, block=block)
    return O, LSE, tol
