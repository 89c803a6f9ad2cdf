"""Pins of the FP8 oracle (oracle/fp8.py) against things other than itself:
PyTorch's float8_e4m3fn conversion (a library routine), scipy's Hadamard
matrix, orthogonality, the exact invariance of the scores under the transform,
the block quantisation's error bound, and the outlier case that the transform
exists for ("3.4 Attention Kernels", "FlashAttention-2 and -3")."""
import math
import sys

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from oracle import fp8 as F

FP8 = sys.modules["oracle.fp8"]


def _torch_e4m3(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_round_matches_torch_conversion():
    rng = np.random.default_rng(1)
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (finite[1:] + finite[:-1]) / 2                      # exact ties: round half to even
    xs = np.concatenate([finite, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
                         rng.uniform(-448, 448, 20000), rng.uniform(-2 ** -5, 2 ** -5, 20000),
                         rng.standard_normal(20000) * 30, [0.0, 447.9, 448.0, 455.0, -463.0]])
    xs = xs.astype(np.float32).astype(np.float64)             # values a float32 kernel can hold
    np.testing.assert_array_equal(F.e4m3_round(xs), _torch_e4m3(xs))


def test_e4m3_round_saturates():
    assert F.e4m3_round(1e6) == 448.0 and F.e4m3_round(-500.0) == -448.0


def test_e4m3_codes_match_torch_bit_patterns():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dec = F.e4m3_decode(codes)
    np.testing.assert_array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(dec[ok], ref[ok])
    np.testing.assert_array_equal(F.e4m3_encode(dec[ok]), codes[ok])
    # a float -> code round trip through torch gives the same bytes
    x = np.random.default_rng(2).uniform(-448, 448, 5000)
    tb = torch.tensor(x, dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F.e4m3_encode(F.e4m3_round(x)), tb)


@pytest.mark.parametrize("d", [1, 2, 4, 8, 64, 128, 256])
def test_hadamard_is_scipy_hadamard(d):
    np.testing.assert_array_equal(F.hadamard(d), scipy.linalg.hadamard(d))


def test_transform_is_orthogonal_and_keeps_scores():
    rng = np.random.default_rng(3)
    signs = rng.choice([-1.0, 1.0], 128)
    M = F.incoherent_transform(signs)
    np.testing.assert_allclose(M @ M.T, np.eye(128), atol=1e-14)
    assert np.all(np.abs(np.abs(M) - 1 / math.sqrt(128)) < 1e-16)
    Q = rng.standard_normal((1, 2, 50, 128))
    K = rng.standard_normal((1, 2, 70, 128))
    V = rng.standard_normal((1, 2, 70, 128))
    O1, L1 = oracle.attention(Q @ M, K @ M, V, causal=True, scale=0.1)
    O2, L2 = oracle.attention(Q, K, V, causal=True, scale=0.1)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(L1, L2, atol=1e-12)


def test_block_quantisation_bounds_and_layout():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 3, 300, 16)) * rng.uniform(0.01, 100, (2, 3, 1, 1))
    x[1, 2, 128:256] = 0.0                                      # an all-zero block
    codes, scales, deq = F.quantize_blocks(x)
    assert codes.shape == x.shape and scales.shape == (2, 3, 3)
    assert scales[1, 2, 1] == 0 and not deq[1, 2, 128:256].any() and not codes[1, 2, 128:256].any()
    for t, (lo, hi) in enumerate([(0, 128), (128, 256), (256, 300)]):
        blk = x[:, :, lo:hi]
        amax = np.abs(blk).max(axis=(-2, -1))
        np.testing.assert_array_equal(scales[:, :, t], amax / 448.0)
        y = F.e4m3_decode(codes[:, :, lo:hi])
        nz = scales[:, :, t] > 0
        # the block's largest magnitude maps onto 448, every code is finite
        assert np.all(np.abs(y).max(axis=(-2, -1))[nz] == 448.0) and np.all(np.isfinite(y))
        # rounding error: half a quantum (2^-4 relative for normals, 2^-10 absolute below 2^-6)
        r = blk / np.where(scales[:, :, t] > 0, scales[:, :, t], 1.0)[..., None, None]
        err = np.abs(y - r)
        assert np.all(err <= np.maximum(np.abs(r) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-12))
        np.testing.assert_array_equal(deq[:, :, lo:hi], y * scales[:, :, t][..., None, None])


def test_fp8_quantize_brute_force_small():
    """A 3-row block written out element by element with scalar Python arithmetic."""
    rng = np.random.default_rng(5)
    signs = np.array([1.0, -1.0, -1.0, 1.0])
    q = rng.standard_normal((1, 1, 3, 4))
    k = rng.standard_normal((1, 1, 3, 4))
    v = rng.standard_normal((1, 1, 3, 4))
    out = F.fp8_quantize(q, k, v, signs)
    Hm = [[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]]
    qt = [[sum(q[0, 0, r, i] * signs[i] * Hm[i][j] for i in range(4)) / 2 for j in range(4)] for r in range(3)]
    amax = max(abs(x) for row in qt for x in row)
    s = amax / 448
    assert out["q_scale"][0, 0, 0] == pytest.approx(s, rel=1e-15)
    for r in range(3):
        for j in range(4):
            want = float(_torch_e4m3([qt[r][j] / s])[0])
            assert F.e4m3_decode(out["q8"][0, 0, r, j]) == want
            assert out["q_hat"][0, 0, r, j] == pytest.approx(want * s, rel=1e-15)
    # V is quantised without the transform
    np.testing.assert_array_equal(F.e4m3_decode(out["v8"][0, 0]),
                                  _torch_e4m3(v[0, 0] / (np.abs(v).max() / 448)))


def test_transform_reduces_error_from_outlier_channels():
    """Q and K with a few large channels: quantising after the transform loses less."""
    rng = np.random.default_rng(6)
    B, H, N, d = 1, 4, 256, 128
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    q[..., [3, 77]] *= 40.0
    k[..., [3, 77]] *= 40.0
    O, _ = oracle.attention(q, k, v, causal=False, scale=1 / math.sqrt(d) / 10)
    plain = F.fp8_attention(F.fp8_quantize(q, k, v, None), causal=False, scale=1 / math.sqrt(d) / 10)[0]
    signs = rng.choice([-1.0, 1.0], d)
    rotated = F.fp8_attention(F.fp8_quantize(q, k, v, signs), causal=False, scale=1 / math.sqrt(d) / 10)[0]
    e_plain = np.abs(plain - O).mean()
    e_rot = np.abs(rotated - O).mean()
    assert e_rot < 0.5 * e_plain, (e_rot, e_plain)


# ---------------------------------------------------------------------------
# planted mistakes in the FP8 oracle (each must fail a pin above)
# ---------------------------------------------------------------------------

def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _round_half_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    qn = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / qn + 0.5) * qn, 448.0), x)


def _no_subnormals(x):
    r = _ORIG_ROUND(x)
    return np.where(np.abs(r) < 2.0 ** -6, 0.0, r)


def _hadamard_columns_rolled(d):
    return np.roll(_ORIG_HADAMARD(d), 1, axis=1)


def _transform_unnormalised(signs):
    s = np.asarray(signs, dtype=np.float64).reshape(-1)
    return s[:, None] * F.hadamard(s.shape[0])


_ORIG_ROUND = F.e4m3_round
_ORIG_HADAMARD = F.hadamard


@pytest.mark.parametrize("name,mutant,checks", [
    ("e4m3_round", _round_half_away, [test_e4m3_round_matches_torch_conversion]),
    ("e4m3_round", _no_subnormals, [test_e4m3_round_matches_torch_conversion]),
    ("hadamard", _hadamard_columns_rolled, [lambda: test_hadamard_is_scipy_hadamard(128)]),
    ("incoherent_transform", _transform_unnormalised, [test_transform_is_orthogonal_and_keeps_scores]),
    ("E4M3_MAX", 256.0, [test_block_quantisation_bounds_and_layout, test_fp8_quantize_brute_force_small]),
])
def test_planted_fp8_mistakes_are_caught(monkeypatch, name, mutant, checks):
    monkeypatch.setattr(FP8, name, mutant)
    for fn in checks:
        assert _fails(fn), f"{name} mutant passed a pin"
