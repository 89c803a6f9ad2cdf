"""Float64 oracle for FP8 attention (test infrastructure only; see the package header).

Source: "3.4 Attention Kernels" (llm-learning-path, part 3), "FlashAttention-2
and -3": FlashAttention-3's FP8 attention quantises by blocks and first applies
an "incoherent processing" step, a random orthogonal transform, so that outlier
channels are spread out before rounding to 8 bits.  The page states the method
in prose only; the readings taken here are the plainest ones it supports:

* the transform is M = diag(signs) H_d / sqrt(d), H_d the Sylvester Hadamard
  matrix (entries (-1)^popcount(i & j)) and signs a random +-1 vector: M is
  orthogonal and random, and (Q M)(K M)^T = Q K^T, so the scores are unchanged
  in exact arithmetic.  V is not transformed (P V would need the inverse on O).
* a block is one 128-row tile of one head (the kernels' tile), with one fp32
  scale = amax / 448 (448: the largest finite e4m3 value); the stored value is
  the e4m3 code of x / scale, rounded to nearest, ties to even, saturating.
* the attention of the quantised inputs is the plain definition applied to the
  dequantised blocks code * scale (``attention`` of this package).

e4m3 here is the "fn" variant: 1 sign bit, 4 exponent bits (bias 7), 3
mantissa bits, no infinities, one NaN pattern per sign (S.1111.111), largest
finite 448 = 1.75 * 2^8, smallest normal 2^-6, subnormals m/8 * 2^-6.
"""
from __future__ import annotations

import numpy as np

from .attention import attention, to_f64

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_round(x) -> np.ndarray:
    """Round float64 values to the nearest e4m3 value (ties to even), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # quantum: 2^(e - 3) for a normal value 2^e <= a < 2^(e+1), 2^-9 below 2^-6
    _, e = np.frexp(np.where(a > 0, a, 1.0))        # a = f * 2^e with 0.5 <= f < 1
    quantum = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    r = np.rint(a / quantum) * quantum               # np.rint rounds half to even; a / quantum is exact
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_encode(x) -> np.ndarray:
    """uint8 codes of values that are exactly e4m3 (as produced by e4m3_round)."""
    x = np.asarray(x, dtype=np.float64)
    sign = (np.signbit(x)).astype(np.uint8) << 7
    a = np.abs(x)
    code = np.zeros(x.shape, dtype=np.uint8)
    sub = a < 2.0 ** -6
    code[sub] = np.rint(a[sub] / 2.0 ** -9).astype(np.uint8)          # exponent field 0
    f, e = np.frexp(np.where(sub, 1.0, a))
    exp_field = (e - 1 + 7).astype(np.int64)
    mant = np.rint((2 * f - 1) * 8).astype(np.int64)
    code[~sub] = ((exp_field << 3) | mant)[~sub].astype(np.uint8)
    if np.any(e4m3_decode(code | sign) != x):
        raise ValueError("value is not an e4m3 number")
    return code | sign


def e4m3_decode(code) -> np.ndarray:
    """float64 values of e4m3 codes (the NaN patterns decode to NaN)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(ef == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * np.ldexp(1.0, ef - 7))
    val = np.where((ef == 0xF) & (m == 0x7), np.nan, val)
    return s * val


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_d, H[i, j] = (-1)^popcount(i & j); d a power of two."""
    if d <= 0 or d & (d - 1):
        raise ValueError("d must be a power of two")
    i = np.arange(d)
    bits = np.bitwise_and(i[:, None], i[None, :])
    pop = np.zeros_like(bits)
    while np.any(bits):
        pop += bits & 1
        bits >>= 1
    return np.where(pop % 2 == 0, 1.0, -1.0)


def incoherent_transform(signs) -> np.ndarray:
    """The random orthogonal matrix M = diag(signs) H_d / sqrt(d)."""
    s = to_f64(signs).reshape(-1)
    d = s.shape[0]
    return (s[:, None] * hadamard(d)) / np.sqrt(d)


def quantize_blocks(x, block: int = BLOCK):
    """Block quantisation of x [..., N, d] along N: one scale per `block` rows.

    Returns (codes uint8 [..., N, d], scales float64 [..., ceil(N / block)],
    dequantised float64 [..., N, d]).  A block of zeros has scale 0 and codes 0.
    """
    xf = to_f64(x)
    N = xf.shape[-2]
    nb = -(-N // block)
    codes = np.zeros(xf.shape, dtype=np.uint8)
    scales = np.zeros(xf.shape[:-2] + (nb,))
    deq = np.zeros(xf.shape)
    for t in range(nb):
        blk = xf[..., t * block:(t + 1) * block, :]
        amax = np.abs(blk).max(axis=(-2, -1)) if blk.size else np.zeros(xf.shape[:-2])
        sc = amax / E4M3_MAX
        safe = np.where(sc > 0, sc, 1.0)[..., None, None]
        r = e4m3_round(blk / safe)
        codes[..., t * block:(t + 1) * block, :] = e4m3_encode(r)
        scales[..., t] = sc
        deq[..., t * block:(t + 1) * block, :] = r * np.where(sc > 0, sc, 0.0)[..., None, None]
    return codes, scales, deq


def fp8_quantize(q, k, v, signs=None, block: int = BLOCK):
    """The FP8 inputs of the attention: Q' = Q M and K' = K M (M from `signs`, or
    no transform when signs is None), then Q', K', V block-quantised.

    q [B, H, Nq, d], k/v [B, Hkv, Nk, d].  Returns a dict with codes, scales and
    the dequantised tensors ``q_hat``, ``k_hat``, ``v_hat`` (float64).
    """
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    if signs is not None:
        M = incoherent_transform(signs)
        qf = qf @ M
        kf = kf @ M
    q8, qs, qh = quantize_blocks(qf, block)
    k8, ks, kh = quantize_blocks(kf, block)
    v8, vs, vh = quantize_blocks(vf, block)
    return {"q8": q8, "q_scale": qs, "q_hat": qh, "k8": k8, "k_scale": ks, "k_hat": kh,
            "v8": v8, "v_scale": vs, "v_hat": vh}


def fp8_attention(quant: dict, *, causal: bool, scale: float):
    """Exact attention of the dequantised FP8 inputs (the plain definition)."""
    return attention(quant["q_hat"], quant["k_hat"], quant["v_hat"], causal=causal, scale=scale)
