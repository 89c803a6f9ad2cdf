"""FP8 attention ("3.4 Attention Kernels", "FlashAttention-2 and -3": block
quantisation with a random orthogonal transform): the quantisation kernel and
the tcgen05 kind::f8f6f4 attention kernel against the float64 oracle.

* attn_fp8_quantize vs oracle.fp8.fp8_quantize: scales to fp32 rounding of the
  transform, and every code within the rounding of the value the oracle
  computes in float64 (a code differs only where that value lies within the
  fp32 error of the transform of a rounding midpoint), V transposed and padded.
* attn_fwd_fp8 fed the ORACLE's codes and scales vs the oracle's attention of
  the dequantised blocks (oracle.fp8.fp8_attention, or oracle.attention_rows on
  sampled rows), element by element within the bound of the kernel's rounding
  (tests/parity.py fp8_bound, built from the oracle's softmax weights), with the
  mean square error within the rounding model and no error correlated with O
  (tests/parity.py check_fp8); LSE within 1e-3.
* the whole FP8 path against exact attention of the bf16 inputs, and the
  transform's benefit on inputs with outlier channels.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as F
from exact_tiled_attention_11_gb300 import (Fp8Inputs, attn_device_error, attn_fp8_padded_keys, attn_fp8_quantize,
                                            attn_fwd_fp8)
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_fp8, check_lse, f64, fp8_bound

pytestmark = pytest.mark.gpu


def _inputs(B, H, Hkv, Nq, Nk, seed, outliers=False):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Nq, 128, generator=g)
    k = torch.randn(B, Hkv, Nk, 128, generator=g)
    v = torch.randn(B, Hkv, Nk, 128, generator=g)
    if outliers:
        q[..., [5, 90]] *= 30.0
        k[..., [5, 90]] *= 30.0
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def _code_window(r, delta):
    """Values the e4m3 rounding of anything in [r - delta, r + delta] can take."""
    return F.e4m3_round(r - delta), F.e4m3_round(r + delta)


def _check_codes(codes_gpu, r_exact, delta, what):
    got = F.e4m3_decode(codes_gpu)
    lo, hi = _code_window(r_exact, delta)
    bad = ~((got >= lo) & (got <= hi))
    assert not bad.any(), f"{what}: {int(bad.sum())} codes outside the rounding window"
    same = got == F.e4m3_round(r_exact)
    assert same.mean() > 0.99, f"{what}: only {same.mean():.4f} of codes equal the float64 rounding"


@pytest.mark.parametrize("signed", [True, False])
@pytest.mark.parametrize("Nq,Nk", [(300, 300), (128, 1000), (1, 129)])
def test_quantize_matches_oracle(cuda, Nq, Nk, signed):
    q, k, v = _inputs(2, 4, 2, Nq, Nk, seed=Nq + Nk, outliers=True)
    signs = W.fp8_signs(128, seed=1) if signed else None
    x = attn_fp8_quantize(q.to(cuda), k.to(cuda), v.to(cuda), None if signs is None else signs.to(cuda))
    torch.cuda.synchronize()
    ref = F.fp8_quantize(q, k, v, None if signs is None else signs.numpy())
    for name in ("q_scale", "k_scale", "v_scale"):
        np.testing.assert_allclose(f64(getattr(x, name)), ref[name], rtol=1e-5, atol=0, err_msg=name)
    M = F.incoherent_transform(signs.numpy()) if signed else np.eye(128)
    for t, codes, sc, transformed, what in ((q, x.q8, ref["q_scale"], True, "q"), (k, x.k8, ref["k_scale"], True, "k"),
                                            (v, None, ref["v_scale"], False, "v")):
        xt = f64(t) @ M if transformed else f64(t)
        n = xt.shape[2]
        sc_rows = np.repeat(sc, 128, axis=-1)[..., :n, None]
        r = xt / np.where(sc_rows > 0, sc_rows, 1.0)
        # fp32 error of the butterfly: 8 roundings of partial sums bounded by the row's l1 norm
        l1 = np.abs(f64(t)).sum(axis=-1, keepdims=True) / math.sqrt(128) if transformed and signed else 0.0
        delta = np.abs(r) * 1e-5 + 8 * 2.0 ** -24 * l1 / np.where(sc_rows > 0, sc_rows, 1.0) + 1e-12
        if what == "v":
            Np = attn_fp8_padded_keys(n)
            vt = x.v8t.cpu().numpy()
            assert vt.shape == (2, 2, 128, Np)
            assert not vt[..., n:].any(), "V^T padding must be zero"
            codes_np = vt[..., :n].transpose(0, 1, 3, 2)
        else:
            codes_np = codes.cpu().numpy()
        _check_codes(codes_np, r, delta, what)


def _upload(ref, cuda):
    v8t = np.ascontiguousarray(ref["v8"].transpose(0, 1, 3, 2))
    Nk = v8t.shape[-1]
    Np = attn_fp8_padded_keys(Nk)
    v8t = np.concatenate([v8t, np.zeros(v8t.shape[:-1] + (Np - Nk,), np.uint8)], axis=-1)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dt).to(cuda)
    return Fp8Inputs(t(ref["q8"], torch.uint8), t(ref["k8"], torch.uint8), t(v8t, torch.uint8),
                     t(ref["q_scale"], torch.float32), t(ref["k_scale"], torch.float32),
                     t(ref["v_scale"], torch.float32))


def _stored_scales(ref):
    """The oracle's scales as the kernel reads them (fp32), and the blocks dequantised with them."""
    out = dict(ref)
    for name, codes, hat in (("q_scale", "q8", "q_hat"), ("k_scale", "k8", "k_hat"), ("v_scale", "v8", "v_hat")):
        s32 = ref[name].astype(np.float32).astype(np.float64)
        out[name] = s32
        rows = ref[codes].shape[2]
        out[hat] = F.e4m3_decode(ref[codes]) * np.repeat(s32, 128, axis=-1)[..., :rows, None]
    return out


def _oracle_and_bound(ref, causal, scale):
    """The oracle's O and LSE of the dequantised blocks, and the error bound of every element."""
    O, L = F.fp8_attention(ref, causal=causal, scale=scale)
    B, H, Nq, _ = ref["q_hat"].shape
    Hkv = ref["k_hat"].shape[1]
    tol, s2 = np.zeros(O.shape), np.zeros(O.shape)
    rows = np.arange(Nq)
    for b in range(B):
        for h in range(H):
            kv = h // (H // Hkv)
            P, _ = oracle.attention_weights(ref["q_hat"], ref["k_hat"], b, h, rows, causal=causal, scale=scale)
            tol[b, h], s2[b, h] = fp8_bound(P, O[b, h], ref["q_hat"][b, h], ref["k_hat"][b, kv], ref["v_hat"][b, kv],
                                            ref["v_scale"][b, kv], scale=scale)
    return O, L, tol, s2


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Hkv,Nq,Nk", [(1, 4, 4, 300, 300), (2, 4, 2, 128, 128), (1, 8, 2, 513, 513),
                                           (1, 2, 1, 100, 700), (1, 2, 2, 700, 100), (1, 2, 1, 1, 257)])
def test_fp8_attention_matches_oracle_on_oracle_blocks(cuda, B, H, Hkv, Nq, Nk, causal):
    q, k, v = _inputs(B, H, Hkv, Nq, Nk, seed=B * 7 + Nq + 3 * Nk)
    ref = _stored_scales(F.fp8_quantize(q, k, v, W.fp8_signs(128, seed=2).numpy()))
    x = _upload(ref, cuda)
    attn_device_error(clear=True)
    o, lse = attn_fwd_fp8(x, causal=causal)
    torch.cuda.synchronize()
    O, L, tol, s2 = _oracle_and_bound(ref, causal, 1 / math.sqrt(128))
    check_fp8(o, O, tol, s2, f"fp8 {B}x{H}x{Nq}x{Nk} causal={causal}")
    check_lse(lse.cpu(), L, f"fp8 {B}x{H}x{Nq}x{Nk} causal={causal}")
    assert attn_device_error() == 0


def test_fp8_zero_blocks_and_no_keys(cuda):
    """A zero V block and a zero K block give finite results; causal rows with no key give O = 0, LSE = -inf."""
    q, k, v = _inputs(1, 2, 1, 300, 200, seed=11)
    k[:, :, 128:] = 0
    v[:, :, :128] = 0
    ref = _stored_scales(F.fp8_quantize(q, k, v, W.fp8_signs(128, seed=3).numpy()))
    o, lse = attn_fwd_fp8(_upload(ref, cuda), causal=True)
    torch.cuda.synchronize()
    O, L, tol, s2 = _oracle_and_bound(ref, True, 1 / math.sqrt(128))
    a = f64(o)
    assert (a[:, :, :100] == 0).all() and torch.isneginf(lse[:, :, :100]).all()
    check_fp8(o, O, tol, s2, "zero blocks")
    check_lse(lse.cpu(), L, "zero blocks")


def test_fp8_path_end_to_end_and_transform_benefit(cuda):
    """GPU quantisation + FP8 attention against exact attention of the bf16 inputs; with
    outlier channels in Q and K the transform lowers the error."""
    B, H, Hkv, N = 1, 8, 2, 1024
    q, k, v = _inputs(B, H, Hkv, N, N, seed=21, outliers=True)
    O, _ = oracle.attention(q, k, v, causal=True, scale=1 / math.sqrt(128) / 4)
    errs, quant_only = {}, {}
    for signed in (False, True):
        signs = W.fp8_signs(128, seed=4) if signed else None
        x = attn_fp8_quantize(q.to(cuda), k.to(cuda), v.to(cuda), None if signs is None else signs.to(cuda))
        o, _ = attn_fwd_fp8(x, causal=True, scale=1 / math.sqrt(128) / 4)
        torch.cuda.synchronize()
        errs[signed] = float(np.abs(f64(o) - O).mean())
        # the error of the input quantisation alone (oracle, float64)
        R = F.fp8_attention(F.fp8_quantize(q, k, v, None if signs is None else signs.numpy()), causal=True,
                            scale=1 / math.sqrt(128) / 4)[0]
        quant_only[signed] = float(np.abs(R - O).mean())
    # P's rounding adds little to the input quantisation's error, and the transform helps
    assert errs[True] < 1.25 * quant_only[True] and errs[False] < 1.25 * quant_only[False], (errs, quant_only)
    assert errs[True] < 0.6 * errs[False], errs


def test_fp8_full_size_sampled(cuda):
    """The benchmark's prefill inputs (B=1, H=32, Hkv=8, N=8192, d=128, causal) through the
    FP8 path: the GPU quantiser on sampled blocks against the float64 quantiser, and the
    FP8 attention of the oracle's blocks on sampled rows against the oracle, within the
    bound of the kernel's rounding."""
    cfg = W.C3
    q, k, v = W.prefill_inputs_for(cfg)
    signs = W.fp8_signs(128)
    x = attn_fp8_quantize(q.to(cuda), k.to(cuda), v.to(cuda), signs.to(cuda))
    torch.cuda.synchronize()
    M = F.incoherent_transform(signs.numpy())
    for name, t, codes, scales, transformed in (("q", q, x.q8, x.q_scale, True), ("k", k, x.k8, x.k_scale, True),
                                               ("v", v, None, x.v_scale, False)):
        for (h, blk) in ((0, 0), (3, 17), (7, 63), (1, 40)):
            h = h % t.shape[1]
            xs = f64(t[0, h, blk * 128:(blk + 1) * 128])
            xs = xs @ M if transformed else xs
            c_ref, s_ref, _ = F.quantize_blocks(xs[None, None])
            np.testing.assert_allclose(float(scales[0, h, blk]), s_ref[0, 0, 0], rtol=1e-5, err_msg=f"{name} {h} {blk}")
            r = xs / s_ref[0, 0, 0]
            l1 = np.abs(f64(t[0, h, blk * 128:(blk + 1) * 128])).sum(axis=-1, keepdims=True) / math.sqrt(128)
            delta = np.abs(r) * 1e-5 + (8 * 2.0 ** -24 * l1 / s_ref[0, 0, 0] if transformed else 0.0) + 1e-12
            if codes is None:
                got = x.v8t[0, h, :, blk * 128:(blk + 1) * 128].cpu().numpy().T
            else:
                got = codes[0, h, blk * 128:(blk + 1) * 128].cpu().numpy()
            _check_codes(got, r, delta, f"{name} head {h} block {blk}")
    # attention over the oracle's blocks: the sampled heads (and their KV heads) carry the
    # oracle's codes, every other head all-zero blocks (valid input, outputs not checked),
    # so the launch keeps the full shape
    heads, kvs = [0, 5, 31], [0, 1, 7]
    sub = _stored_scales(F.fp8_quantize(q[:, heads], k[:, kvs], v[:, kvs], signs.numpy()))
    full = {"q8": np.zeros((1, 32, cfg.N, 128), np.uint8), "k8": np.zeros((1, 8, cfg.N, 128), np.uint8),
            "v8": np.zeros((1, 8, cfg.N, 128), np.uint8), "q_scale": np.zeros((1, 32, cfg.N // 128)),
            "k_scale": np.zeros((1, 8, cfg.N // 128)), "v_scale": np.zeros((1, 8, cfg.N // 128))}
    for dst, src, idx in (("q", "q", heads), ("k", "k", kvs), ("v", "v", kvs)):
        full[dst + "8"][:, idx] = sub[src + "8"]
        full[dst + "_scale"][:, idx] = sub[src + "_scale"]
    o, lse = attn_fwd_fp8(_upload(full, cuda), causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    rng = np.random.default_rng(0)
    outs, refs, tols, s2s = [], [], [], []
    for i, h in enumerate(heads):
        rows = np.unique(np.concatenate([[0, 1, 127, 128, 8191], rng.integers(0, cfg.N, 60)]))
        O, L = oracle.attention_rows(sub["q_hat"], sub["k_hat"], sub["v_hat"], 0, i, rows, causal=True,
                                     scale=cfg.scale)
        P, _ = oracle.attention_weights(sub["q_hat"], sub["k_hat"], 0, i, rows, causal=True, scale=cfg.scale)
        tol, s2 = fp8_bound(P, O, sub["q_hat"][0, i][rows], sub["k_hat"][0, i], sub["v_hat"][0, i],
                            sub["v_scale"][0, i], scale=cfg.scale)
        check_lse(lse[0, h, rows].cpu(), L, f"fp8 full size head {h}")
        outs.append(f64(o[0, h, rows])), refs.append(O), tols.append(tol), s2s.append(s2)
    check_fp8(*[np.concatenate(x) for x in (outs, refs, tols, s2s)], "fp8 full size, sampled rows")
    assert attn_device_error() == 0
