"""Prefill parity: the CUDA attn_fwd (through the C ABI) against the float64 oracle."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_fwd
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o, f64

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run(q, k, v, causal, scale, dev):
    o, lse = attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


# ---------------------------------------------------------------- workload 1: fp32, N = 256, d = 64

@pytest.mark.parametrize("q_mult", W.C1.q_mults)
def test_c1_fp32_exact(cuda, q_mult):
    q, k, v = W.prefill_inputs_for(W.C1, q_mult=q_mult)
    o, lse = run(q, k, v, False, W.C1.scale, cuda)
    O, L = oracle.attention(q, k, v, causal=False, scale=W.C1.scale)
    check_o(o, O, torch.float32, f"C1 x{q_mult}")
    check_lse(lse, L, f"C1 x{q_mult}")


# ---------------------------------------------------------------- small and ragged shapes

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 16, 100, 128, 129, 255, 384])
def test_small_and_ragged(cuda, N, causal, d, dtype):
    B, H, Hkv = 2, 4, 2
    q, k, v = W.prefill_inputs(B, H, Hkv, N, d, dtype, seed=N * 7 + d)
    scale = 1 / math.sqrt(d)
    o, lse = run(q, k, v, causal, scale, cuda)
    O, L = oracle.attention(q, k, v, causal=causal, scale=scale)
    check_o(o, O, W.torch_dtype(dtype), f"N={N} d={d} causal={causal} {dtype}")
    check_lse(lse, L, f"N={N} d={d} causal={causal} {dtype}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(8, 8), (8, 1), (16, 4)])
def test_gqa_groups_multi_tile(cuda, H, Hkv, causal):
    N, d = 640, 128
    q, k, v = W.prefill_inputs(1, H, Hkv, N, d, "bf16", seed=H * 10 + Hkv)
    o, lse = run(q, k, v, causal, 1 / math.sqrt(d), cuda)
    O, L = oracle.attention(q, k, v, causal=causal, scale=1 / math.sqrt(d))
    check_o(o, O, torch.bfloat16, f"GQA {H}/{Hkv}")
    check_lse(lse, L, f"GQA {H}/{Hkv}")


@pytest.mark.parametrize("q_mult", [30.0, 40.0])
@pytest.mark.parametrize("d", [64, 128])
def test_large_scores_rescale(cuda, q_mult, d):
    """Queries x30 / x40 push scores into the hundreds: the running-max rescale must hold."""
    q, k, v = W.prefill_inputs(1, 2, 2, 1000, d, "bf16", q_mult=q_mult, seed=5)
    for causal in (False, True):
        o, lse = run(q, k, v, causal, 1 / math.sqrt(d), cuda)
        O, L = oracle.attention(q, k, v, causal=causal, scale=1 / math.sqrt(d))
        check_o(o, O, torch.bfloat16, f"x{q_mult} causal={causal}")
        check_lse(lse, L, f"x{q_mult} causal={causal}")


# ---------------------------------------------------------------- workload 2: B4 H12 N2048 d64, both maskings

@pytest.mark.parametrize("causal", [False, True])
def test_c2_full_size(cuda, causal):
    cfg = W.C2
    q, k, v = W.prefill_inputs_for(cfg)
    o, lse = run(q, k, v, causal, cfg.scale, cuda)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # every head of batch 0 and 3 in full, the rest on sampled rows
    for b in (0, 3):
        for h in range(cfg.H):
            rows = np.arange(cfg.N)
            O, L = oracle.attention_rows(q, k, v, b, h, rows, causal=causal, scale=cfg.scale)
            check_o(o[b, h], O, torch.bfloat16, f"C2 b{b} h{h}")
            check_lse(lse[b, h], L, f"C2 b{b} h{h}")
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, 127, 128, 2047], rng.integers(0, cfg.N, 24)]))
    for b in (1, 2):
        for h in range(cfg.H):
            O, L = oracle.attention_rows(q, k, v, b, h, rows, causal=causal, scale=cfg.scale)
            check_o(o[b, h, rows], O, torch.bfloat16, f"C2 b{b} h{h} rows")
            check_lse(lse[b, h, rows], L, f"C2 b{b} h{h} rows")


# ---------------------------------------------------------------- workloads 3 and 5 at full size, sampled rows

def _sampled_rows(N, rng):
    fixed = [0, 1, 126, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    return np.unique(np.concatenate([fixed, rng.integers(0, N, 20)]))


def _check_sampled(cfg, q, k, v, o, lse, heads, tag):
    rng = np.random.default_rng(17)
    for b in range(cfg.B):
        for h in heads:
            rows = _sampled_rows(cfg.N, rng)
            O, L = oracle.attention_rows(q, k, v, b, h, rows, causal=True, scale=cfg.scale)
            check_o(o[b, h, rows], O, torch.bfloat16, f"{tag} b{b} h{h}")
            check_lse(lse[b, h, rows], L, f"{tag} b{b} h{h}")


def test_c3_full_size_sampled(cuda):
    cfg = W.C3
    q, k, v = W.prefill_inputs_for(cfg)
    o, lse = run(q, k, v, True, cfg.scale, cuda)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    _check_sampled(cfg, q, k, v, o, lse, heads=[0, 3, 4, 17, 31], tag="C3")


@pytest.mark.parametrize("q_mult", W.C5.q_mults)
def test_c5_full_size_sampled(cuda, q_mult):
    cfg = W.C5
    q, k, v = W.prefill_inputs_for(cfg, q_mult=q_mult)
    o, lse = run(q, k, v, True, cfg.scale, cuda)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    _check_sampled(cfg, q, k, v, o, lse, heads=[0, 9, 15], tag=f"C5 x{q_mult}")


@pytest.mark.parametrize("causal", [True, False])
def test_grouped_planes_gqa_sampled(cuda, causal):
    """One CTA per query-tile pair with all planes' K and V beyond half of L2 (67 MB here): on
    GB300 the launcher takes the query heads in groups of whole GQA groups whose K and V fit
    in half of L2 (28 heads = 7 KV heads, then a last group of 4).  Sampled rows of heads in
    both groups and on both sides of the boundary against the oracle."""
    cfg = W.PrefillConfig("gqa_b1_h32_hkv8_n16384_d128", 1, 32, 8, 16384, 128, "bf16", (causal,))
    q, k, v = W.prefill_inputs_for(cfg, seed=3)
    o, lse = run(q, k, v, causal, cfg.scale, cuda)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(23)
    for h in (0, 13, 27, 28, 31):
        rows = _sampled_rows(cfg.N, rng)
        O, L = oracle.attention_rows(q, k, v, 0, h, rows, causal=causal, scale=cfg.scale)
        check_o(o[0, h, rows], O, torch.bfloat16, f"grouped GQA h{h} causal={causal}")
        check_lse(lse[0, h, rows], L, f"grouped GQA h{h} causal={causal}")


# ---------------------------------------------------------------- the pages' worked examples on the GPU

def _p4_inputs(d, dtype):
    g = json.load(open(os.path.join(GOLDEN, "p4_worked_example.json")))
    N = len(g["K"])
    q = torch.zeros(1, 1, N, d)
    q[0, 0, 0, :2] = torch.tensor(g["q"])
    k = torch.zeros(1, 1, N, d)
    k[0, 0, :, :2] = torch.tensor(g["K"])
    v = torch.zeros(1, 1, N, d)
    v[0, 0, :, 0] = torch.tensor(g["V"])
    t = W.torch_dtype(dtype)
    return g, q.to(t), k.to(t), v.to(t)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_p4_worked_example_on_gpu(cuda, dtype):
    """The empirq example (one query, four keys in two blocks, no scale), zero-padded to d = 64."""
    g, q, k, v = _p4_inputs(64, dtype)
    o, lse = run(q, k, v, False, 1.0, cuda)
    O, L = oracle.attention(q, k, v, causal=False, scale=1.0)
    check_o(o, O, W.torch_dtype(dtype), "P4")
    check_lse(lse, L, "P4")
    tol = 0.5e-3 if dtype == "f32" else 2e-2
    assert abs(float(o[0, 0, 0, 0]) - g["printed"]["final_output"]) <= tol


def test_p2_lab_value_on_gpu_fp32(cuda):
    """The studybydoing lab: scores s_j as keys s_j e_1 against q = e_1, values v_j e_1."""
    g = json.load(open(os.path.join(GOLDEN, "p2_online_softmax_lab.json")))
    s, vals = g["scores"], g["values"]
    n, d = len(s), 64
    q = torch.zeros(1, 1, n, d)
    q[0, 0, :, 0] = 1.0
    k = torch.zeros(1, 1, n, d)
    k[0, 0, :, 0] = torch.tensor(s)
    v = torch.zeros(1, 1, n, d)
    v[0, 0, :, 0] = torch.tensor(vals, dtype=torch.float32)
    o, _ = run(q, k, v, False, 1.0, cuda)
    O, _ = oracle.attention(q, k, v, causal=False, scale=1.0)
    got = float(o[0, 0, 0, 0])
    # outputs here are ~54, not ~1: hold the fp32 bound relative to that magnitude
    assert abs(got - O[0, 0, 0, 0]) <= 1e-5 * abs(O[0, 0, 0, 0]) / 10
    assert abs(got - g["printed_batch"]) <= 1e-5 * abs(g["printed_batch"])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_closed_form_zero_keys_gpu(cuda, causal, dtype):
    N, d = 300, 128
    q, _, v = W.prefill_inputs(1, 2, 2, N, d, dtype, q_mult=30.0, seed=9)
    k = torch.zeros_like(v)
    o, lse = run(q, k, v, causal, 1 / math.sqrt(d), cuda)
    vf = f64(v)[0]
    if causal:
        csum = np.cumsum(vf, axis=1) / np.arange(1, N + 1)[None, :, None]
        ref, ref_lse = csum, np.log(np.arange(1, N + 1))[None].repeat(2, 0)
    else:
        ref = np.repeat(vf.mean(axis=1, keepdims=True), N, axis=1)
        ref_lse = np.full((2, N), math.log(N))
    check_o(o[0], ref, W.torch_dtype(dtype), "K=0")
    check_lse(lse[0], ref_lse, "K=0")


def test_deterministic(cuda):
    q, k, v = W.prefill_inputs(1, 4, 2, 777, 128, "bf16", seed=4)
    a = run(q, k, v, True, 0.1, cuda)
    b = run(q, k, v, True, 0.1, cuda)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_no_device_error_recorded(cuda):
    from exact_tiled_attention_11_gb300 import attn_device_error
    assert attn_device_error(clear=False) == 0
