"""The FP8 attention error bound (tests/parity.py ``fp8_bound`` and ``check_fp8``)
against a float64 emulation of the FP8 kernel's rounding scheme, on the CPU.

The emulation follows the kernel's arithmetic step by step, in float64 except at
the points where the kernel rounds by design: per 128-key tile, scores in log2
units, the lazy reference maximum (moved only when a tile's maximum exceeds it
by more than 2^8), p = 2^(s - m), p * r_j rounded to e4m3 (nearest, ties to
even) for the P V product, the unrounded p in the row sum, and the output
o~ * max v_scale / l rounded to bf16.  Its output must satisfy every check the
GPU tests apply (each element within the bound, mean square error within the
rounding model, no error correlated with O), and plausible mistakes planted in
it (P rounded toward zero, the last key tile dropped, V block scales shifted by
one block, o~ not rescaled when the reference moves) must each fail one.
The reference values are the oracle's.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as F
from tests.parity import check_fp8, check_lse, fp8_bound

LN2 = math.log(2.0)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _e4m3_toward_zero(x):
    a = np.abs(x)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    quantum = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / quantum) * quantum, F.E4M3_MAX), x)


def emulate_fp8_kernel(q_hat_rows, k_hat, v_codes, v_scale, rows, Nq, *, causal, scale, mistake=None, block=128):
    """O and LSE of the FP8 kernel's scheme for query rows ``rows`` of one head.

    q_hat_rows [n, d], k_hat [Nk, d]: dequantised blocks; v_codes [Nk, d]: V's e4m3
    values (codes decoded, before the block scale); v_scale: V block scales."""
    n, Nk = len(rows), k_hat.shape[0]
    d = v_codes.shape[1]
    s = (scale / LN2) * (q_hat_rows @ k_hat.T)
    if causal:
        s = np.where(np.arange(Nk)[None, :] <= np.asarray(rows)[:, None] + (Nk - Nq), s, -np.inf)
    vs = np.asarray(v_scale, dtype=np.float64)
    vmax = vs.max()
    r_blk = np.where(vs > 0, np.maximum(vs / vmax, 2.0 ** -20), 1.0)
    if mistake == "vscale_shifted":
        r_blk = np.roll(r_blk, 1)
    rnd = _e4m3_toward_zero if mistake == "p_toward_zero" else F.e4m3_round
    tiles = list(range(-(-Nk // block)))
    if mistake == "drop_last_tile" and len(tiles) > 1:
        tiles = tiles[:-1]
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    o = np.zeros((n, d))
    for t in tiles:
        cols = slice(t * block, min(Nk, (t + 1) * block))
        st = s[:, cols]
        tmax = st.max(axis=1)
        move = tmax > m + 8.0
        m_new = np.where(move, tmax, m)
        corr = np.where(move, np.where(np.isfinite(m), np.exp2(m - np.where(np.isfinite(m_new), m_new, 0.0)), 0.0), 1.0)
        ref = np.where(np.isfinite(m_new), m_new, 0.0)
        p = np.exp2(st - ref[:, None])
        pq = rnd(p * r_blk[t])
        o = (o if mistake == "no_rescale" else o * corr[:, None]) + pq @ v_codes[cols]
        l = l * corr + p.sum(axis=1)
        m = m_new
    live = l > 0
    O = _bf16(np.where(live[:, None], o * vmax / np.where(live, l, 1.0)[:, None], 0.0))
    LSE = np.where(live, (np.where(live, m, 0.0) + np.log2(np.where(live, l, 1.0))) * LN2, -np.inf)
    return O, LSE


def _case(B, H, Hkv, Nq, Nk, seed, q_mult=1.0, tiny_v_block=None, zero_v_block=None):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Nq, 128, generator=g) * q_mult
    k = torch.randn(B, Hkv, Nk, 128, generator=g)
    v = torch.randn(B, Hkv, Nk, 128, generator=g)
    if tiny_v_block is not None:
        v[:, :, tiny_v_block * 128:(tiny_v_block + 1) * 128] *= 1e-7
    if zero_v_block is not None:
        v[:, :, zero_v_block * 128:(zero_v_block + 1) * 128] = 0
    q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    ref = F.fp8_quantize(q, k, v, np.where(np.arange(128) % 3 == 0, -1.0, 1.0))
    # scales as the kernel stores them (fp32), blocks dequantised with those
    for name, codes, hat in (("q_scale", "q8", "q_hat"), ("k_scale", "k8", "k_hat"), ("v_scale", "v8", "v_hat")):
        s32 = ref[name].astype(np.float32).astype(np.float64)
        ref[name] = s32
        ref[hat] = F.e4m3_decode(ref[codes]) * np.repeat(s32, 128, axis=-1)[..., :ref[codes].shape[2], None]
    return ref


def _run(ref, causal, mistake=None):
    """Emulated outputs of every head against the oracle: (O errors' checks, LSE)."""
    scale = 1 / math.sqrt(128)
    B, H, Nq, _ = ref["q_hat"].shape
    Hkv = ref["k_hat"].shape[1]
    rows = np.arange(Nq)
    outs, refs, tols, sig2 = [], [], [], []
    for b in range(B):
        for h in range(H):
            kv = h // (H // Hkv)
            Oe, Le = emulate_fp8_kernel(ref["q_hat"][b, h], ref["k_hat"][b, kv], F.e4m3_decode(ref["v8"][b, kv]),
                                        ref["v_scale"][b, kv], rows, Nq, causal=causal, scale=scale,
                                        mistake=mistake)
            Oo, Lo = oracle.attention_rows(ref["q_hat"], ref["k_hat"], ref["v_hat"], b, h, rows, causal=causal,
                                           scale=scale)
            P, _ = oracle.attention_weights(ref["q_hat"], ref["k_hat"], b, h, rows, causal=causal, scale=scale)
            tol, s2 = fp8_bound(P, Oo, ref["q_hat"][b, h], ref["k_hat"][b, kv], ref["v_hat"][b, kv],
                                ref["v_scale"][b, kv], scale=scale)
            check_lse(Le, Lo, f"head {h}")
            outs.append(Oe), refs.append(Oo), tols.append(tol), sig2.append(s2)
    return [np.concatenate(x) for x in (outs, refs, tols, sig2)]


CASES = {
    "n300": dict(B=1, H=2, Hkv=1, Nq=300, Nk=300, seed=1),
    "gqa513": dict(B=1, H=4, Hkv=2, Nq=513, Nk=513, seed=2),
    "cross100x700": dict(B=1, H=2, Hkv=1, Nq=100, Nk=700, seed=3),
    "cross700x100": dict(B=1, H=2, Hkv=2, Nq=700, Nk=100, seed=4),
    "large_scores_q30": dict(B=1, H=2, Hkv=1, Nq=640, Nk=640, seed=5, q_mult=30.0),
    "tiny_and_zero_v_blocks": dict(B=1, H=2, Hkv=1, Nq=400, Nk=520, seed=6, tiny_v_block=1, zero_v_block=2),
}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_emulated_kernel_within_bound(name, causal):
    O, R, tol, s2 = _run(_case(**CASES[name]), causal)
    worst, ms_ratio, slope = check_fp8(O, R, tol, s2, name)
    assert ms_ratio < 0.7, ms_ratio  # the model's own expectation is at most 1/3 plus the deterministic terms


@pytest.mark.parametrize("mistake", ["p_toward_zero", "drop_last_tile", "vscale_shifted", "no_rescale"])
def test_planted_mistake_fails_a_check(mistake):
    caught = []
    for name in ("gqa513", "large_scores_q30", "cross100x700"):
        for causal in (False, True):
            try:
                O, R, tol, s2 = _run(_case(**CASES[name]), causal, mistake)
                check_fp8(O, R, tol, s2, name)
            except AssertionError as e:
                caught.append((name, causal, str(e)[:80]))
    assert caught, f"no check caught {mistake}"
