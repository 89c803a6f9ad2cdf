"""merge_partials parity: the CUDA merge kernel (through the C ABI) against the oracle's merge rule."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import merge_partials
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu


def make_partials(B, H, S, d, counts, seed):
    """Partials of real key subsets: (m, l, o~) of random score/value chunks, per (b, h, s)."""
    rng = np.random.default_rng(seed)
    m = np.full((B, H, S), -np.inf)
    l = np.zeros((B, H, S))
    o = np.zeros((B, H, S, d))
    ref_o = np.zeros((B, H, d))
    ref_lse = np.full((B, H), -np.inf)
    for b in range(B):
        for h in range(H):
            parts = []
            for s in range(counts[b]):
                n = int(rng.integers(0, 40))       # 0 keys: an empty partial (-inf, 0, 0)
                sc = rng.standard_normal(n) * 8
                v = rng.standard_normal((n, d))
                parts.append(oracle.partial_state(sc, v))
                m[b, h, s], l[b, h, s], o[b, h, s] = parts[-1]
            if parts:
                ref_o[b, h], ref_lse[b, h] = oracle.finalize(*oracle.merge_partials(parts))
    # fp32 storage, as the kernel reads it; the oracle re-merges the stored values
    m32, l32, o32 = m.astype(np.float32), l.astype(np.float32), o.astype(np.float32)
    for b in range(B):
        for h in range(H):
            parts = [(m32[b, h, s], l32[b, h, s], o32[b, h, s]) for s in range(counts[b])]
            if parts:
                ref_o[b, h], ref_lse[b, h] = oracle.finalize(*oracle.merge_partials(parts))
    return m32, l32, o32, ref_o, ref_lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_merge_variable_counts(cuda, d, out):
    B, H, S = 6, 5, 9
    counts = [9, 1, 0, 4, 7, 2]
    m, l, o, ref_o, ref_lse = make_partials(B, H, S, d, counts, seed=d)
    t = lambda a: torch.from_numpy(a).to(cuda)  # noqa: E731
    O, L = merge_partials(t(m), t(l), t(o), torch.tensor(counts, dtype=torch.int32, device=cuda), out_dtype=out)
    torch.cuda.synchronize()
    # fp32 outputs of unit scale: max |dO| <= 1e-5 like the fp32 attention path
    check_o(O.cpu(), ref_o, out, f"merge d={d}")
    check_lse(L.cpu(), ref_lse, f"merge d={d}")
    assert (O[2] == 0).all() and torch.isneginf(L[2]).all()


def test_merge_all_parts_when_counts_null(cuda):
    B, H, S, d = 3, 4, 5, 128
    m, l, o, ref_o, ref_lse = make_partials(B, H, S, d, [S] * B, seed=1)
    t = lambda a: torch.from_numpy(a).to(cuda)  # noqa: E731
    O, L = merge_partials(t(m), t(l), t(o), None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_o(O.cpu(), ref_o, torch.float32, "merge all")
    check_lse(L.cpu(), ref_lse, "merge all")


def test_merge_order_independent(cuda):
    """Permuting the partials changes nothing beyond fp32 rounding (merge is associative)."""
    B, H, S, d = 2, 3, 16, 128
    m, l, o, ref_o, _ = make_partials(B, H, S, d, [S] * B, seed=2)
    perm = np.random.default_rng(0).permutation(S)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda)  # noqa: E731
    O1, _ = merge_partials(t(m), t(l), t(o), None, out_dtype=torch.float32)
    O2, _ = merge_partials(t(m[:, :, perm]), t(l[:, :, perm]), t(o[:, :, perm]), None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert (O1 - O2).abs().max().item() <= 1e-5
