"""Seeded random shapes for the tcgen05 prefill against the float64 oracle.

Each case draws batch, heads, GQA group, query and key lengths (1 .. 700, so the two
query tiles of a CTA get unequal, equal or no key tiles, and tiles end mid-way),
head dimension and causality, then compares O and the LSE element by element with
the oracle at the bf16 tolerance.  A second set draws ragged batches for the indptr
entry point.  The draws come from numpy's seeded generator; the inputs from the
same seeded recipe as the other tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_device_error, attn_fwd_cross, attn_fwd_varlen
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu


def _case(seed):
    r = np.random.default_rng(seed)
    Hkv = int(r.choice([1, 2, 4]))
    H = Hkv * int(r.choice([1, 2, 4]))
    return dict(B=int(r.integers(1, 3)), H=H, Hkv=Hkv, Nq=int(r.integers(1, 701)), Nk=int(r.integers(1, 701)),
                d=int(r.choice([64, 128])), causal=bool(r.integers(0, 2)))


@pytest.mark.parametrize("seed", range(24))
def test_random_cross_attention(cuda, seed):
    c = _case(seed)
    g = torch.Generator().manual_seed(1000 + seed)
    q = torch.randn(c["B"], c["H"], c["Nq"], c["d"], generator=g).to(torch.bfloat16)
    k = torch.randn(c["B"], c["Hkv"], c["Nk"], c["d"], generator=g).to(torch.bfloat16)
    v = torch.randn(c["B"], c["Hkv"], c["Nk"], c["d"], generator=g).to(torch.bfloat16)
    scale = 1 / math.sqrt(c["d"])
    o, lse = attn_fwd_cross(q.to(cuda), k.to(cuda), v.to(cuda), causal=c["causal"], scale=scale)
    torch.cuda.synchronize()
    O, L = oracle.attention(q, k, v, causal=c["causal"], scale=scale)
    check_o(o.cpu(), O, torch.bfloat16, str(c))
    check_lse(lse.cpu(), L, str(c))
    assert attn_device_error() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_ragged_batches(cuda, seed):
    r = np.random.default_rng(500 + seed)
    n = int(r.integers(1, 6))
    lens_q = [int(x) for x in r.integers(0, 400, n)]
    lens_k = [lq + int(x) for lq, x in zip(lens_q, r.integers(0, 300, n))]  # chunks: queries are the last tokens
    d = int(r.choice([64, 128]))
    causal = bool(r.integers(0, 2))
    H, Hkv = 8, 2
    g = torch.Generator().manual_seed(600 + seed)
    q = torch.randn(sum(lens_q), H, d, generator=g).to(torch.bfloat16)
    k = torch.randn(sum(lens_k), Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(sum(lens_k), Hkv, d, generator=g).to(torch.bfloat16)
    qo = torch.tensor([0] + list(np.cumsum(lens_q)), dtype=torch.int32)
    kvp = torch.tensor([0] + list(np.cumsum(lens_k)), dtype=torch.int32)
    o, lse = attn_fwd_varlen(q.to(cuda), k.to(cuda), v.to(cuda), qo.to(cuda), kvp.to(cuda), max(lens_q + [1]),
                             causal=causal)
    torch.cuda.synchronize()
    O, L = oracle.varlen_attention(q, k, v, qo, kvp, causal=causal, scale=1 / math.sqrt(d))
    what = f"lens_q={lens_q} lens_k={lens_k} d={d} causal={causal}"
    check_o(o.cpu(), O, torch.bfloat16, what)
    check_lse(lse.cpu(), L, what)
    assert attn_device_error() == 0
