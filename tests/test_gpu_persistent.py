"""The persistent form of the bf16 prefill (dense layout, causal, d = 128, many short items:
at least four (query-tile pair, batch, head) items per SM and at most 48 key tiles per item
on average), against the float64 oracle.  Barrier phases there run on across the items a CTA
takes, so these shapes cover item boundaries with unequal chain lengths, a ragged last pair
(N not a multiple of 256: chain B short or absent), GQA, and causal cross-attention with
N_q > N_k, where whole items attend no key at all (no K or V tile is loaded for them).  The
same shapes non-causal and at d = 64 run the one-item form and are checked alike."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_fwd, attn_fwd_cross, attn_device_error
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu


def _uses_persistent_form(B, H, Nq, Nk, causal, d, sms):
    items = ((Nq + 255) // 256) * B * H
    kt = (Nk + 127) // 128
    return d == 128 and causal and items >= 4 * sms and ((kt + 1) // 2 if causal else kt) <= 48


def _inputs(B, H, Hkv, Nq, Nk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16)
    return q, k, v


def _check_planes(o, lse, q, k, v, causal, scale, planes, what):
    for b, h in planes:
        rows = np.arange(q.shape[2])
        O, L = oracle.attention_rows(q, k, v, b, h, rows, causal=causal, scale=scale)
        check_o(o[b, h].cpu(), O, torch.bfloat16, f"{what} plane ({b}, {h})")
        check_lse(lse[b, h].cpu(), L, f"{what} plane ({b}, {h})")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d,N", [(128, 2000), (128, 1024), (64, 1920)])
def test_persistent_self_attention(cuda, causal, d, N):
    B, H, Hkv = 8, 32, 8
    sms = torch.cuda.get_device_properties(cuda).multi_processor_count
    assert _uses_persistent_form(B, H, N, N, causal, d, sms) == (causal and d == 128)
    q, k, v = _inputs(B, H, Hkv, N, N, d, seed=N + d + causal)
    attn_device_error(clear=True)
    o, lse = attn_fwd(q.to(cuda), k.to(cuda), v.to(cuda), causal=causal, scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    _check_planes(o, lse, q, k, v, causal, 1 / math.sqrt(d), [(0, 0), (3, 17), (7, 31), (5, 6)],
                  f"persistent N={N} d={d} causal={causal}")
    assert attn_device_error() == 0


@pytest.mark.parametrize("B,Nq,Nk", [(2, 4096, 1000), (8, 1000, 3000)])
def test_persistent_cross_attention(cuda, B, Nq, Nk):
    """N_q > N_k, causal: the first N_q - N_k query rows attend nothing (O = 0, LSE = -inf),
    and the items made only of such rows load no tile; N_q < N_k: every row sees extra keys."""
    H, Hkv, d = 32, 8, 128
    sms = torch.cuda.get_device_properties(cuda).multi_processor_count
    assert _uses_persistent_form(B, H, Nq, Nk, True, d, sms)
    q, k, v = _inputs(B, H, Hkv, Nq, Nk, d, seed=Nq + 3 * Nk)
    attn_device_error(clear=True)
    o, lse = attn_fwd_cross(q.to(cuda), k.to(cuda), v.to(cuda), causal=True, scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    if Nq > Nk:
        dead = Nq - Nk
        assert (o[:, :, :dead].float() == 0).all() and torch.isneginf(lse[:, :, :dead]).all()
        assert torch.isfinite(lse[:, :, dead:]).all()
    _check_planes(o, lse, q, k, v, True, 1 / math.sqrt(d), [(0, 0), (1, 31), (1, 9)],
                  f"persistent cross Nq={Nq} Nk={Nk}")
    assert attn_device_error() == 0
