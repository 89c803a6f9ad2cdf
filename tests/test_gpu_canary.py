"""Guard regions: no kernel writes outside its outputs.

Every output below (O, LSE, the decode workspace, the FP8 codes and scales) is a view
into a larger device buffer whose bytes before and after it hold a fixed pattern.  The
shapes are ragged and odd (partial 128-row tiles, sequences of 0, 1 and 17 tokens,
page-table tails), where an off-by-one in a tile bound would store past the end.  After
each call the guard bytes must be untouched and no kernel may have recorded an error.
"""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_11_gb300 import (
    Fp8Inputs,
    attn_cascade_decode,
    attn_cascade_workspace_size,
    attn_decode_max_splits,
    attn_decode_paged,
    attn_decode_workspace_size,
    attn_device_error,
    attn_fp8_padded_keys,
    attn_fp8_quantize,
    attn_fwd,
    attn_fwd_cross,
    attn_fwd_fp8,
    attn_fwd_paged,
    attn_fwd_varlen,
    merge_partials,
)
from exact_tiled_attention_11_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096     # bytes on each side (keeps every view 256-byte aligned)
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` inside a pattern-filled device buffer."""

    def __init__(self, shape, dtype, device):
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.t = self.buf[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        return bool((self.buf[:GUARD] == PATTERN).all()) and bool((self.buf[-GUARD:] == PATTERN).all())


def _check(*guarded):
    torch.cuda.synchronize()
    for i, g in enumerate(guarded):
        assert g.intact(), f"guard region {i} was written"
    assert attn_device_error() == 0


@pytest.mark.parametrize("d,dtype", [(64, torch.bfloat16), (128, torch.bfloat16), (64, torch.float32)])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill(cuda, d, dtype, causal):
    B, H, Hkv, N = 2, 4, 2, 300
    q, k, v = (t.to(cuda) for t in W.prefill_inputs(B, H, Hkv, N, d, dtype="bf16" if dtype == torch.bfloat16 else "f32",
                                                     seed=d))
    o = Guarded((B, H, N, d), dtype, cuda)
    lse = Guarded((B, H, N), torch.float32, cuda)
    attn_fwd(q, k, v, o.t, lse.t, causal=causal)
    _check(o, lse)


def test_cross_attention(cuda):
    B, H, Hkv, Nq, Nk, d = 1, 4, 1, 130, 517, 128
    g = torch.Generator().manual_seed(3)
    q = torch.randn(B, H, Nq, d, generator=g).to(torch.bfloat16).to(cuda)
    k = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16).to(cuda)
    v = torch.randn(B, Hkv, Nk, d, generator=g).to(torch.bfloat16).to(cuda)
    o = Guarded((B, H, Nq, d), torch.bfloat16, cuda)
    lse = Guarded((B, H, Nq), torch.float32, cuda)
    attn_fwd_cross(q, k, v, o.t, lse.t, causal=True)
    _check(o, lse)


def test_varlen_and_paged_prefill(cuda):
    H, Hkv, d = 8, 2, 128
    lens = [1, 0, 130, 257, 17]
    g = torch.Generator().manual_seed(5)
    tq = sum(lens)
    q = torch.randn(tq, H, d, generator=g).to(torch.bfloat16).to(cuda)
    k = torch.randn(tq, Hkv, d, generator=g).to(torch.bfloat16).to(cuda)
    v = torch.randn(tq, Hkv, d, generator=g).to(torch.bfloat16).to(cuda)
    ind = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=cuda)
    o = Guarded((tq, H, d), torch.bfloat16, cuda)
    lse = Guarded((tq, H), torch.float32, cuda)
    attn_fwd_varlen(q, k, v, ind, ind, max(lens), o.t, lse.t, causal=True)
    _check(o, lse)

    kv = W.decode_inputs(len(lens), H, Hkv, d, 16, 1, 1, seed=6, kv_lens=lens)
    o2 = Guarded((tq, H, d), torch.bfloat16, cuda)
    lse2 = Guarded((tq, H), torch.float32, cuda)
    attn_fwd_paged(q, kv.k_pages.to(cuda), kv.v_pages.to(cuda), kv.page_table.to(cuda), kv.kv_lens.to(cuda), ind,
                   max(lens), o2.t, lse2.t, causal=True)
    _check(o2, lse2)


@pytest.mark.parametrize("num_splits", [0, 3])
def test_decode_and_merge(cuda, num_splits):
    lens = [1, 0, 16, 17, 300, 4100]
    B, H, Hkv, d = len(lens), 32, 8, 128
    kv = W.decode_inputs(B, H, Hkv, d, 16, 1, 1, seed=7, kv_lens=lens)
    t = [x.to(cuda) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
    S = num_splits if num_splits > 0 else attn_decode_max_splits(B, H, Hkv, kv.page_table.shape[1])
    ws = Guarded((attn_decode_workspace_size(B, H, d, S),), torch.uint8, cuda)
    o = Guarded((B, H, d), torch.bfloat16, cuda)
    lse = Guarded((B, H), torch.float32, cuda)
    attn_decode_paged(*t, o.t, lse.t, num_splits=num_splits, workspace=ws.t)
    _check(ws, o, lse)

    S = 5
    g = torch.Generator().manual_seed(8)
    m = torch.randn(B, H, S, generator=g).to(cuda)
    l = torch.rand(B, H, S, generator=g).to(cuda) + 0.5
    ot = torch.randn(B, H, S, d, generator=g).to(cuda)
    parts = torch.tensor([0, 1, 5, 2, 3, 4], dtype=torch.int32, device=cuda)
    o2 = Guarded((B, H, d), torch.bfloat16, cuda)
    lse2 = Guarded((B, H), torch.float32, cuda)
    merge_partials(m, l, ot, parts, o=o2.t, lse=lse2.t)
    _check(o2, lse2)


def test_cascade_decode(cuda):
    lens = [0, 1, 17, 300]
    B, H, Hkv, d, Lp = len(lens), 32, 8, 128, 129
    kv = W.decode_inputs(B, H, Hkv, d, 16, 1, 1, seed=9, kv_lens=lens)
    g = torch.Generator().manual_seed(10)
    pk = torch.randn(Hkv, Lp, d, generator=g).to(torch.bfloat16).to(cuda)
    pv = torch.randn(Hkv, Lp, d, generator=g).to(torch.bfloat16).to(cuda)
    t = [x.to(cuda) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
    S = 2
    ws = Guarded((attn_cascade_workspace_size(B, H, d, S),), torch.uint8, cuda)
    o = Guarded((B, H, d), torch.bfloat16, cuda)
    lse = Guarded((B, H), torch.float32, cuda)
    attn_cascade_decode(t[0], pk, pv, *t[1:], o.t, lse.t, num_splits=S, workspace=ws.t)
    _check(ws, o, lse)


def test_fp8_quantize_and_attention(cuda):
    B, H, Hkv, N, d = 1, 4, 2, 300, 128
    q, k, v = (t.to(cuda) for t in W.prefill_inputs(B, H, Hkv, N, d, seed=11))
    nb = -(-N // 128)
    parts = [Guarded((B, H, N, d), torch.uint8, cuda), Guarded((B, Hkv, N, d), torch.uint8, cuda),
             Guarded((B, Hkv, d, attn_fp8_padded_keys(N)), torch.uint8, cuda),
             Guarded((B, H, nb), torch.float32, cuda), Guarded((B, Hkv, nb), torch.float32, cuda),
             Guarded((B, Hkv, nb), torch.float32, cuda)]
    x = attn_fp8_quantize(q, k, v, W.fp8_signs(d).to(cuda), Fp8Inputs(*(p.t for p in parts)))
    _check(*parts)
    o = Guarded((B, H, N, d), torch.bfloat16, cuda)
    lse = Guarded((B, H, N), torch.float32, cuda)
    attn_fwd_fp8(x, o.t, lse.t, causal=True)
    _check(o, lse)
