"""Long contexts: prefill at 64K and 128K tokens, decode of a 128K-token sequence.

Beyond the benchmark workloads' lengths, so that any 32-bit index product, tile
count or page offset that would overflow or wrap shows here.  The oracle
computes sampled rows (prefill: the first and last rows of the first, middle
and last tiles, plus random rows) and the long sequence in full (decode).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_decode_paged, attn_device_error, attn_fwd
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu


def _rows(N, seed):
    fixed = [0, 1, 127, 128, N // 2 - 1, N // 2, N - 129, N - 128, N - 1]
    return np.unique(np.concatenate([fixed, np.random.default_rng(seed).integers(0, N, 12)]))


@pytest.mark.parametrize("N,d,causal,q_mult", [(131072, 128, True, 1.0), (65536, 64, False, 1.0),
                                               (65536, 128, True, 40.0)])
def test_long_prefill_sampled_rows(cuda, N, d, causal, q_mult):
    B, H, Hkv = 1, 2, 1
    q, k, v = W.prefill_inputs(B, H, Hkv, N, d, "bf16", q_mult=q_mult, seed=N // 1024 + d)
    scale = 1 / math.sqrt(d)
    o, lse = attn_fwd(q.to(cuda), k.to(cuda), v.to(cuda), causal=causal, scale=scale)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    for h in range(H):
        rows = _rows(N, h)
        O, L = oracle.attention_rows(q, k, v, 0, h, rows, causal=causal, scale=scale)
        what = f"N={N} d={d} causal={causal} x{q_mult} h{h}"
        check_o(o[0, h, rows], O, torch.bfloat16, what)
        check_lse(lse[0, h, rows], L, what)
    assert attn_device_error() == 0


@pytest.mark.parametrize("num_splits", [0, 5])
def test_long_decode_sequence(cuda, num_splits):
    lens = [131072, 1, 4097]   # 8192 pages, one token, a page past a 256-page boundary
    kv = W.decode_inputs(len(lens), 8, 2, 128, 16, 1, 1, seed=23, kv_lens=lens)
    t = [x.to(cuda) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
    o, lse = attn_decode_paged(*t, scale=1 / math.sqrt(128), num_splits=num_splits)
    torch.cuda.synchronize()
    O, L = oracle.decode_paged(kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens, scale=1 / math.sqrt(128))
    check_o(o.cpu(), O, torch.bfloat16, f"long decode, num_splits={num_splits}")
    check_lse(lse.cpu(), L, f"long decode, num_splits={num_splits}")
    assert attn_device_error() == 0
