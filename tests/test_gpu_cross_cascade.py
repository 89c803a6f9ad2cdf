"""Parity of attn_fwd_cross (Nq != Nk, causal mask aligned to the last key) and of
attn_cascade_decode (shared prefix + own paged suffix) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_cascade_decode, attn_decode_paged, attn_device_error, attn_fwd_cross
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu


def _qkv(B, H, Hkv, Nq, Nk, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    t = W.torch_dtype(dtype)
    q = torch.randn(B, H, Nq, d, generator=g).to(t)
    k = torch.randn(B, Hkv, Nk, d, generator=g).to(t)
    v = torch.randn(B, Hkv, Nk, d, generator=g).to(t)
    return q, k, v


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk,d", [(100, 300, 128), (300, 100, 128), (128, 1000, 64), (1, 777, 128),
                                     (500, 500, 64), (257, 513, 128), (640, 129, 64)])
def test_cross_attention(cuda, Nq, Nk, d, causal, dtype):
    q, k, v = _qkv(2, 4, 2, Nq, Nk, d, dtype, seed=Nq + Nk + d)
    o, lse = attn_fwd_cross(q.to(cuda), k.to(cuda), v.to(cuda), causal=causal)
    torch.cuda.synchronize()
    O, L = oracle.attention(q, k, v, causal=causal, scale=1 / math.sqrt(d))
    check_o(o.cpu(), O, W.torch_dtype(dtype), f"cross {Nq}x{Nk} d{d} causal={causal}")
    check_lse(lse.cpu(), L, f"cross {Nq}x{Nk} d{d} causal={causal}")


def test_cross_attention_chunked_prefill_rows(cuda):
    """The last Nq rows of causal self-attention over Nk tokens, computed as a chunk of
    queries against the whole cache, match the oracle's rows."""
    Nk, Nq, d = 2000, 300, 128
    q_all, k, v = _qkv(1, 8, 2, Nk, Nk, d, "bf16", seed=9)
    q = q_all[:, :, Nk - Nq:].contiguous()
    o, lse = attn_fwd_cross(q.to(cuda), k.to(cuda), v.to(cuda), causal=True)
    torch.cuda.synchronize()
    for h in range(8):
        O, L = oracle.attention_rows(q_all, k, v, 0, h, np.arange(Nk - Nq, Nk), causal=True, scale=1 / math.sqrt(d))
        check_o(o[0, h].cpu(), O, torch.bfloat16, f"chunk h{h}")
        check_lse(lse[0, h].cpu(), L, f"chunk h{h}")


def _cascade_case(B, H, Hkv, Lp, lens, seed):
    kv = W.decode_inputs(B, H, Hkv, 128, 16, 1, 1, seed=seed, kv_lens=lens)
    g = torch.Generator().manual_seed(seed + 1000)
    pk = torch.randn(Hkv, Lp, 128, generator=g).to(torch.bfloat16)
    pv = torch.randn(Hkv, Lp, 128, generator=g).to(torch.bfloat16)
    return kv, pk, pv


@pytest.mark.parametrize("Lp", [0, 1, 100, 1000, 2048])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_cascade_decode(cuda, Lp, num_splits):
    lens = [0, 1, 16, 300, 4000, 77]
    kv, pk, pv = _cascade_case(len(lens), 32, 8, Lp, lens, seed=Lp + 7)
    t = [x.to(cuda) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
    o, lse = attn_cascade_decode(t[0], pk.to(cuda), pv.to(cuda), *t[1:], num_splits=num_splits)
    torch.cuda.synchronize()
    O, L = oracle.cascade_decode(kv.q, pk, pv, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens,
                                 scale=1 / math.sqrt(128))
    if Lp == 0:
        # request 0 has neither prefix nor suffix: O = 0, LSE = -inf
        assert (o[0] == 0).all() and torch.isneginf(lse[0]).all()
    check_o(o.cpu(), O, torch.bfloat16, f"cascade Lp={Lp}")
    check_lse(lse.cpu(), L, f"cascade Lp={Lp}")
    assert attn_device_error() == 0


def test_cascade_many_requests_gqa(cuda):
    """300 requests (more than two 128-row query tiles) sharing a 3000-token prefix."""
    B = 300
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 600, B).tolist()
    kv, pk, pv = _cascade_case(B, 32, 8, 3000, lens, seed=11)
    t = [x.to(cuda) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
    o, lse = attn_cascade_decode(t[0], pk.to(cuda), pv.to(cuda), *t[1:])
    torch.cuda.synchronize()
    seqs = [0, 1, 127, 128, 255, 256, 299]
    O, L = oracle.cascade_decode(kv.q, pk, pv, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens,
                                 scale=1 / math.sqrt(128), seqs=seqs)
    check_o(o[seqs].cpu(), O[seqs], torch.bfloat16, "cascade 300")
    check_lse(lse[seqs].cpu(), L[seqs], "cascade 300")
    # the same requests with the prefix held as ordinary attention keys give the same answer
    assert torch.isfinite(o.float()).all()


def test_cascade_matches_decode_when_prefix_is_in_the_pages(cuda):
    """A page-aligned prefix held once as shared pages at the front of every page table
    (plain paged decode) and the same prefix passed to attn_cascade_decode agree."""
    B, H, Hkv, d, ps = 4, 32, 8, 128, 16
    npre = 40
    lens = [10, 0, 333, 1500]
    kv = W.decode_inputs(B, H, Hkv, d, ps, 1, 1, seed=21, kv_lens=lens)
    g = torch.Generator().manual_seed(22)
    pre_pages_k = torch.randn(npre, Hkv, ps, d, generator=g).to(torch.bfloat16)
    pre_pages_v = torch.randn(npre, Hkv, ps, d, generator=g).to(torch.bfloat16)
    P = kv.k_pages.shape[0]
    kp = torch.cat([kv.k_pages, pre_pages_k])
    vp = torch.cat([kv.v_pages, pre_pages_v])
    table = torch.cat([torch.arange(P, P + npre, dtype=torch.int32).repeat(B, 1), kv.page_table], dim=1)
    # the suffix pages of each request follow the shared prefix pages in its row
    o_d, lse_d = attn_decode_paged(kv.q.to(cuda), kp.to(cuda), vp.to(cuda), table.to(cuda),
                                   (kv.kv_lens + npre * ps).to(cuda))
    pk = pre_pages_k.permute(1, 0, 2, 3).reshape(Hkv, npre * ps, d).contiguous()
    pv = pre_pages_v.permute(1, 0, 2, 3).reshape(Hkv, npre * ps, d).contiguous()
    o_c, lse_c = attn_cascade_decode(kv.q.to(cuda), pk.to(cuda), pv.to(cuda), kv.k_pages.to(cuda),
                                     kv.v_pages.to(cuda), kv.page_table.to(cuda), kv.kv_lens.to(cuda))
    torch.cuda.synchronize()
    check_o(o_c.cpu(), o_d.cpu(), torch.bfloat16, "cascade vs paged")
    check_lse(lse_c.cpu(), lse_d.cpu(), "cascade vs paged")


@pytest.mark.parametrize("Lp", [0, 300])
def test_cascade_decode_head_dim_64(cuda, Lp):
    lens = [0, 1, 16, 700]
    kv = W.decode_inputs(len(lens), 16, 4, 64, 16, 1, 1, seed=Lp + 3, kv_lens=lens)
    g = torch.Generator().manual_seed(Lp + 4)
    pk = torch.randn(4, Lp, 64, generator=g).to(torch.bfloat16)
    pv = torch.randn(4, Lp, 64, generator=g).to(torch.bfloat16)
    t = [x.to(cuda) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
    o, lse = attn_cascade_decode(t[0], pk.to(cuda), pv.to(cuda), *t[1:])
    torch.cuda.synchronize()
    O, L = oracle.cascade_decode(kv.q, pk, pv, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens,
                                 scale=1 / math.sqrt(64))
    check_o(o.cpu(), O, torch.bfloat16, f"cascade d=64 Lp={Lp}")
    check_lse(lse.cpu(), L, f"cascade d=64 Lp={Lp}")
    assert attn_device_error() == 0
