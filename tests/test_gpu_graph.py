"""CUDA-graph capture of the decode step ("3.4 Attention Kernels", "Kernel launch
overhead and CUDA graphs": capture once, copy each step's inputs into the
captured static buffers, replay).

The library allocates nothing and never synchronises, so attn_decode_paged (with
a caller-owned workspace) and attn_fwd can be captured; replays on new inputs
must equal eager calls bit for bit and match the oracle.
"""
import math

import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import (attn_decode_max_splits, attn_decode_paged, attn_decode_workspace_size,
                                            attn_fwd)
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu


def test_decode_step_graph_replay_matches_eager_and_oracle(cuda):
    B, H, Hkv, d, ps, maxp = 6, 32, 8, 128, 16, 64
    # one pool large enough for every step's sequences; steps differ in q, lengths and page tables
    P = B * maxp
    g = torch.Generator().manual_seed(3)
    k_pages = torch.randn(P, Hkv, ps, d, generator=g).to(torch.bfloat16).to(cuda)
    v_pages = torch.randn(P, Hkv, ps, d, generator=g).to(torch.bfloat16).to(cuda)

    def step_inputs(seed):
        gg = torch.Generator().manual_seed(seed)
        lens = torch.randint(1, maxp * ps + 1, (B,), generator=gg, dtype=torch.int32)
        perm = torch.randperm(P, generator=gg).to(torch.int32).reshape(B, maxp)
        q = torch.randn(B, H, d, generator=gg).to(torch.bfloat16)
        return q, perm, lens

    S = attn_decode_max_splits(B, H, Hkv, maxp)
    ws = torch.empty(attn_decode_workspace_size(B, H, d, S), dtype=torch.uint8, device=cuda)
    sq = torch.empty(B, H, d, dtype=torch.bfloat16, device=cuda)
    spt = torch.empty(B, maxp, dtype=torch.int32, device=cuda)
    slen = torch.empty(B, dtype=torch.int32, device=cuda)
    so = torch.empty(B, H, d, dtype=torch.bfloat16, device=cuda)
    slse = torch.empty(B, H, dtype=torch.float32, device=cuda)

    def load(q, pt, lens):
        sq.copy_(q)
        spt.copy_(pt)
        slen.copy_(lens)

    load(*step_inputs(100))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            attn_decode_paged(sq, k_pages, v_pages, spt, slen, so, slse, num_splits=S, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        attn_decode_paged(sq, k_pages, v_pages, spt, slen, so, slse, num_splits=S, workspace=ws)

    for seed in (1, 2, 3):
        q, pt, lens = step_inputs(seed)
        load(q, pt, lens)
        graph.replay()
        torch.cuda.synchronize()
        o_graph, lse_graph = so.clone(), slse.clone()
        o_eager, lse_eager = attn_decode_paged(q.to(cuda), k_pages, v_pages, pt.to(cuda), lens.to(cuda),
                                               num_splits=S)
        torch.cuda.synchronize()
        assert torch.equal(o_graph, o_eager) and torch.equal(lse_graph, lse_eager)
        O, L = oracle.decode_paged(q, k_pages.cpu(), v_pages.cpu(), pt, lens, scale=1 / math.sqrt(d))
        check_o(o_graph.cpu(), O, torch.bfloat16, f"graph step {seed}")
        check_lse(lse_graph.cpu(), L, f"graph step {seed}")


def test_prefill_graph_replay_matches_eager(cuda):
    B, H, Hkv, N, d = 1, 8, 2, 700, 128
    sq = torch.empty(B, H, N, d, dtype=torch.bfloat16, device=cuda)
    sk = torch.empty(B, Hkv, N, d, dtype=torch.bfloat16, device=cuda)
    sv = torch.empty_like(sk)
    so = torch.empty_like(sq)
    slse = torch.empty(B, H, N, dtype=torch.float32, device=cuda)
    q, k, v = W.prefill_inputs(B, H, Hkv, N, d, "bf16", seed=1)
    sq.copy_(q), sk.copy_(k), sv.copy_(v)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            attn_fwd(sq, sk, sv, so, slse, causal=True)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        attn_fwd(sq, sk, sv, so, slse, causal=True)
    for seed in (2, 3):
        q, k, v = W.prefill_inputs(B, H, Hkv, N, d, "bf16", seed=seed)
        sq.copy_(q), sk.copy_(k), sv.copy_(v)
        graph.replay()
        torch.cuda.synchronize()
        o_eager, lse_eager = attn_fwd(q.to(cuda), k.to(cuda), v.to(cuda), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(so, o_eager) and torch.equal(slse, lse_eager)
