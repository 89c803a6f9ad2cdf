"""attn_fwd_host: host tensors in and out, copies pipelined with the attention inside the
call.  Its result must equal attn_fwd on the same inputs bit for bit (the same kernel on
each group of KV heads), and match the oracle."""
import math

import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_device_error, attn_fwd, attn_fwd_host
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,H,Hkv,N,d,causal", [(1, 8, 2, 700, 128, True), (3, 4, 4, 257, 64, False),
                                                (2, 16, 8, 1024, 128, True), (1, 2, 1, 130, 128, True)])
def test_fwd_host_matches_attn_fwd(cuda, B, H, Hkv, N, d, causal, dtype):
    q, k, v = W.prefill_inputs(B, H, Hkv, N, d, dtype, seed=N + B)
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = attn_fwd_host(qp, kp, vp, causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = attn_fwd(q.to(cuda), k.to(cuda), v.to(cuda), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref.cpu()) and torch.equal(lse, lse_ref.cpu())
    heads = [0, H - 1]
    for h in heads:
        rows = torch.arange(0, N, max(1, N // 37))
        O, L = oracle.attention_rows(q, k, v, B - 1, h, rows.numpy(), causal=causal, scale=1 / math.sqrt(d))
        check_o(o[B - 1, h, rows], O, W.torch_dtype(dtype), f"host path h{h}")
        check_lse(lse[B - 1, h, rows], L, f"host path h{h}")
    assert attn_device_error() == 0


def test_fwd_host_orders_after_earlier_work_and_reuses_buffers(cuda):
    """Device buffers reused across calls on one stream: each call's copies wait for the
    previous call's kernels, and each result is complete at the stream's sync point."""
    B, H, Hkv, N, d = 1, 8, 2, 512, 128
    bufs = (torch.empty(B, H, N, d, dtype=torch.bfloat16, device=cuda),
            torch.empty(B, Hkv, N, d, dtype=torch.bfloat16, device=cuda),
            torch.empty(B, Hkv, N, d, dtype=torch.bfloat16, device=cuda),
            torch.empty(B, H, N, d, dtype=torch.bfloat16, device=cuda),
            torch.empty(B, H, N, dtype=torch.float32, device=cuda))
    stream = torch.cuda.Stream()
    outs = []
    inputs = [W.prefill_inputs(B, H, Hkv, N, d, "bf16", seed=s) for s in (1, 2, 3)]
    with torch.cuda.stream(stream):
        for (q, k, v) in inputs:
            outs.append(attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), buffers=bufs, causal=True,
                                      stream=stream))
    stream.synchronize()
    for (q, k, v), (o, lse) in zip(inputs, outs):
        o_ref, lse_ref = attn_fwd(q.to(cuda), k.to(cuda), v.to(cuda), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref.cpu()) and torch.equal(lse, lse_ref.cpu())
