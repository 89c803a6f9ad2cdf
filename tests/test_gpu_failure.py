"""Failure detection on the GPU without a fault: the bounded pipeline waits.

The self-test kernel's two warps wait, through the same bounded wait the attention
kernels use, on mbarriers that nothing arrives on.  The waits must give up (after
about one wait limit, the second through the shared abort flag), the device error
word must carry ATTN_DEVERR_WAIT_TIMEOUT, and the context must stay usable: an
attention call afterwards still matches the oracle and records no error.
"""
import time

import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_device_error, attn_fwd, attn_selftest_wait_timeout
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 0x1  # ATTN_DEVERR_WAIT_TIMEOUT in include/attn.h


def test_bounded_wait_gives_up_and_the_context_survives(cuda):
    attn_device_error(clear=True)
    t0 = time.perf_counter()
    gave_up = attn_selftest_wait_timeout(cuda)  # reads the result back: synchronises
    elapsed = time.perf_counter() - t0
    assert gave_up == [1, 1]
    # one wait limit (2 s), not two: the second warp stops on the first one's abort flag
    # or runs out at the same moment; well under the sum of two limits
    assert 1.5 < elapsed < 3.9, elapsed
    code = attn_device_error(clear=True)
    assert code & WAIT_TIMEOUT, hex(code)
    assert attn_device_error() == 0

    q, k, v = W.prefill_inputs(1, 4, 2, 300, 128, seed=7)
    o, lse = attn_fwd(q.to(cuda), k.to(cuda), v.to(cuda), causal=True, scale=128 ** -0.5)
    torch.cuda.synchronize()
    O, L = oracle.attention(q, k, v, causal=True, scale=128 ** -0.5)
    check_o(o.cpu(), O, torch.bfloat16, "after the self-test")
    check_lse(lse.cpu(), L, "after the self-test")
    assert attn_device_error() == 0
