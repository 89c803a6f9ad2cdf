"""attn_decode_paged_noalloc: paged decode for callers that cannot allocate device memory.

Such callers (a plugin or custom op that another runtime hands only its input and
output buffers, or a serving loop that must not call cudaMalloc because it can
synchronise the device) get the same decode with the partials kept in a fixed
device array of the library.  These checks call the entry point through the C
ABI and compare it with attn_decode_paged given an ordinary workspace and with
the float64 oracle, on two calls in a row so that the second call runs on the
scratch contents the first one left behind.
"""
import ctypes
import math

import pytest
import torch

import oracle

from exact_tiled_attention_11_gb300 import attn_decode_paged, load_library
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu

ATTN_ERR_WORKSPACE = 3


def _call_noalloc(lib, q, kp, vp, pt, kl, o, lse, num_splits):
    B, H, d = q.shape
    P, Hkv, ps, _ = kp.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.attn_decode_paged_noalloc(p(q), p(kp), p(vp), p(pt), p(kl), p(o), p(lse), B, H, Hkv, d, ps,
                                         pt.shape[1], P, 1.0 / math.sqrt(d), num_splits,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_decode_on_two_calls(cuda):
    lib = load_library()
    cases = [
        (W.decode_inputs(6, 32, 8, 128, 16, 1, 1, seed=11, kv_lens=[1, 17, 300, 5000, 12000, 2049]), 0),
        (W.decode_inputs(4, 32, 8, 128, 16, 1, 1, seed=12, kv_lens=[9000, 3, 640, 16]), 7),
    ]
    for kv, splits in cases:
        t = [x.to(cuda) for x in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]
        B, H, d = kv.q.shape
        o = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device=cuda)
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=cuda)
        assert _call_noalloc(lib, *t, o, lse, splits) == 0
        o_ref, lse_ref = attn_decode_paged(*t, num_splits=splits)
        torch.cuda.synchronize()
        check_o(o.cpu(), o_ref.cpu(), torch.bfloat16, f"noalloc splits={splits}")
        check_lse(lse.cpu(), lse_ref.cpu(), f"noalloc splits={splits}")
        O, L = oracle.decode_paged(kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens, scale=1.0 / math.sqrt(d))
        check_o(o.cpu(), O, torch.bfloat16, f"noalloc vs oracle splits={splits}")
        check_lse(lse.cpu(), L, f"noalloc vs oracle splits={splits}")


def test_noalloc_rejects_requests_beyond_its_scratch(cuda):
    """256 sequences x 64 heads x 64 partials need far more than the fixed array: the
    call must return ATTN_ERR_WORKSPACE before launching anything."""
    lib = load_library()
    B, H, Hkv, d, maxp = 256, 64, 8, 128, 64
    q = torch.zeros(B, H, d, dtype=torch.bfloat16, device=cuda)
    kp = torch.zeros(1, Hkv, 16, d, dtype=torch.bfloat16, device=cuda)
    vp = torch.zeros_like(kp)
    pt = torch.zeros(B, maxp, dtype=torch.int32, device=cuda)
    kl = torch.full((B,), 16, dtype=torch.int32, device=cuda)
    o = torch.zeros(B, H, d, dtype=torch.bfloat16, device=cuda)
    lse = torch.zeros(B, H, dtype=torch.float32, device=cuda)
    assert lib.attn_decode_workspace_size(B, H, d, maxp) > 40 * 1024 * 1024
    assert _call_noalloc(lib, q, kp, vp, pt, kl, o, lse, maxp) == ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
