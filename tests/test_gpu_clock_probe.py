"""The clock probe: two records on one SM around real work give a plausible SM clock."""
import pytest
import torch

from exact_tiled_attention_11_gb300 import attn_clock_probe, attn_device_error, attn_fwd
from exact_tiled_attention_11_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_clock_probe_brackets_work_on_one_sm(cuda):
    q, k, v = (t.to(cuda) for t in W.prefill_inputs(1, 8, 2, 4096, 128, seed=3))
    probe = torch.zeros(8, dtype=torch.int64, device=cuda)
    attn_clock_probe(probe[:4])
    for _ in range(20):
        attn_fwd(q, k, v, causal=True, scale=128 ** -0.5)
    attn_clock_probe(probe[4:], match=probe[:4])
    torch.cuda.synchronize()
    t0, c0, sm0, ok0, t1, c1, sm1, ok1 = probe.cpu().tolist()
    assert ok0 == 1 and ok1 == 1, "a probe found no block on its SM"
    assert sm0 == sm1
    assert t1 > t0 and c1 > c0
    mhz = 1000.0 * (c1 - c0) / (t1 - t0)
    assert 300.0 < mhz < 3000.0, mhz
    assert attn_device_error() == 0
