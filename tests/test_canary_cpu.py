"""The guard-region helper of the GPU canary tests detects stray writes (checked on the CPU)."""
import torch

from tests.test_gpu_canary import GUARD, Guarded


def test_guard_detects_writes_on_either_side():
    for side in ("before", "after"):
        g = Guarded((3, 5), torch.float32, "cpu")
        g.t.fill_(1.0)  # writing the tensor itself leaves the guards intact
        assert g.intact()
        if side == "before":
            g.buf[GUARD - 1] = 0
        else:
            g.buf[-GUARD] = 0
        assert not g.intact(), side


def test_views_are_aligned_and_sized():
    g = Guarded((7, 33), torch.bfloat16, "cpu")
    assert g.t.shape == (7, 33) and g.t.dtype == torch.bfloat16
    assert g.t.storage_offset() * g.t.element_size() == GUARD
    assert g.buf.numel() == 2 * GUARD + 7 * 33 * 2
