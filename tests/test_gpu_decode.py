"""Paged split-KV decode parity: attn_decode_paged (through the C ABI) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_decode_paged, attn_device_error
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o, f64

pytestmark = pytest.mark.gpu


def to_dev(kv, dev):
    return [t.to(dev) for t in (kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens)]


def run(kv, dev, num_splits=0, scale=None):
    q, kp, vp, pt, kl = to_dev(kv, dev)
    d = q.shape[-1]
    o, lse = attn_decode_paged(q, kp, vp, pt, kl, scale=scale or 1 / math.sqrt(d), num_splits=num_splits)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def ref(kv, scale=None, seqs=None):
    d = kv.q.shape[-1]
    return oracle.decode_paged(kv.q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens,
                               scale=scale or 1 / math.sqrt(d), seqs=seqs)


EDGE_LENS = [1, 15, 16, 17, 33, 300, 1000, 2049]


@pytest.mark.parametrize("num_splits", [0, 1, 2, 3, 7, 16, 33, 96, 200])
def test_splits_sweep(cuda, num_splits):
    kv = W.decode_inputs(len(EDGE_LENS), 32, 8, 128, 16, 1, 1, seed=1, kv_lens=EDGE_LENS)
    o, lse = run(kv, cuda, num_splits)
    O, L = ref(kv)
    check_o(o, O, torch.bfloat16, f"splits={num_splits}")
    check_lse(lse, L, f"splits={num_splits}")


@pytest.mark.parametrize("H,Hkv", [(16, 16), (32, 8), (32, 4), (64, 8), (32, 2)])
def test_group_sizes(cuda, H, Hkv):
    kv = W.decode_inputs(4, H, Hkv, 128, 16, 1, 1, seed=H + Hkv, kv_lens=[5, 160, 999, 4096])
    for s in (0, 5):
        o, lse = run(kv, cuda, s)
        O, L = ref(kv)
        check_o(o, O, torch.bfloat16, f"g={H // Hkv} splits={s}")
        check_lse(lse, L, f"g={H // Hkv} splits={s}")


def test_empty_sequence(cuda):
    kv = W.decode_inputs(3, 32, 8, 128, 16, 1, 1, seed=2, kv_lens=[0, 40, 0])
    o, lse = run(kv, cuda, 4)
    assert (o[0] == 0).all() and (o[2] == 0).all()
    assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all()
    O, L = ref(kv)
    check_o(o, O, torch.bfloat16, "empty")
    check_lse(lse, L, "empty")


def test_single_token_closed_form(cuda):
    """L = 1: O = v_0 (one bf16 value, exactly representable) and LSE = scale * q . k_0."""
    kv = W.decode_inputs(2, 32, 8, 128, 16, 1, 1, seed=3, kv_lens=[1, 1])
    o, lse = run(kv, cuda, 1)
    for b in range(2):
        page = int(kv.page_table[b, 0])
        for h in range(32):
            v0 = kv.v_pages[page, h // 4, 0]
            assert torch.equal(o[b, h], v0)
            s0 = float((f64(kv.q[b, h]) * f64(kv.k_pages[page, h // 4, 0])).sum()) / math.sqrt(128)
            assert abs(float(lse[b, h]) - s0) < 1e-3


def test_large_scores(cuda):
    kv = W.decode_inputs(4, 32, 8, 128, 16, 1, 1, seed=4, kv_lens=[7, 100, 1000, 3000])
    kv.q = (kv.q.float() * 40).to(torch.bfloat16)
    o, lse = run(kv, cuda, 6)
    O, L = ref(kv)
    check_o(o, O, torch.bfloat16, "x40")
    check_lse(lse, L, "x40")


def test_deterministic_per_split_count(cuda):
    kv = W.decode_inputs(5, 32, 8, 128, 16, 1, 1, seed=5, kv_lens=[77, 1234, 16, 4000, 900])
    for s in (0, 3, 17):
        a = run(kv, cuda, s)
        b = run(kv, cuda, s)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_c4_full_size_sampled(cuda):
    """The full workload (64 sequences, lengths 512..32768, random page placement)
    in the benchmark's launch configuration (automatic split count); sampled
    sequences against the oracle, every sequence checked for finiteness."""
    kv = W.decode_inputs_for(W.C4)
    o, lse = run(kv, cuda, 0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    lens = kv.kv_lens.numpy()
    seqs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 0, 31, 63, 17})
    O, L = ref(kv, seqs=seqs)
    check_o(o[seqs], O[seqs], torch.bfloat16, "C4")
    check_lse(lse[seqs], L[seqs], "C4")
    assert attn_device_error(clear=False) == 0


@pytest.mark.parametrize("num_splits", [0, 1, 4, 33])
@pytest.mark.parametrize("H,Hkv", [(8, 8), (32, 8), (64, 4)])
def test_head_dim_64(cuda, H, Hkv, num_splits):
    """d = 64: one 64-column block per page, a 16-stage ring (the same bytes in flight)."""
    kv = W.decode_inputs(6, H, Hkv, 64, 16, 1, 1, seed=H * 3 + Hkv, kv_lens=[1, 16, 17, 300, 2049, 0])
    o, lse = run(kv, cuda, num_splits)
    O, L = ref(kv)
    check_o(o, O, torch.bfloat16, f"d=64 g={H // Hkv} splits={num_splits}")
    check_lse(lse, L, f"d=64 g={H // Hkv} splits={num_splits}")
    assert attn_device_error() == 0


def poison_tail_slots(kv):
    """Fill every slot past kv_lens[b] in each sequence's last page of K and V with NaN,
    +Inf and -Inf (in turn), as a recycled or never-written page pool may hold."""
    ps = kv.page_size
    bad = torch.tensor([float("nan"), float("inf"), -float("inf")], dtype=torch.bfloat16)
    n = 0
    for b, L in enumerate(kv.kv_lens.tolist()):
        if L % ps == 0:
            continue
        page = int(kv.page_table[b, L // ps])
        for slot in range(L % ps, ps):
            kv.k_pages[page, :, slot, :] = bad[n % 3]
            kv.v_pages[page, :, slot, :] = bad[(n + 1) % 3]
            n += 1
    assert n > 0
    return kv


@pytest.mark.parametrize("num_splits", [0, 1, 3])
@pytest.mark.parametrize("d", [64, 128])
def test_non_finite_tail_slots_do_not_reach_the_output(cuda, d, num_splits):
    """The slots of a last page past the sequence's length may hold anything: with NaN and
    +-Inf there, O and the LSE still match the oracle (which reads only the first kv_lens[b]
    tokens)."""
    kv = poison_tail_slots(W.decode_inputs(8, 32, 8, d, 16, 1, 1, seed=41 + d,
                                           kv_lens=[1, 15, 17, 33, 300, 1000, 2049, 5]))
    attn_device_error(clear=True)
    o, lse = run(kv, cuda, num_splits=num_splits)
    O, L = ref(kv)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    check_o(o, O, torch.bfloat16, f"poisoned tails d={d} splits={num_splits}")
    check_lse(lse, L, f"poisoned tails d={d} splits={num_splits}")
    assert attn_device_error() == 0
