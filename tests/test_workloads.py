"""Host logic: the seeded workload recipe and the work/bytes formulas the
benchmark reports, checked against the numbers the pages print."""
import json
import os

import torch

from exact_tiled_attention_11_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_flop_and_byte_formulas_match_p1_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "p1_worked_example.json")))
    cfg = W.PrefillConfig("one_head", 1, 1, 1, g["N"], g["d"], "bf16", (False,))
    flops = cfg.flops(causal=False)
    assert f"{flops:.1e}" == f"{g['printed_flops']:.1e}"
    qkvo = cfg.compulsory_bytes() - cfg.N * 4          # the LSE is not in the page's count
    assert qkvo == g["printed_flash_compulsory_MiB_per_head"] * 2 ** 20
    assert cfg.N * cfg.N * g["bytes_per_element"] == g["printed_score_matrix_MiB"] * 2 ** 20
    assert cfg.flops(causal=True) == flops / 2


def test_config_work_figures():
    assert W.C2.flops(False) == 4 * 2048 ** 2 * 64 * 4 * 12
    assert abs(W.C3.flops(True) - 5.50e11) / 5.50e11 < 0.01
    assert abs(W.C5.flops(True) - 2.20e12) / 2.20e12 < 0.01


def test_decode_recipe_seed0():
    g = torch.Generator().manual_seed(0)
    lens = torch.randint(W.C4.len_lo, W.C4.len_hi + 1, (W.C4.B,), generator=g)
    pages = (lens + 15) // 16
    assert (int(lens.min()), int(lens.max())) == (1420, 32523)
    assert int(pages.sum()) == 62753 and int(pages.max()) == 2033
    assert int(lens.sum()) * 8 * 128 * 2 * 2 == 4110630912


def test_decode_inputs_small_structure():
    kv = W.decode_inputs(5, 8, 2, 128, 16, 1, 100, seed=3, kv_lens=[1, 16, 17, 0, 100])
    assert kv.q.shape == (5, 8, 128) and kv.q.dtype == torch.bfloat16
    pages = [1, 1, 2, 0, 7]
    P = sum(pages)
    assert kv.k_pages.shape == (P, 2, 16, 128)
    used = []
    for b, n in enumerate(pages):
        used += kv.page_table[b, :n].tolist()
        assert (kv.page_table[b, n:] == 0).all()
    assert sorted(used) == list(range(P))            # each page belongs to exactly one sequence
    assert kv.kv_lens.tolist() == [1, 16, 17, 0, 100]
    again = W.decode_inputs(5, 8, 2, 128, 16, 1, 100, seed=3, kv_lens=[1, 16, 17, 0, 100])
    assert torch.equal(kv.k_pages, again.k_pages) and torch.equal(kv.page_table, again.page_table)


def test_prefill_inputs_recipe():
    q, k, v = W.prefill_inputs(1, 2, 1, 8, 64, "bf16", q_mult=30.0, seed=0)
    g = torch.Generator().manual_seed(0)
    q0 = torch.randn(1, 2, 8, 64, generator=g)
    assert torch.equal(q, (q0 * 30.0).to(torch.bfloat16))
    assert k.shape == (1, 1, 8, 64) and v.dtype == torch.bfloat16
