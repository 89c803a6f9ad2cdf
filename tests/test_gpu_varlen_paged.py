"""Parity of the ragged (indptr) and paged prefill entry points against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_11_gb300 import attn_device_error, attn_fwd_paged, attn_fwd_varlen
from exact_tiled_attention_11_gb300 import workloads as W
from tests.parity import check_lse, check_o

pytestmark = pytest.mark.gpu


def _ragged(lens_q, lens_k, H, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    tq, tk = sum(lens_q), sum(lens_k)
    q = torch.randn(tq, H, d, generator=g).to(torch.bfloat16)
    k = torch.randn(tk, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(tk, Hkv, d, generator=g).to(torch.bfloat16)
    qo = torch.tensor([0] + list(np.cumsum(lens_q)), dtype=torch.int32)
    kvp = torch.tensor([0] + list(np.cumsum(lens_k)), dtype=torch.int32)
    return q, k, v, qo, kvp


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_varlen_self_attention(cuda, causal, d):
    lens = [1, 7, 128, 129, 300, 1000, 0, 513]
    q, k, v, qo, kvp = _ragged(lens, lens, 8, 2, d, seed=d + causal)
    o, lse = attn_fwd_varlen(q.to(cuda), k.to(cuda), v.to(cuda), qo.to(cuda), kvp.to(cuda), max(lens), causal=causal)
    torch.cuda.synchronize()
    O, L = oracle.varlen_attention(q, k, v, qo, kvp, causal=causal, scale=1 / math.sqrt(d))
    check_o(o.cpu(), O, torch.bfloat16, f"varlen d={d} causal={causal}")
    check_lse(lse.cpu(), L, f"varlen d={d} causal={causal}")
    assert attn_device_error() == 0


def test_varlen_chunks_against_longer_keys(cuda):
    """Each sequence's queries are the last Lq of its Lk tokens (chunked prefill)."""
    lq = [1, 50, 128, 300, 17]
    lk = [10, 50, 700, 1200, 17]
    q, k, v, qo, kvp = _ragged(lq, lk, 32, 8, 128, seed=3)
    o, lse = attn_fwd_varlen(q.to(cuda), k.to(cuda), v.to(cuda), qo.to(cuda), kvp.to(cuda), max(lq), causal=True)
    torch.cuda.synchronize()
    O, L = oracle.varlen_attention(q, k, v, qo, kvp, causal=True, scale=1 / math.sqrt(128))
    check_o(o.cpu(), O, torch.bfloat16, "varlen chunks")
    check_lse(lse.cpu(), L, "varlen chunks")


@pytest.mark.parametrize("d", [64, 128])
def test_paged_prefill(cuda, d):
    kv_lens = [17, 300, 1000, 2049, 5]
    q_lens = [17, 1, 128, 300, 5]       # each chunk is the last q_len tokens of its sequence
    kv = W.decode_inputs(len(kv_lens), 8, 2, d, 16, 1, 1, seed=d, kv_lens=kv_lens)
    g = torch.Generator().manual_seed(d + 1)
    q = torch.randn(sum(q_lens), 8, d, generator=g).to(torch.bfloat16)
    qo = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    o, lse = attn_fwd_paged(q.to(cuda), kv.k_pages.to(cuda), kv.v_pages.to(cuda), kv.page_table.to(cuda),
                            kv.kv_lens.to(cuda), qo.to(cuda), max(q_lens), causal=True)
    torch.cuda.synchronize()
    O, L = oracle.paged_prefill(q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens, qo, causal=True,
                                scale=1 / math.sqrt(d))
    check_o(o.cpu(), O, torch.bfloat16, f"paged prefill d={d}")
    check_lse(lse.cpu(), L, f"paged prefill d={d}")
    assert attn_device_error() == 0


def test_paged_prefill_full_sequences_match_varlen(cuda):
    """Whole sequences read from pages equal the same sequences read as ragged tensors."""
    lens = [200, 1, 999]
    kv = W.decode_inputs(len(lens), 16, 4, 128, 16, 1, 1, seed=5, kv_lens=lens)
    g = torch.Generator().manual_seed(6)
    q = torch.randn(sum(lens), 16, 128, generator=g).to(torch.bfloat16)
    qo = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    o_p, lse_p = attn_fwd_paged(q.to(cuda), kv.k_pages.to(cuda), kv.v_pages.to(cuda), kv.page_table.to(cuda),
                                kv.kv_lens.to(cuda), qo.to(cuda), max(lens), causal=True)
    ks, vs = [], []
    for b in range(len(lens)):
        n = -(-lens[b] // 16)
        pg = kv.page_table[b, :n].long()
        ks.append(kv.k_pages[pg].permute(0, 2, 1, 3).reshape(n * 16, 4, 128)[:lens[b]])
        vs.append(kv.v_pages[pg].permute(0, 2, 1, 3).reshape(n * 16, 4, 128)[:lens[b]])
    k = torch.cat(ks).contiguous()
    v = torch.cat(vs).contiguous()
    o_r, lse_r = attn_fwd_varlen(q.to(cuda), k.to(cuda), v.to(cuda), qo.to(cuda), qo.to(cuda), max(lens), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_p.cpu(), o_r.cpu()) and torch.equal(lse_p.cpu(), lse_r.cpu())


def test_varlen_bad_offsets_skip_the_sequence_and_set_the_error_bit(cuda):
    """A sequence longer than max_q_len, or whose offsets leave the tensors, is not
    computed; the others are, and ATTN_DEVERR_BAD_LENGTH (0x8) is recorded."""
    lens = [100, 300, 50]
    q, k, v, qo, kvp = _ragged(lens, lens, 4, 4, 128, seed=8)
    attn_device_error(clear=True)
    sentinel = torch.full_like(q, 7.0).to(cuda)
    o, lse = attn_fwd_varlen(q.to(cuda), k.to(cuda), v.to(cuda), qo.to(cuda), kvp.to(cuda), 128, o=sentinel,
                             causal=True)
    assert attn_device_error(clear=True) & 0x8
    O, L = oracle.varlen_attention(q, k, v, qo, kvp, causal=True, scale=1 / math.sqrt(128))
    rows0, rows1, rows2 = slice(0, 100), slice(100, 400), slice(400, 450)
    check_o(o[rows0].cpu(), O[rows0], torch.bfloat16, "seq 0")
    check_o(o[rows2].cpu(), O[rows2], torch.bfloat16, "seq 2")
    assert (o[rows1] == 7.0).all()                    # skipped: left unwritten
    bad_kv = kvp.clone()
    bad_kv[1] = 10 ** 6                               # keys of sequences 0 and 1 leave k
    attn_fwd_varlen(q.to(cuda), k.to(cuda), v.to(cuda), qo.to(cuda), bad_kv.to(cuda), 300, causal=True)
    assert attn_device_error(clear=True) & 0x8


@pytest.mark.parametrize("d", [64, 128])
def test_paged_prefill_non_finite_tail_slots(cuda, d):
    """NaN and +-Inf in the slots past each sequence's length (its last page's tail) do
    not reach O or the LSE of the paged prefill."""
    from tests.test_gpu_decode import poison_tail_slots
    kv_lens = [17, 300, 1001, 2049, 5, 129]
    q_lens = [17, 1, 128, 300, 5, 129]
    kv = poison_tail_slots(W.decode_inputs(len(kv_lens), 8, 2, d, 16, 1, 1, seed=d + 7, kv_lens=kv_lens))
    g = torch.Generator().manual_seed(d + 8)
    q = torch.randn(sum(q_lens), 8, d, generator=g).to(torch.bfloat16)
    qo = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    attn_device_error(clear=True)
    for causal in (True, False):
        o, lse = attn_fwd_paged(q.to(cuda), kv.k_pages.to(cuda), kv.v_pages.to(cuda), kv.page_table.to(cuda),
                                kv.kv_lens.to(cuda), qo.to(cuda), max(q_lens), causal=causal)
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        O, L = oracle.paged_prefill(q, kv.k_pages, kv.v_pages, kv.page_table, kv.kv_lens, qo, causal=causal,
                                    scale=1 / math.sqrt(d))
        check_o(o.cpu(), O, torch.bfloat16, f"paged prefill poisoned tails d={d} causal={causal}")
        check_lse(lse.cpu(), L, f"paged prefill poisoned tails d={d} causal={causal}")
    assert attn_device_error() == 0
