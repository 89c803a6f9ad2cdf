"""Seeded synthetic workloads for exact tiled attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path (through the tests and the
benchmark) and the float64 CPU oracle are fed from here, so the two sides
always see the same stored tensors.

Recipe (one ``torch.Generator().manual_seed(seed)`` on the CPU per workload):

* prefill: ``randn`` in fp32, drawn in the order Q, K, V; Q is then multiplied
  by ``q_mult`` in fp32 (the large-score stress runs use 30 and 40) and all
  three are cast to the storage dtype.  Layout ``[B, H, N, d]`` for Q and
  ``[B, Hkv, N, d]`` for K and V, d contiguous.
* paged decode: per-sequence KV lengths ``randint(len_lo, len_hi + 1)``, then a
  random permutation of the shared page pool, then ``randn`` for q
  ``[B, H, d]``, the K pool and the V pool, each pool ``[P, Hkv, page_size,
  d]`` where P is the number of pages all sequences need.  Sequence b owns
  pages ``perm[off_b : off_b + pages_b]`` in order; ``page_table`` is int32
  ``[B, max_pages]`` padded with 0 past ``pages_b``.

The pages this library follows name no dataset or benchmark suite, so every
input is synthetic: iid N(0, 1) values with the shapes of the five workloads
below.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    dtype: str            # "f32" or "bf16"
    causal: tuple         # the causal settings the workload is run with
    q_mults: tuple = (1.0,)

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5

    def flops(self, causal: bool) -> float:
        """4 N^2 d per (batch, head), halved for causal attention."""
        f = 4.0 * self.N * self.N * self.d * self.B * self.H
        return f / 2.0 if causal else f

    def compulsory_bytes(self) -> int:
        """Read Q, K, V once, write O once (storage dtype) and the fp32 LSE."""
        eb = 4 if self.dtype == "f32" else 2
        q = self.B * self.H * self.N * self.d
        kv = self.B * self.Hkv * self.N * self.d
        return (2 * q + 2 * kv) * eb + self.B * self.H * self.N * 4


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    H: int
    Hkv: int
    d: int
    page_size: int
    len_lo: int
    len_hi: int

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5


C1 = PrefillConfig("exact_fp32_b1_h1_n256_d64", 1, 1, 1, 256, 64, "f32", (False,), (1.0, 30.0))
C2 = PrefillConfig("prefill_bf16_b4_h12_n2048_d64", 4, 12, 12, 2048, 64, "bf16", (False, True))
C3 = PrefillConfig("prefill_bf16_b1_h32_hkv8_n8192_d128_causal", 1, 32, 8, 8192, 128, "bf16", (True,))
C4 = DecodeConfig("decode_paged_bf16_b64_h32_hkv8_d128_len512_32768_page16", 64, 32, 8, 128, 16, 512, 32768)
C5 = PrefillConfig("prefill_bf16_b2_h16_n16384_d128_causal", 2, 16, 16, 16384, 128, "bf16", (True,), (1.0, 40.0))

PREFILL_CONFIGS = (C1, C2, C3, C5)

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


def prefill_inputs(B, H, Hkv, N, d, dtype="bf16", q_mult=1.0, seed=0):
    """Return (Q, K, V) CPU tensors in the storage dtype, per the recipe above."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, d, generator=g, dtype=torch.float32)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32)
    if q_mult != 1.0:
        q = q * torch.tensor(q_mult, dtype=torch.float32)
    t = torch_dtype(dtype)
    return q.to(t), k.to(t), v.to(t)


def prefill_inputs_for(cfg: PrefillConfig, q_mult=1.0, seed=0):
    return prefill_inputs(cfg.B, cfg.H, cfg.Hkv, cfg.N, cfg.d, cfg.dtype, q_mult, seed)


@dataclass
class PagedKV:
    q: torch.Tensor            # [B, H, d] bf16
    k_pages: torch.Tensor      # [P, Hkv, page_size, d] bf16
    v_pages: torch.Tensor      # [P, Hkv, page_size, d] bf16
    page_table: torch.Tensor   # [B, max_pages] int32
    kv_lens: torch.Tensor      # [B] int32
    page_size: int
    extra: dict = field(default_factory=dict)

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    def kv_bytes(self) -> int:
        """Bytes of K and V for the tokens actually attended."""
        Hkv, d = self.k_pages.shape[1], self.k_pages.shape[3]
        return int(self.kv_lens.to(torch.int64).sum()) * Hkv * d * 2 * self.k_pages.element_size()


def _randn_bf16(shape, g, chunk_rows=4096):
    """randn drawn in fp32 then cast, in chunks along dim 0 to bound host memory."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        out[s:e] = torch.randn((e - s,) + tuple(shape[1:]), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def decode_inputs(B, H, Hkv, d, page_size, len_lo, len_hi, seed=0, kv_lens=None):
    """Paged KV cache per the recipe above.  ``kv_lens`` overrides the drawn lengths
    (used for edge cases such as one-token or page-aligned sequences)."""
    g = torch.Generator().manual_seed(seed)
    drawn = torch.randint(len_lo, len_hi + 1, (B,), generator=g, dtype=torch.int64)
    lens = drawn if kv_lens is None else torch.as_tensor(kv_lens, dtype=torch.int64).reshape(-1)
    B = int(lens.shape[0])
    pages = (lens + page_size - 1) // page_size
    P = int(pages.sum())
    perm = torch.randperm(max(P, 1), generator=g)[:P]
    max_pages = max(int(pages.max()) if B > 0 else 0, 1)
    table = torch.zeros(B, max_pages, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(pages[b])
        table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = torch.randn(B, H, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    pool = (max(P, 1), Hkv, page_size, d)
    k_pages = _randn_bf16(pool, g)
    v_pages = _randn_bf16(pool, g)
    return PagedKV(q, k_pages, v_pages, table, lens.to(torch.int32), page_size)


def decode_inputs_for(cfg: DecodeConfig, seed=0, kv_lens=None, B=None):
    return decode_inputs(cfg.B if B is None else B, cfg.H, cfg.Hkv, cfg.d, cfg.page_size,
                         cfg.len_lo, cfg.len_hi, seed, kv_lens)


def fp8_signs(d: int, seed: int = 0) -> torch.Tensor:
    """The random +-1 diagonal of the FP8 path's orthogonal transform (fp32, seeded)."""
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.float32)
