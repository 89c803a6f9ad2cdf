"""Float64 oracle functions (test infrastructure only; see the package header).

Sources, by page title and section:

* "3.4 Attention Kernels" (llm-learning-path, part 3) -- "Naive attention and
  its memory traffic" (S = Q K^T / sqrt(d), softmax, P V), "Online softmax"
  (stable softmax with m and l; running (m, l, o~); the merge of two partial
  results), "FlashAttention: tiling" (B_r x B_c tiles, O = o~ / l, the
  log-sum-exp m + log l, causal tile skipping), "Decode attention and
  Flash-Decoding" (split the keys, per-chunk (m_c, l_c, o~_c), merge),
  "Paged and ragged layouts: FlashInfer" (block table of page indices per
  sequence), "Code" (the causal mask aligned to the last key).
* "FlashAttention and Optimized Kernels" (programmer.ie, chapter 13) -- "The
  online softmax" (per-tile update, skip tiles wholly in the future), "It is
  exact" (visited block-pair fractions), "The decode shape: splitting the keys"
  (the partial triple and merge_partials).
* "3.4 Attention Kernels", "Paged and ragged layouts: FlashInfer" and
  "Check your understanding" -- cascade attention: requests sharing a prefix
  attend to the prefix followed by their own suffix; ragged tensors (tokens
  concatenated, an indptr of sequence starts) and paged K/V for prefill.
* "Multi-Head Attention to Flash Attention" (empirq) -- "Online Softmax
  Calculation" (the per-block update formulas; step 2 read as
  max(m_{j-1}, rowmax S_j), as its worked example does).

Conventions that the pages leave open (each is a reading):

* scale is the caller's value (1/sqrt(d) in every workload); the pages' scalar
  worked examples use 1.
* the log-sum-exp is the natural log of the scaled scores.
* grouped-query attention: query head h reads KV head h // (H / Hkv).
* a row with no attended key has O = 0 and LSE = -inf; an empty partial is
  (m, l, o~) = (-inf, 0, 0), and exp(-inf - m) is taken as 0.
* the causal mask keeps key j for query i when j <= i + (Nk - N), i.e. aligned
  to the last key; for self-attention (Nk == N) this is j <= i.
"""
from __future__ import annotations

import numpy as np


def to_f64(x) -> np.ndarray:
    """Upcast a stored tensor (numpy array or torch CPU tensor, any float dtype) to float64."""
    if hasattr(x, "detach"):  # torch tensor; bf16 has no numpy dtype, so go through fp32
        import torch
        x = x.detach().to("cpu")
        if x.dtype in (torch.bfloat16, torch.float16):
            x = x.to(torch.float32)
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _causal_keep(rows: np.ndarray, Nk: int, N: int) -> np.ndarray:
    """Boolean [len(rows), Nk]: key j is attended by query row i when j <= i + (Nk - N)."""
    cols = np.arange(Nk)
    return cols[None, :] <= (rows[:, None] + (Nk - N))


def _softmax_weights(S: np.ndarray):
    """Stable softmax of each row of S (entries may be -inf).

    m = rowmax S, E = exp(S - m), l = sum E, P = E / l, LSE = m + ln l.
    Rows whose every entry is -inf attend to nothing: P = 0, LSE = -inf.
    Returns (P [rows, Nk], LSE [rows]).
    """
    n_rows = S.shape[0]
    P = np.zeros(S.shape)
    lse = np.full(n_rows, -np.inf)
    if S.shape[1] == 0 or n_rows == 0:
        return P, lse
    m = S.max(axis=1)
    live = np.isfinite(m)
    if not live.any():
        return P, lse
    ml = m[live]
    E = np.exp(S[live] - ml[:, None])     # exp(-inf) = 0 for masked keys
    l = E.sum(axis=1)
    P[live] = E / l[:, None]
    lse[live] = ml + np.log(l)
    return P, lse


def _softmax_rows(S: np.ndarray, Vh: np.ndarray):
    """The softmax weights of S applied to V: O = P V, LSE as in _softmax_weights.

    Rows that attend to nothing have P = 0, so O = 0 and LSE = -inf.
    """
    P, lse = _softmax_weights(S)
    return P @ Vh, lse


def _scores(Q, K, b: int, h: int, rows, *, causal: bool, scale: float):
    """S = scale * q K^T for query rows ``rows`` of head (b, h) against KV head
    h // (H / Hkv), keys after the query set to -inf when causal."""
    H, N = Q.shape[1], Q.shape[2]
    Hkv, Nk = K.shape[1], K.shape[2]
    kvh = h // (H // Hkv)
    rows = np.asarray(rows, dtype=np.int64)
    q = to_f64(Q[b, h])[rows]
    Kh = to_f64(K[b, kvh])
    S = scale * (q @ Kh.T)                 # [rows, Nk], materialised
    if causal:
        S = np.where(_causal_keep(rows, Nk, N), S, -np.inf)
    return S


def attention_weights(Q, K, b: int, h: int, rows, *, causal: bool, scale: float):
    """The softmax weights P = softmax(scale q K^T) of query rows ``rows`` of head (b, h).

    Q: [B, H, N, d], K: [B, Hkv, Nk, d].  Row i of P holds the weight of every
    key in row i's output, O_i = sum_j P_ij V_j; masked keys have weight 0 and
    a row with no attended key is all zero.  Returns (P [len(rows), Nk],
    LSE [len(rows)]) in float64.
    """
    return _softmax_weights(_scores(Q, K, b, h, rows, causal=causal, scale=scale))


def attention_rows(Q, K, V, b: int, h: int, rows, *, causal: bool, scale: float):
    """The plain definition restricted to query rows ``rows`` of head (b, h).

    Q: [B, H, N, d], K/V: [B, Hkv, Nk, d] (any float dtype; upcast to float64).
    Returns (O [len(rows), d], LSE [len(rows)]) in float64.
    """
    H, Hkv = Q.shape[1], K.shape[1]
    Vh = to_f64(V[b, h // (H // Hkv)])
    return _softmax_rows(_scores(Q, K, b, h, rows, causal=causal, scale=scale), Vh)


def attention(Q, K, V, *, causal: bool, scale: float, row_chunk: int = 2048):
    """Exact attention by its plain definition, in float64 on the CPU.

    For every (b, h): S = scale * Q K^T with KV head h // (H/Hkv); keys after
    the query masked to -inf when causal; m = rowmax S; P = exp(S - m);
    l = rowsum P; O = P V / l; LSE = m + ln l.
    Returns (O [B, H, N, d], LSE [B, H, N]) as float64 numpy arrays.
    """
    B, H, N, d = Q.shape
    O = np.zeros((B, H, N, d))
    LSE = np.full((B, H, N), -np.inf)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, row_chunk):
                rows = np.arange(r0, min(N, r0 + row_chunk))
                O[b, h, rows], LSE[b, h, rows] = attention_rows(Q, K, V, b, h, rows, causal=causal, scale=scale)
    return O, LSE


# ----------------------------------------------------------------------------
# The block-wise algorithm and its partial results
# ----------------------------------------------------------------------------

def partial_state(s: np.ndarray, v: np.ndarray):
    """(m, l, o~) of one query row over a key subset.

    s: scores [n] (already scaled; may contain -inf), v: values [n, d].
    m = max s, l = sum exp(s - m), o~ = sum exp(s - m) v.  An empty or fully
    masked subset gives (-inf, 0, 0).
    """
    s = np.asarray(s, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    v = v.reshape(len(s), v.shape[-1] if v.ndim > 1 else 1)
    if len(s) == 0 or not np.isfinite(s).any():
        return -np.inf, 0.0, np.zeros(v.shape[1])
    m = s.max()
    p = np.exp(s - m)
    return m, p.sum(), p @ v


def merge_partials(parts):
    """Exact merge of partial results over disjoint key sets.

    m = max_i m_i, l = sum_i exp(m_i - m) l_i, o~ = sum_i exp(m_i - m) o~_i,
    with exp(-inf - m) = 0 for empty partials.  ``parts`` is an iterable of
    (m, l, o~); all empty gives (-inf, 0, 0).
    """
    parts = [(float(m), float(l), np.asarray(o, dtype=np.float64)) for m, l, o in parts]
    d = parts[0][2].shape[0] if parts else 0
    m = max((p[0] for p in parts), default=-np.inf)
    if m == -np.inf:
        return -np.inf, 0.0, np.zeros(d)
    w = [np.exp(mi - m) if mi != -np.inf else 0.0 for mi, _, _ in parts]
    l = sum(wi * li for wi, (_, li, _) in zip(w, parts))
    o = sum(wi * oi for wi, (_, _, oi) in zip(w, parts))
    return m, l, o


def finalize(m, l, o_tilde):
    """o = o~ / l and LSE = m + ln l; (O = 0, LSE = -inf) when nothing was attended."""
    o_tilde = np.asarray(o_tilde, dtype=np.float64)
    if l == 0.0 or m == -np.inf:
        return np.zeros_like(o_tilde), -np.inf
    return o_tilde / l, m + np.log(l)


def tiled_attention(Q, K, V, *, causal: bool, scale: float, block_q: int, block_k: int):
    """The FlashAttention forward pass for one head, in float64.

    Q: [N, d], K/V: [Nk, d].  Q is cut into row blocks of ``block_q``; for each
    one the running state (m = -inf, l = 0, o~ = 0) is updated tile by tile over
    K/V blocks of ``block_k`` keys.  When causal, key tiles wholly after the
    block's last query are never visited and the diagonal tile is masked.
    Per tile: s = scale q K_j^T, m' = max(m, rowmax s), p = exp(s - m'),
    l = exp(m - m') l + rowsum p, o~ = exp(m - m') o~ + p V_j, m = m'.
    Finally O = o~ / l and LSE = m + ln l.

    Returns (O [N, d], LSE [N], visited_pairs, total_pairs).
    """
    Q, K, V = to_f64(Q), to_f64(K), to_f64(V)
    N, d = Q.shape
    Nk = K.shape[0]
    O = np.zeros((N, V.shape[1]))
    LSE = np.full(N, -np.inf)
    visited = 0
    n_kb = -(-Nk // block_k)
    total = (-(-N // block_q)) * n_kb
    for i0 in range(0, N, block_q):
        rows = np.arange(i0, min(N, i0 + block_q))
        q = Q[rows]
        m = np.full(len(rows), -np.inf)
        l = np.zeros(len(rows))
        acc = np.zeros((len(rows), V.shape[1]))
        last_key = rows[-1] + (Nk - N) if causal else Nk - 1
        for j0 in range(0, Nk, block_k):
            if j0 > last_key:            # wholly in the future: skipped
                break
            cols = np.arange(j0, min(Nk, j0 + block_k))
            visited += 1
            s = scale * (q @ K[cols].T)
            if causal:
                s = np.where(cols[None, :] <= rows[:, None] + (Nk - N), s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            # a row that has seen no key yet keeps m' = -inf; use 0 as its
            # reference so that exp(m - m') and p come out 0 rather than nan
            ref = np.where(np.isfinite(m_new), m_new, 0.0)
            corr = np.exp(m - ref)
            p = np.exp(s - ref[:, None])
            l = corr * l + p.sum(axis=1)
            acc = corr[:, None] * acc + p @ V[cols]
            m = m_new
        ok = l > 0
        O[rows[ok]] = acc[ok] / l[ok, None]
        LSE[rows[ok]] = m[ok] + np.log(l[ok])
    return O, LSE, visited, total


# ----------------------------------------------------------------------------
# Paged decode
# ----------------------------------------------------------------------------

def gather_sequence(k_pages, v_pages, page_table, kv_lens, b: int):
    """K and V of sequence b, token by token, through its page table.

    Token t of sequence b sits in page page_table[b, t // page_size] at slot
    t % page_size.  Returns (K_b, V_b), each [Hkv, kv_lens[b], d] float64.
    """
    ps = k_pages.shape[2]
    L = int(kv_lens[b])
    npg = -(-L // ps)
    pages = np.asarray([int(page_table[b, p]) for p in range(npg)], dtype=np.int64)
    Kb = to_f64(k_pages[pages]) if len(pages) else np.zeros((0,) + tuple(k_pages.shape[1:]))
    Vb = to_f64(v_pages[pages]) if len(pages) else np.zeros((0,) + tuple(v_pages.shape[1:]))
    # [npg, Hkv, ps, d] -> [Hkv, npg * ps, d] -> first L tokens
    Hkv, d = Kb.shape[1], Kb.shape[3]
    Kb = Kb.transpose(1, 0, 2, 3).reshape(Hkv, npg * ps, d)[:, :L]
    Vb = Vb.transpose(1, 0, 2, 3).reshape(Hkv, npg * ps, d)[:, :L]
    return Kb, Vb


def decode_paged(q, k_pages, v_pages, page_table, kv_lens, *, scale: float, seqs=None):
    """One query token per sequence against its whole paged KV cache (no mask).

    q: [B, H, d]; k_pages/v_pages: [P, Hkv, page_size, d]; page_table: [B, max_pages];
    kv_lens: [B].  For each sequence the keys are gathered in page-table order
    and attention is taken by the plain definition.  Returns (O [B, H, d],
    LSE [B, H]) float64; rows of sequences not in ``seqs`` stay (0, -inf).
    """
    B, H, d = q.shape
    Hkv = k_pages.shape[1]
    g = H // Hkv
    O = np.zeros((B, H, d))
    LSE = np.full((B, H), -np.inf)
    qf = to_f64(q)
    for b in (range(B) if seqs is None else seqs):
        Kb, Vb = gather_sequence(k_pages, v_pages, page_table, kv_lens, b)
        for h in range(H):
            S = scale * (qf[b, h][None, :] @ Kb[h // g].T)    # [1, L]
            o, lse = _softmax_rows(S, Vb[h // g])
            O[b, h], LSE[b, h] = o[0], lse[0]
    return O, LSE


def cascade_decode(q, prefix_k, prefix_v, k_pages, v_pages, page_table, kv_lens, *, scale: float, seqs=None):
    """Decode for requests that share a prefix, by the plain definition.

    Request b's query attends to the shared prefix's keys (prefix_k/prefix_v
    [Hkv, prefix_len, d]) followed by its own suffix gathered through its page
    table (kv_lens[b] tokens), with no mask.  Returns (O [B, H, d], LSE [B, H])
    float64; rows of requests not in ``seqs`` stay (0, -inf).
    """
    B, H, d = q.shape
    Hkv = k_pages.shape[1]
    g = H // Hkv
    Pk, Pv = to_f64(prefix_k), to_f64(prefix_v)
    O = np.zeros((B, H, d))
    LSE = np.full((B, H), -np.inf)
    qf = to_f64(q)
    for b in (range(B) if seqs is None else seqs):
        Kb, Vb = gather_sequence(k_pages, v_pages, page_table, kv_lens, b)
        for h in range(H):
            keys = np.concatenate([Pk[h // g], Kb[h // g]], axis=0)
            vals = np.concatenate([Pv[h // g], Vb[h // g]], axis=0)
            S = scale * (qf[b, h][None, :] @ keys.T)
            o, lse = _softmax_rows(S, vals)
            O[b, h], LSE[b, h] = o[0], lse[0]
    return O, LSE


def varlen_attention(q, k, v, qo_indptr, kv_indptr, *, causal: bool, scale: float):
    """Ragged batch by the plain definition, one sequence at a time.

    q [total_q, H, d], k/v [total_k, Hkv, d]; sequence b owns query rows
    [qo_indptr[b], qo_indptr[b+1]) and key rows [kv_indptr[b], kv_indptr[b+1]).
    The causal mask is aligned to each sequence's last key.  Returns
    (O [total_q, H, d], LSE [total_q, H]) float64.
    """
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    total_q, H, d = qf.shape
    Hkv = kf.shape[1]
    O = np.zeros((total_q, H, d))
    LSE = np.full((total_q, H), -np.inf)
    qo = [int(x) for x in qo_indptr]
    kvp = [int(x) for x in kv_indptr]
    for b in range(len(qo) - 1):
        qs, qe, ks, ke = qo[b], qo[b + 1], kvp[b], kvp[b + 1]
        if qe == qs:
            continue
        Qb = qf[qs:qe].transpose(1, 0, 2)[None]          # [1, H, Lq, d]
        Kb = kf[ks:ke].transpose(1, 0, 2)[None]          # [1, Hkv, Lk, d]
        Vb = vf[ks:ke].transpose(1, 0, 2)[None]
        Ob, Lb = attention(Qb, Kb, Vb, causal=causal, scale=scale)
        O[qs:qe] = Ob[0].transpose(1, 0, 2)
        LSE[qs:qe] = Lb[0].T
    return O, LSE


def paged_prefill(q, k_pages, v_pages, page_table, kv_lens, qo_indptr, *, causal: bool, scale: float):
    """Ragged query chunks against each sequence's paged cache, by the plain definition.

    Sequence b's queries (rows [qo_indptr[b], qo_indptr[b+1]) of q [total_q, H, d])
    are the last tokens of its kv_lens[b] keys, gathered token by token through its
    page table.  Returns (O [total_q, H, d], LSE [total_q, H]) float64.
    """
    qf = to_f64(q)
    total_q, H, d = qf.shape
    O = np.zeros((total_q, H, d))
    LSE = np.full((total_q, H), -np.inf)
    qo = [int(x) for x in qo_indptr]
    for b in range(len(qo) - 1):
        qs, qe = qo[b], qo[b + 1]
        if qe == qs:
            continue
        Kb, Vb = gather_sequence(k_pages, v_pages, page_table, kv_lens, b)   # [Hkv, L, d]
        Ob, Lb = attention(qf[qs:qe].transpose(1, 0, 2)[None], Kb[None], Vb[None], causal=causal, scale=scale)
        O[qs:qe] = Ob[0].transpose(1, 0, 2)
        LSE[qs:qe] = Lb[0].T
    return O, LSE
