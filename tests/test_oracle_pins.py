"""Pins for the float64 oracle, against what the pages and the mathematics fix.

Every check here runs on the CPU.  None of them re-types the oracle's own
formula: they use the numbers the pages print for their worked examples, a
scalar pure-Python brute force written with nested loops and ``math.exp``,
closed forms, and invariants of exact attention.
"""
import json
import math
import os
import random

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Scalar brute force (independent of NumPy): nested loops over plain lists.
# ---------------------------------------------------------------------------

def brute_attention(Q, K, V, causal, scale):
    """Q: nested lists [B][H][N][d]; K, V: [B][Hkv][Nk][d].  Returns (O, LSE) as lists."""
    B, H = len(Q), len(Q[0])
    Hkv = len(K[0])
    group = H // Hkv
    O, LSE = [], []
    for b in range(B):
        Ob, Lb = [], []
        for h in range(H):
            kv = h // group
            N, Nk = len(Q[b][h]), len(K[b][kv])
            Oh, Lh = [], []
            for i in range(N):
                keys = [j for j in range(Nk) if (not causal) or j <= i + (Nk - N)]
                if not keys:
                    Oh.append([0.0] * len(V[b][kv][0]) if Nk else [])
                    Lh.append(-math.inf)
                    continue
                s = {}
                for j in keys:
                    acc = 0.0
                    for t in range(len(Q[b][h][i])):
                        acc += Q[b][h][i][t] * K[b][kv][j][t]
                    s[j] = acc * scale
                top = max(s.values())
                z = 0.0
                for j in keys:
                    z += math.exp(s[j] - top)
                row = []
                for t in range(len(V[b][kv][0])):
                    acc = 0.0
                    for j in keys:
                        acc += math.exp(s[j] - top) / z * V[b][kv][j][t]
                    row.append(acc)
                Oh.append(row)
                Lh.append(top + math.log(z))
            Ob.append(Oh)
            Lb.append(Lh)
        O.append(Ob)
        LSE.append(Lb)
    return O, LSE


def brute_weights(q_rows, keys, causal, scale, shift):
    """Softmax weights of each query row over the keys, by scalar loops.

    q_rows: [n][d] lists, keys: [Nk][d]; row i attends key j when not causal or
    j <= i + shift.  Returns [n][Nk] lists (all zeros for a row with no key)."""
    W = []
    for i, q in enumerate(q_rows):
        keep = [j for j in range(len(keys)) if (not causal) or j <= i + shift]
        row = [0.0] * len(keys)
        if keep:
            s = {j: scale * sum(a * b for a, b in zip(q, keys[j])) for j in keep}
            top = max(s.values())
            z = sum(math.exp(s[j] - top) for j in keep)
            for j in keep:
                row[j] = math.exp(s[j] - top) / z
        W.append(row)
    return W


def _rand(shape, rng):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_p4_worked_example_final_output():
    g = _golden("p4_worked_example.json")
    Q = np.array(g["q"]).reshape(1, 1, 1, 2)
    K = np.array(g["K"]).reshape(1, 1, 4, 2)
    V = np.array(g["V"]).reshape(1, 1, 4, 1)
    O, LSE = oracle.attention(Q, K, V, causal=False, scale=1.0)
    half_ulp = 0.5 * 10 ** -g["printed_decimals"]
    assert abs(O[0, 0, 0, 0] - g["printed"]["final_output"]) <= half_ulp
    # the page's final state is m = 3 with l = 1.638 (rounded); LSE = m + ln l
    assert abs(LSE[0, 0, 0] - (3.0 + math.log(g["printed"]["block2"]["l"]))) < 2e-3


def test_p4_worked_example_block_states():
    g = _golden("p4_worked_example.json")
    q = np.array(g["q"])
    K = np.array(g["K"])
    V = np.array(g["V"]).reshape(4, 1)
    bk = g["block_k"]
    s = K @ q  # scale 1 on the page
    pr = g["printed"]
    np.testing.assert_allclose(s[:bk], pr["block1_scores"])
    np.testing.assert_allclose(s[bk:], pr["block2_scores"])
    m1, l1, o1 = oracle.partial_state(s[:bk], V[:bk])
    tol = 0.5 * 10 ** -g["printed_decimals"]
    assert abs(m1 - pr["block1"]["m"]) <= tol
    assert abs(l1 - pr["block1"]["l"]) <= tol
    # the page multiplies 3-decimal weights (0.368, 0.135) by the values, so
    # its o~ carries up to max|v| half-units of the third decimal
    carried = float(np.abs(V).max()) * tol
    assert abs(o1[0] - pr["block1"]["o_tilde"]) <= carried
    m2, l2, o2 = oracle.merge_partials([(m1, l1, o1), oracle.partial_state(s[bk:], V[bk:])])
    # block 2 rescales the rounded block-1 sums by a rounded 0.368 and adds
    # rounded weights again: a few half-units of the last digit for l,
    # values times that for o~
    assert abs(m2 - pr["block2"]["m"]) <= tol
    assert abs(l2 - pr["block2"]["l"]) <= 4 * tol
    assert abs(o2[0] - pr["block2"]["o_tilde"]) <= 2 * carried
    assert abs(math.exp(m1 - m2) - pr["block2_correction"]) <= tol
    # the tiled pass with the page's blocks of two reaches the same output
    O, LSE, visited, total = oracle.tiled_attention(q[None], K, V, causal=False, scale=1.0, block_q=1, block_k=bk)
    assert visited == total == 2
    assert abs(O[0, 0] - pr["final_output"]) <= tol


@pytest.mark.parametrize("tile", [4, 2, 1, 3, 10])
def test_p2_online_softmax_lab(tile):
    g = _golden("p2_online_softmax_lab.json")
    s = np.array(g["scores"], dtype=np.float64)
    v = np.array(g["values"], dtype=np.float64)
    n = len(s)
    # one query, d = 1: q = 1 and k_j = s_j make the scaled scores the lab's scores
    Q = np.ones((1, 1, 1, 1))
    K = s.reshape(1, 1, n, 1)
    V = v.reshape(1, 1, n, 1)
    O, _ = oracle.attention(Q, K, V, causal=False, scale=1.0)
    assert abs(O[0, 0, 0, 0] - g["printed_batch"]) < 0.5e-10
    Ot, _, _, _ = oracle.tiled_attention(np.ones((1, 1)), s.reshape(n, 1), v.reshape(n, 1),
                                         causal=False, scale=1.0, block_q=1, block_k=tile)
    assert abs(Ot[0, 0] - g["printed_online"]) < 0.5e-10
    assert abs(Ot[0, 0] - O[0, 0, 0, 0]) < g["match_below"]


def test_p3_causal_block_pairs():
    g = _golden("p3_causal_block_pairs.json")
    rng = np.random.default_rng(1)
    for case in g["cases"]:
        N, bs = case["N"], case["block"]
        Q, K, V = (rng.standard_normal((N, 2)) for _ in range(3))
        _, _, visited, total = oracle.tiled_attention(Q, K, V, causal=True, scale=1.0, block_q=bs, block_k=bs)
        if "printed_percent" in case:
            assert round(100.0 * visited / total) == case["printed_percent"]
        if "printed_pairs" in case:
            assert visited == case["printed_pairs"]


# ---------------------------------------------------------------------------
# Brute force on tiny inputs (scalar loops, math.exp)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,Nk,d,H,Hkv", [(1, 1, 3, 1, 1), (5, 5, 4, 4, 2), (17, 17, 8, 4, 1),
                                          (7, 7, 1, 2, 2), (3, 9, 5, 2, 1), (16, 16, 64, 1, 1)])
def test_oracle_matches_scalar_brute_force(N, Nk, d, H, Hkv, causal):
    rng = np.random.default_rng(N * 1000 + d * 10 + H)
    B = 2
    Q = _rand((B, H, N, d), rng)
    K = _rand((B, Hkv, Nk, d), rng)
    V = _rand((B, Hkv, Nk, d), rng)
    scale = 0.37 + rng.random()
    O, LSE = oracle.attention(Q, K, V, causal=causal, scale=scale)
    Ob, Lb = brute_attention(Q.tolist(), K.tolist(), V.tolist(), causal, scale)
    np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, np.array(Lb), rtol=0, atol=1e-12)


def test_oracle_brute_force_d128():
    rng = np.random.default_rng(7)
    Q, K, V = (_rand((1, 2, 9, 128), rng) for _ in range(3))
    for causal in (False, True):
        O, LSE = oracle.attention(Q, K, V, causal=causal, scale=1 / math.sqrt(128))
        Ob, Lb = brute_attention(Q.tolist(), K.tolist(), V.tolist(), causal, 1 / math.sqrt(128))
        np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE, np.array(Lb), rtol=0, atol=1e-12)


def test_decode_oracle_matches_scalar_gather():
    """Page gather by explicit token loops through the page table."""
    rng = np.random.default_rng(3)
    B, H, Hkv, d, ps = 3, 4, 2, 8, 4
    lens = [1, 9, 16]
    P = sum(-(-L // ps) for L in lens)
    perm = rng.permutation(P)
    maxp = max(-(-L // ps) for L in lens)
    table = np.zeros((B, maxp), dtype=np.int64)
    off = 0
    for b, L in enumerate(lens):
        n = -(-L // ps)
        table[b, :n] = perm[off:off + n]
        off += n
    kp = rng.standard_normal((P, Hkv, ps, d))
    vp = rng.standard_normal((P, Hkv, ps, d))
    q = rng.standard_normal((B, H, d))
    scale = 0.3
    O, LSE = oracle.decode_paged(q, kp, vp, table, np.array(lens), scale=scale)
    for b, L in enumerate(lens):
        for h in range(H):
            kv = h // (H // Hkv)
            keys = [[kp[table[b, t // ps], kv, t % ps, e] for e in range(d)] for t in range(L)]
            vals = [[vp[table[b, t // ps], kv, t % ps, e] for e in range(d)] for t in range(L)]
            Ob, Lb = brute_attention([[[q[b, h].tolist()]]], [[keys]], [[vals]], False, scale)
            np.testing.assert_allclose(O[b, h], np.array(Ob[0][0][0]), rtol=0, atol=1e-12)
            assert abs(LSE[b, h] - Lb[0][0][0]) < 1e-12


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_closed_form_zero_keys(causal):
    """K = 0: every score is 0, so each row averages the V rows it may attend."""
    rng = np.random.default_rng(11)
    N, d = 37, 16
    Q = _rand((1, 1, N, d), rng) * 30
    K = np.zeros((1, 1, N, d))
    V = _rand((1, 1, N, d), rng)
    O, LSE = oracle.attention(Q, K, V, causal=causal, scale=0.125)
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(O[0, 0, i], V[0, 0, :n].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(LSE[0, 0, i] - math.log(n)) < 1e-13


def test_closed_form_two_keys_logistic():
    """Two keys: the weight of key 0 is the logistic function of s0 - s1."""
    for s0, s1 in [(0.3, -1.7), (5.0, 5.0), (-40.0, 12.5), (300.0, 299.0)]:
        Q = np.ones((1, 1, 1, 1))
        K = np.array([s0, s1]).reshape(1, 1, 2, 1)
        V = np.array([1.0, 0.0]).reshape(1, 1, 2, 1)
        O, LSE = oracle.attention(Q, K, V, causal=False, scale=1.0)
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        assert abs(O[0, 0, 0, 0] - w0) < 1e-14
        assert abs(LSE[0, 0, 0] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-12


def test_closed_form_single_key_decode():
    """L = 1: O = v_0 and LSE = s_0 = scale * q . k_0."""
    rng = np.random.default_rng(5)
    H, Hkv, d, ps = 8, 2, 32, 16
    kp = rng.standard_normal((3, Hkv, ps, d))
    vp = rng.standard_normal((3, Hkv, ps, d))
    q = rng.standard_normal((1, H, d))
    table = np.array([[2]])
    O, LSE = oracle.decode_paged(q, kp, vp, table, np.array([1]), scale=0.2)
    for h in range(H):
        kv = h // (H // Hkv)
        np.testing.assert_allclose(O[0, h], vp[2, kv, 0], rtol=0, atol=1e-15)
        assert abs(LSE[0, h] - 0.2 * float(q[0, h] @ kp[2, kv, 0])) < 1e-12


def test_empty_rows_and_partials():
    # no keys at all: O = 0, LSE = -inf
    O, LSE = oracle.attention(np.ones((1, 1, 2, 4)), np.zeros((1, 1, 0, 4)), np.zeros((1, 1, 0, 4)),
                              causal=False, scale=1.0)
    assert (O == 0).all() and np.isneginf(LSE).all()
    # an empty partial contributes nothing to a merge
    v = np.arange(6.0).reshape(3, 2)
    full = oracle.partial_state(np.array([0.1, 0.2, 0.3]), v)
    empty = oracle.partial_state(np.array([]), np.zeros((0, 2)))
    assert empty[0] == -np.inf and empty[1] == 0.0
    merged = oracle.merge_partials([empty, full, empty])
    np.testing.assert_allclose(merged[2], full[2], rtol=0, atol=0)
    assert merged[1] == full[1]
    o, lse = oracle.finalize(*oracle.merge_partials([empty, empty]))
    assert (o == 0).all() and lse == -np.inf


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_invariant_a_block_shape_independence(causal):
    rng = np.random.default_rng(21)
    N, d = 200, 16
    Q, K, V = (_rand((N, d), rng) for _ in range(3))
    O, LSE = oracle.attention(Q[None, None], K[None, None], V[None, None], causal=causal, scale=0.25)
    for bq, bk in [(1, 1), (3, 3), (16, 16), (64, 64), (128, 128), (N, N), (16, 64), (128, 3)]:
        Ot, Lt, _, _ = oracle.tiled_attention(Q, K, V, causal=causal, scale=0.25, block_q=bq, block_k=bk)
        np.testing.assert_allclose(Ot, O[0, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(Lt, LSE[0, 0], rtol=0, atol=1e-12)


def test_p1_self_checks():
    """The tutorial's NumPy setups: causal tiled (B_r = B_c = 16) vs plain at N = 100,
    d = 64; an 8-way key split vs plain for one decode query over L = 1000 keys."""
    rng = np.random.default_rng(0)
    N, d = 100, 64
    Q, K, V = (rng.standard_normal((N, d)) for _ in range(3))
    O, _ = oracle.attention(Q[None, None], K[None, None], V[None, None], causal=True, scale=1 / math.sqrt(d))
    Ot, _, _, _ = oracle.tiled_attention(Q, K, V, causal=True, scale=1 / math.sqrt(d), block_q=16, block_k=16)
    assert np.abs(Ot - O[0, 0]).max() < 1e-12
    L = 1000
    Kc, Vc, q = rng.standard_normal((L, d)), rng.standard_normal((L, d)), rng.standard_normal(d)
    s = Kc @ q / math.sqrt(d)
    cuts = np.linspace(0, L, 9).astype(int)
    parts = [oracle.partial_state(s[a:b], Vc[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    o, _ = oracle.finalize(*oracle.merge_partials(parts))
    ref, _ = oracle.attention(q[None, None, None], Kc[None, None], Vc[None, None], causal=False, scale=1 / math.sqrt(d))
    assert np.abs(o - ref[0, 0, 0]).max() < 1e-12


def _random_tree_merge(parts, rng):
    parts = list(parts)
    while len(parts) > 1:
        i = rng.randrange(len(parts) - 1)
        parts[i:i + 2] = [oracle.merge_partials([parts[i], parts[i + 1]])]
    return parts[0]


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16, 33, 64, 96])
def test_invariant_b_merge_any_partition_order_association(splits):
    rng = np.random.default_rng(splits)
    pyr = random.Random(splits)
    L, d = 500, 8
    s = rng.standard_normal(L) * 6
    v = rng.standard_normal((L, d))
    ref_o, ref_lse = oracle.finalize(*oracle.partial_state(s, v))
    # contiguous chunks (some may be empty when splits > useful), in order
    cuts = np.sort(rng.integers(0, L + 1, splits - 1))
    bounds = np.concatenate([[0], cuts, [L]])
    parts = [oracle.partial_state(s[a:b], v[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
    o, lse = oracle.finalize(*oracle.merge_partials(parts))
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    assert abs(lse - ref_lse) < 1e-12
    # random disjoint subsets, shuffled, merged along a random binary tree
    label = rng.integers(0, splits, L)
    parts = [oracle.partial_state(s[label == k], v[label == k]) for k in range(splits)]
    pyr.shuffle(parts)
    o, lse = oracle.finalize(*_random_tree_merge(parts, pyr))
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    assert abs(lse - ref_lse) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_invariant_c_convex_combination(causal):
    rng = np.random.default_rng(31)
    N, d = 120, 16
    Q = _rand((1, 2, N, d), rng) * 4
    K = _rand((1, 2, N, d), rng)
    V = _rand((1, 2, N, d), rng)
    O, _ = oracle.attention(Q, K, V, causal=causal, scale=0.25)
    for h in range(2):
        for i in range(N):
            att = V[0, h, : (i + 1 if causal else N)]
            assert (O[0, h, i] >= att.min(axis=0) - 1e-12).all()
            assert (O[0, h, i] <= att.max(axis=0) + 1e-12).all()


@pytest.mark.parametrize("mult", [30.0, 40.0])
def test_invariant_d_large_scores_no_overflow(mult):
    rng = np.random.default_rng(41)
    N, d = 256, 64
    Q = _rand((1, 1, N, d), rng) * mult
    K, V = (_rand((1, 1, N, d), rng) for _ in range(2))
    for causal in (False, True):
        O, LSE = oracle.attention(Q, K, V, causal=causal, scale=1 / 8)
        assert np.isfinite(O).all() and np.isfinite(LSE).all()
        assert LSE.max() > 100.0        # scores in the hundreds, as the pages' stress runs
        Ot, Lt, _, _ = oracle.tiled_attention(Q[0, 0], K[0, 0], V[0, 0], causal=causal, scale=1 / 8,
                                              block_q=64, block_k=64)
        np.testing.assert_allclose(Ot, O[0, 0], rtol=0, atol=1e-12)


def test_gqa_head_mapping_consecutive_heads_share():
    """Query heads h and h' with the same h // (H/Hkv) see the same K/V: giving them
    identical queries must give identical outputs, and other heads differ."""
    rng = np.random.default_rng(51)
    H, Hkv, N, d = 8, 2, 10, 4
    q1 = rng.standard_normal((N, d))
    Q = np.stack([q1] * H)[None]
    K, V = (_rand((1, Hkv, N, d), rng) for _ in range(2))
    O, _ = oracle.attention(Q, K, V, causal=False, scale=0.5)
    for h in range(H):
        np.testing.assert_array_equal(O[0, h], O[0, (h // 4) * 4])
    assert np.abs(O[0, 0] - O[0, 4]).max() > 1e-3


# ---------------------------------------------------------------------------
# Cascade decode: shared prefix + own suffix
# ---------------------------------------------------------------------------

def test_cascade_equals_decode_with_prefix_pages():
    """A page-aligned prefix stored as pages and prepended to every page table gives
    the same result through decode_paged as through cascade_decode."""
    rng = np.random.default_rng(61)
    B, H, Hkv, d, ps = 3, 8, 2, 16, 4
    npre = 3                                        # prefix of 3 pages = 12 tokens
    lens = [0, 5, 9]
    own = [-(-L // ps) for L in lens]
    P = npre + sum(own)
    kp = rng.standard_normal((P, Hkv, ps, d))
    vp = rng.standard_normal((P, Hkv, ps, d))
    q = rng.standard_normal((B, H, d))
    own_table = np.zeros((B, max(own)), dtype=np.int64)
    full_table = np.zeros((B, npre + max(own)), dtype=np.int64)
    off = npre
    for b, n in enumerate(own):
        own_table[b, :n] = np.arange(off, off + n)
        full_table[b, :npre] = np.arange(npre)
        full_table[b, npre:npre + n] = np.arange(off, off + n)
        off += n
    prefix_k = kp[:npre].transpose(1, 0, 2, 3).reshape(Hkv, npre * ps, d)
    prefix_v = vp[:npre].transpose(1, 0, 2, 3).reshape(Hkv, npre * ps, d)
    Oc, Lc = oracle.cascade_decode(q, prefix_k, prefix_v, kp, vp, own_table, np.array(lens), scale=0.3)
    Od, Ld = oracle.decode_paged(q, kp, vp, full_table, np.array(lens) + npre * ps, scale=0.3)
    np.testing.assert_allclose(Oc, Od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lc, Ld, rtol=0, atol=1e-12)


def test_cascade_brute_force_and_merge_identity():
    """Scalar brute force over prefix + suffix, and the merge of the two parts' states."""
    rng = np.random.default_rng(62)
    H, Hkv, d, ps, Lp, L = 2, 1, 4, 4, 5, 6
    kp = rng.standard_normal((2, Hkv, ps, d))
    vp = rng.standard_normal((2, Hkv, ps, d))
    pk = rng.standard_normal((Hkv, Lp, d))
    pv = rng.standard_normal((Hkv, Lp, d))
    q = rng.standard_normal((1, H, d))
    table = np.array([[1, 0]])
    O, LSE = oracle.cascade_decode(q, pk, pv, kp, vp, table, np.array([L]), scale=0.7)
    suffix_k = [kp[table[0, t // ps], 0, t % ps].tolist() for t in range(L)]
    suffix_v = [vp[table[0, t // ps], 0, t % ps].tolist() for t in range(L)]
    keys = pk[0].tolist() + suffix_k
    vals = pv[0].tolist() + suffix_v
    for h in range(H):
        Ob, Lb = brute_attention([[[q[0, h].tolist()]]], [[keys]], [[vals]], False, 0.7)
        np.testing.assert_allclose(O[0, h], np.array(Ob[0][0][0]), rtol=0, atol=1e-12)
        assert abs(LSE[0, h] - Lb[0][0][0]) < 1e-12
        sp = 0.7 * (pk[0] @ q[0, h])
        ss = 0.7 * (np.array(suffix_k) @ q[0, h])
        o2, l2 = oracle.finalize(*oracle.merge_partials([oracle.partial_state(sp, pv[0]),
                                                         oracle.partial_state(ss, np.array(suffix_v))]))
        np.testing.assert_allclose(o2, O[0, h], rtol=0, atol=1e-12)
        assert abs(l2 - LSE[0, h]) < 1e-12


@pytest.mark.parametrize("N,Nk", [(6, 3), (2, 9), (9, 2)])
def test_cross_attention_bottom_right_mask_brute_force(N, Nk):
    """Nq != Nk with the causal mask aligned to the last key; with Nq > Nk the first
    Nq - Nk rows attend nothing (O = 0, LSE = -inf)."""
    rng = np.random.default_rng(N * 10 + Nk)
    Q = rng.standard_normal((1, 2, N, 4))
    K = rng.standard_normal((1, 1, Nk, 4))
    V = rng.standard_normal((1, 1, Nk, 4))
    O, LSE = oracle.attention(Q, K, V, causal=True, scale=0.5)
    Ob, Lb = brute_attention(Q.tolist(), K.tolist(), V.tolist(), True, 0.5)
    np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(LSE), np.isneginf(np.array(Lb)))
    fin = np.isfinite(LSE)
    np.testing.assert_allclose(LSE[fin], np.array(Lb)[fin], rtol=0, atol=1e-12)
    if N > Nk:
        assert np.isneginf(LSE[0, :, : N - Nk]).all() and (O[0, :, : N - Nk] == 0).all()


# ---------------------------------------------------------------------------
# Ragged batches (indptr) and paged prefill
# ---------------------------------------------------------------------------

def test_varlen_equal_lengths_is_dense_attention():
    rng = np.random.default_rng(71)
    B, H, Hkv, N, d = 3, 4, 2, 9, 8
    Q = rng.standard_normal((B, H, N, d))
    K = rng.standard_normal((B, Hkv, N, d))
    V = rng.standard_normal((B, Hkv, N, d))
    indptr = np.arange(B + 1) * N
    q = Q.transpose(0, 2, 1, 3).reshape(B * N, H, d)
    k = K.transpose(0, 2, 1, 3).reshape(B * N, Hkv, d)
    v = V.transpose(0, 2, 1, 3).reshape(B * N, Hkv, d)
    for causal in (False, True):
        O, LSE = oracle.attention(Q, K, V, causal=causal, scale=0.4)
        Ov, Lv = oracle.varlen_attention(q, k, v, indptr, indptr, causal=causal, scale=0.4)
        np.testing.assert_allclose(Ov, O.transpose(0, 2, 1, 3).reshape(B * N, H, d), rtol=0, atol=1e-12)
        np.testing.assert_allclose(Lv, LSE.transpose(0, 2, 1).reshape(B * N, H), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_unequal_lengths_brute_force(causal):
    """Ragged batch whose query and key lengths differ per sequence (Lq < Lk, Lq > Lk,
    Lq = 0, Lk = 0, Lq = Lk), each sequence checked against the scalar brute force on
    its own slices: query rows [qo_indptr[b], qo_indptr[b+1]) against key rows
    [kv_indptr[b], kv_indptr[b+1]), the causal mask aligned to the sequence's last key.
    A sequence with queries but no keys has O = 0 and LSE = -inf."""
    rng = np.random.default_rng(73)
    H, Hkv, d = 4, 2, 5
    q_lens = [3, 0, 6, 2, 4, 1]
    k_lens = [7, 4, 2, 0, 4, 9]
    qo = np.concatenate([[0], np.cumsum(q_lens)])
    kvp = np.concatenate([[0], np.cumsum(k_lens)])
    q = rng.standard_normal((qo[-1], H, d))
    k = rng.standard_normal((kvp[-1], Hkv, d))
    v = rng.standard_normal((kvp[-1], Hkv, d))
    O, LSE = oracle.varlen_attention(q, k, v, qo, kvp, causal=causal, scale=0.45)
    assert O.shape == (qo[-1], H, d) and LSE.shape == (qo[-1], H)
    for b in range(len(q_lens)):
        rows = slice(qo[b], qo[b + 1])
        if q_lens[b] == 0:
            continue
        if k_lens[b] == 0:
            assert (O[rows] == 0).all() and np.isneginf(LSE[rows]).all()
            continue
        Qb = [[q[rows, h].tolist() for h in range(H)]]
        Kb = [[k[kvp[b]:kvp[b + 1], g].tolist() for g in range(Hkv)]]
        Vb = [[v[kvp[b]:kvp[b + 1], g].tolist() for g in range(Hkv)]]
        Ob, Lb = brute_attention(Qb, Kb, Vb, causal, 0.45)
        np.testing.assert_allclose(O[rows], np.array(Ob[0]).transpose(1, 0, 2), rtol=0, atol=1e-12)
        Lb = np.array(Lb[0]).T
        np.testing.assert_array_equal(np.isneginf(LSE[rows]), np.isneginf(Lb))
        fin = np.isfinite(Lb)
        np.testing.assert_allclose(LSE[rows][fin], Lb[fin], rtol=0, atol=1e-12)
    if causal:  # sequence 2 has 6 queries and 2 keys: its first 4 rows attend nothing
        assert np.isneginf(LSE[qo[2]:qo[2] + 4]).all() and (O[qo[2]:qo[2] + 4] == 0).all()
        assert np.isfinite(LSE[qo[2] + 4:qo[3]]).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,Nk,H,Hkv", [(1, 1, 1, 1), (6, 6, 2, 1), (4, 9, 4, 2), (9, 4, 2, 2), (17, 17, 1, 1)])
def test_attention_weights_brute_force(N, Nk, H, Hkv, causal):
    """oracle.attention_weights against the scalar softmax weights, head by head (GQA,
    cross shapes with the mask aligned to the last key)."""
    rng = np.random.default_rng(N * 31 + Nk * 7 + H + causal)
    d = 6
    Q = rng.standard_normal((1, H, N, d)) * 2.0
    K = rng.standard_normal((1, Hkv, Nk, d))
    rows = np.arange(N)
    for h in range(H):
        P, LSE = oracle.attention_weights(Q, K, 0, h, rows, causal=causal, scale=0.6)
        Wb = np.array(brute_weights(Q[0, h].tolist(), K[0, h // (H // Hkv)].tolist(), causal, 0.6, Nk - N))
        np.testing.assert_allclose(P, Wb, rtol=0, atol=1e-14)
        live = Wb.sum(axis=1) > 0
        np.testing.assert_allclose(P[live].sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.isneginf(LSE[~live]).all() and np.isfinite(LSE[live]).all()


def test_attention_weights_closed_form_zero_keys():
    """K = 0: causal row i weighs its i + 1 keys equally, non-causal rows weigh all N keys equally."""
    Q = np.random.default_rng(5).standard_normal((1, 1, 7, 4))
    K = np.zeros((1, 1, 7, 4))
    P, _ = oracle.attention_weights(Q, K, 0, 0, np.arange(7), causal=True, scale=1.0)
    expect = np.tril(np.ones((7, 7))) / np.arange(1, 8)[:, None]
    np.testing.assert_allclose(P, expect, rtol=0, atol=1e-15)
    P, _ = oracle.attention_weights(Q, K, 0, 0, np.arange(7), causal=False, scale=1.0)
    np.testing.assert_allclose(P, np.full((7, 7), 1 / 7), rtol=0, atol=1e-15)


def test_paged_prefill_brute_force():
    """Query chunks that are the last tokens of each sequence, keys gathered page by page."""
    rng = np.random.default_rng(72)
    H, Hkv, d, ps = 2, 1, 4, 4
    kv_lens = [6, 9]
    q_lens = [2, 9]
    pages = [-(-L // ps) for L in kv_lens]
    P = sum(pages)
    perm = rng.permutation(P)
    table = np.zeros((2, max(pages)), dtype=np.int64)
    table[0, :pages[0]] = perm[:pages[0]]
    table[1, :pages[1]] = perm[pages[0]:]
    kp = rng.standard_normal((P, Hkv, ps, d))
    vp = rng.standard_normal((P, Hkv, ps, d))
    qo = np.array([0, 2, 11])
    q = rng.standard_normal((11, H, d))
    O, LSE = oracle.paged_prefill(q, kp, vp, table, np.array(kv_lens), qo, causal=True, scale=0.6)
    for b in range(2):
        L, Lq = kv_lens[b], q_lens[b]
        keys = [[kp[table[b, t // ps], 0, t % ps, e] for e in range(d)] for t in range(L)]
        vals = [[vp[table[b, t // ps], 0, t % ps, e] for e in range(d)] for t in range(L)]
        rows = q[qo[b]:qo[b + 1]]
        Qb = [[rows[:, h].tolist() for h in range(H)]]
        Ob, Lb = brute_attention(Qb, [[keys]], [[vals]], True, 0.6)
        np.testing.assert_allclose(O[qo[b]:qo[b + 1]], np.array(Ob[0]).transpose(1, 0, 2), rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE[qo[b]:qo[b + 1]], np.array(Lb[0]).T, rtol=0, atol=1e-12)
