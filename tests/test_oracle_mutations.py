"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each.

Each mutation patches one internal step of the oracle module for the duration
of a test and runs the pins that should fail because of it.
"""
import sys

import numpy as np
import pytest

import oracle  # noqa: F401  (loads the submodule)
from tests import test_oracle_pins as pins

ORC = sys.modules["oracle.attention"]


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _mut_mask_transposed(rows, Nk, N):
    cols = np.arange(Nk)
    return cols[None, :] >= rows[:, None]


def _mut_mask_strict(rows, Nk, N):
    cols = np.arange(Nk)
    return cols[None, :] < rows[:, None] + (Nk - N)


def _mut_softmax_log2(S, Vh):
    O, lse = _ORIG_SOFTMAX(S, Vh)
    return O, lse / np.log(2.0)


def _mut_softmax_sign(S, Vh):
    return _ORIG_SOFTMAX(-S, Vh)


def _mut_softmax_no_norm(S, Vh):
    m = S.max(axis=1)
    P = np.exp(S - m[:, None])
    return P @ Vh, m + np.log(P.sum(axis=1))


def _mut_softmax_transposed_v(S, Vh):
    if Vh.shape[0] == Vh.shape[1]:
        return _ORIG_SOFTMAX(S, Vh.T.copy())
    return _ORIG_SOFTMAX(S, Vh[::-1].copy())


_ORIG_SOFTMAX = ORC._softmax_rows


@pytest.mark.parametrize("mutant,checks", [
    (("_causal_keep", _mut_mask_transposed), ["zero_keys_causal", "brute_causal"]),
    (("_causal_keep", _mut_mask_strict), ["zero_keys_causal", "brute_causal"]),
    (("_softmax_rows", _mut_softmax_log2), ["zero_keys", "p4_final"]),
    (("_softmax_rows", _mut_softmax_sign), ["p4_final", "p2_lab"]),
    (("_softmax_rows", _mut_softmax_no_norm), ["zero_keys", "p2_lab"]),
    (("_softmax_rows", _mut_softmax_transposed_v), ["brute", "zero_keys"]),
])
def test_pins_catch_planted_mistake(monkeypatch, mutant, checks):
    name, fn = mutant
    monkeypatch.setattr(ORC, name, fn)
    table = {
        "zero_keys_causal": (pins.test_closed_form_zero_keys, True),
        "zero_keys": (pins.test_closed_form_zero_keys, False),
        "brute_causal": (pins.test_oracle_matches_scalar_brute_force, 5, 5, 4, 4, 2, True),
        "brute": (pins.test_oracle_matches_scalar_brute_force, 5, 5, 4, 4, 2, False),
        "p4_final": (pins.test_p4_worked_example_final_output,),
        "p2_lab": (pins.test_p2_online_softmax_lab, 4),
    }
    caught = [c for c in checks if _fails(*table[c])]
    assert caught, f"no pin caught mutation {name}={fn.__name__}"


def test_pins_catch_dropped_scale(monkeypatch):
    orig = ORC.attention_rows

    def no_scale(Q, K, V, b, h, rows, *, causal, scale):
        return orig(Q, K, V, b, h, rows, causal=causal, scale=1.0)

    monkeypatch.setattr(ORC, "attention_rows", no_scale)
    assert _fails(pins.test_oracle_matches_scalar_brute_force, 5, 5, 4, 4, 2, False)


def test_pins_catch_wrong_gqa_mapping(monkeypatch):
    orig = ORC.attention_rows

    def modulo_map(Q, K, V, b, h, rows, *, causal, scale):
        Hkv = K.shape[1]
        H = Q.shape[1]
        # interleaved mapping h % Hkv, emulated by permuting heads before the call
        perm = [(hh % Hkv) * (H // Hkv) + hh // Hkv for hh in range(H)]
        return orig(Q[:, perm], K, V, b, h, rows, causal=causal, scale=scale)

    monkeypatch.setattr(ORC, "attention_rows", modulo_map)
    assert _fails(pins.test_oracle_matches_scalar_brute_force, 5, 5, 4, 4, 2, False)


def test_pins_catch_merge_without_rescale(monkeypatch):
    def bad_merge(parts):
        parts = [(float(m), float(l), np.asarray(o, dtype=np.float64)) for m, l, o in parts]
        m = max(p[0] for p in parts)
        return m, sum(p[1] for p in parts), sum(p[2] for p in parts)

    monkeypatch.setattr(ORC, "merge_partials", bad_merge)
    monkeypatch.setattr(oracle, "merge_partials", bad_merge)
    assert _fails(pins.test_p4_worked_example_block_states)
    assert _fails(pins.test_invariant_b_merge_any_partition_order_association, 7)


def _varlen_swapped(orig):
    def swapped(q, k, v, qo_indptr, kv_indptr, *, causal, scale):
        return orig(q, k, v, kv_indptr, qo_indptr, causal=causal, scale=scale)
    return swapped


def _varlen_keys_by_query_offsets(q, k, v, qo_indptr, kv_indptr, *, causal, scale):
    """Slices each sequence's keys with the query offsets (a plausible copy-paste slip)."""
    return _ORIG_VARLEN(q, k, v, qo_indptr, qo_indptr, causal=causal, scale=scale)


_ORIG_VARLEN = ORC.varlen_attention


@pytest.mark.parametrize("mutant", ["swapped", "keys_by_query_offsets"])
def test_unequal_length_pin_catches_indptr_mistakes(monkeypatch, mutant):
    """Swapped or mis-sliced indptr arrays pass the equal-length pin (both arrays are
    the same there) and fail the pin with unequal query and key lengths."""
    fn = _varlen_swapped(_ORIG_VARLEN) if mutant == "swapped" else _varlen_keys_by_query_offsets
    monkeypatch.setattr(ORC, "varlen_attention", fn)
    monkeypatch.setattr(oracle, "varlen_attention", fn)
    assert not _fails(pins.test_varlen_equal_lengths_is_dense_attention)
    assert _fails(pins.test_varlen_unequal_lengths_brute_force, False) or \
        _fails(pins.test_varlen_unequal_lengths_brute_force, True)


def _weights_unnormalised(S):
    P, lse = _ORIG_WEIGHTS(S)
    return P * 1.5, lse


def _weights_transposed_mask(S):
    n, Nk = S.shape
    if n == Nk:
        S = np.where(np.isneginf(S), S.T, S)
    return _ORIG_WEIGHTS(S)


def _weights_base2(S):
    return _ORIG_WEIGHTS(S / np.log(2.0))


_ORIG_WEIGHTS = ORC._softmax_weights


@pytest.mark.parametrize("fn", [_weights_unnormalised, _weights_transposed_mask, _weights_base2])
def test_weight_pins_catch_planted_mistake(monkeypatch, fn):
    monkeypatch.setattr(ORC, "_softmax_weights", fn)
    caught = _fails(pins.test_attention_weights_brute_force, 6, 6, 2, 1, True) or \
        _fails(pins.test_attention_weights_closed_form_zero_keys)
    assert caught, f"no pin caught {fn.__name__}"
