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
