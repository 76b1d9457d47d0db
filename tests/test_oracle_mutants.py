"""The oracle's pins are strong enough: each plausible mistake, planted in a
copy of the oracle's source on the CPU, makes at least one pin fail."""

import os
import types

import numpy as np
import pytest

from tests import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "attention.py")

# (name, text in the oracle, planted replacement)
MUTANTS = [
    ("causal_off_by_one", "vis &= j <= i", "vis &= j < i"),
    ("window_exclusive", "vis &= np.abs(i - j) <= window", "vis &= np.abs(i - j) < window"),
    ("window_causal_sign", "vis &= (i - j) <= window", "vis &= (j - i) <= window"),
    ("transposed_scores", "S = scale * (q @ k.T)", "S = scale * (k @ q.T)"),
    ("dropped_scale", "S = scale * (q @ k.T)", "S = (q @ k.T)"),
    ("no_max_subtraction", "E = np.exp(S - m_safe[:, None])", "E = np.exp(S)"),
    ("unnormalised_p", "P = E / l_safe[:, None]", "P = E"),
    ("lse_drops_max", "m_safe + np.log(l_safe)", "np.log(l_safe)"),
    ("lse_log2", "m_safe + np.log(l_safe)", "m_safe + np.log2(l_safe)"),
    ("gqa_modulo", "hk = h // G\n            O[b, :, h]", "hk = h % Hkv\n            O[b, :, h]"),
    ("merge_no_rescale_l", "l1 * w1 + l2 * w2", "l1 + l2"),
    ("merge_min", "M = max(m1, m2)", "M = min(m1, m2)"),
    ("tree_drops_odd", "        if len(level) % 2:\n            nxt.append(level[-1])\n", ""),
    ("split_bounds", "lo, hi = c * chunk, min((c + 1) * chunk, n)",
     "lo, hi = c * chunk, min((c + 1) * chunk - 1, n)"),
    ("partial_no_exp_o", "return m, e.sum(), e @ vv", "return m, e.sum(), vv.sum(axis=0)"),
    ("band_narrow", "c1 = min(N, r1 + window)", "c1 = min(N, r1 + window - 1)"),
    ("varlen_slice_end", "O[a:e] = o_s[0]", "O[a:e] = o_s[0][::-1]"),
    ("bwd_drops_row_term", "dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))", "dS = P * dP"),
    ("bwd_dk_no_scale", "dK[b, :, hk] += scale * (dS.T @ q[b, :, h])", "dK[b, :, hk] += dS.T @ q[b, :, h]"),
    ("bwd_dv_untransposed", "dV[b, :, hk] += P.T @ do", "dV[b, :, hk] += P @ do"),
    ("bwd_gqa_overwrites", "dK[b, :, hk] += scale", "dK[b, :, hk] = scale"),
    ("empty_row_lse_zero", "lse = np.where(empty, NEG_INF, m_safe + np.log(l_safe))",
     "lse = np.where(empty, 0.0, m_safe + np.log(l_safe))"),
]


def _mutant_module(old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor must occur exactly once: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def _some_pin_fails(mod):
    for pin in oracle_pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except Exception:  # AssertionError, or a crash the mistake causes
            return pin.__name__
    return None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    caught = _some_pin_fails(_mutant_module(old, new))
    assert caught is not None, f"no pin catches the planted mistake {name!r}"


def test_unmutated_copy_passes():
    src = open(SRC).read()
    mod = types.ModuleType("oracle_copy")
    exec(compile(src, "oracle_copy", "exec"), mod.__dict__)
    assert _some_pin_fails(mod) is None
