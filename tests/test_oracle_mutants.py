"""The oracle's pins are strong enough: each plausible mistake, planted in a
copy of the oracle's source on the CPU, makes at least one pin fail."""

import os
import types

import numpy as np
import pytest

from tests import oracle_pins, oracle_pins_fp8

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "attention.py")
SRC_FP8 = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "fp8.py")

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
    # the spot-check and head-subset forms used on full-size launches
    ("rows_mask_shifted", "vis = visible(N, N, causal, window)[rows]",
     "vis = visible(N, N, causal, window)[rows - 1]"),
    ("rows_wrong_kv_head", "hk = h // (Hq // Hkv)", "hk = h % Hkv"),
    ("rows_first_batch", "_f64(q[b, rows, h])", "_f64(q[0, rows, h])"),
    ("decode_cache_reused", "if (b, hk) not in cached:", "if not cached:"),
    ("decode_cache_kept_per_batch", "if (b, hk) not in cached:",
     "if b not in [key[0] for key in cached]:"),
    ("decode_first_length", "n = int(kv_len[b])\n        hk = h // G\n        if (b, hk)",
     "n = int(kv_len[0])\n        hk = h // G\n        if (b, hk)"),
    ("decode_gqa_modulo", "hk = h // G\n        if (b, hk) not in cached",
     "hk = h % Hkv\n        if (b, hk) not in cached"),
]


# the same for the FP8 module (e4m3 rounding, scale exponents, tile layout,
# the P-rounding error bound)
MUTANTS_FP8 = [
    ("round_half_away", "r = np.rint(a / step) * step", "r = np.floor(a / step + 0.5) * step"),
    ("subnormal_step", "E4M3_SUBNORMAL_STEP = 2.0 ** -9", "E4M3_SUBNORMAL_STEP = 2.0 ** -10"),
    ("no_saturation", "r = np.minimum(r, E4M3_MAX)", "r = r"),
    ("exponent_tie_side", "e = np.where(f <= 0.875, 9 - x, 8 - x)",
     "e = np.where(f < 0.875, 9 - x, 8 - x)"),
    ("exponent_one_high", "e = np.where(f <= 0.875, 9 - x, 8 - x)",
     "e = np.where(f <= 0.875, 10 - x, 9 - x)"),
    ("dequant_wrong_sign", "deq[b, t * tile:(t + 1) * tile, h] = g * 2.0 ** -e",
     "deq[b, t * tile:(t + 1) * tile, h] = g * 2.0 ** e"),
    ("tile_overlaps_next", "blk = x[b, t * tile:(t + 1) * tile, h]",
     "blk = x[b, t * tile:(t + 1) * tile + 1, h]"),
    ("v_not_transposed_order", "codes[b, h, :, :N] = e4m3_encode(g).T",
     "codes[b, h, :, :N] = e4m3_encode(g).T[::-1]"),
    ("bound_no_floor", "eps = np.maximum(2.0 ** -4 * p, 2.0 ** -10) * (P > 0)",
     "eps = 2.0 ** -4 * p * (P > 0)"),
    ("bound_unnormalised", "l = 1.0 / pmax  # sum_j p_j = 1 / max_j P_j", "l = 1.0"),
]


def _mutant_module(old, new, src_path=SRC):
    src = open(src_path).read()
    assert src.count(old) == 1, f"mutation anchor must occur exactly once: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    mod.__package__ = "oracle"  # relative imports resolve to the real oracle package
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def _some_pin_fails(mod, pins=None):
    for pin in (oracle_pins.ALL_PINS if pins is None else pins):
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


@pytest.mark.parametrize("name,old,new", MUTANTS_FP8, ids=[m[0] for m in MUTANTS_FP8])
def test_planted_fp8_mistake_is_caught(name, old, new):
    caught = _some_pin_fails(_mutant_module(old, new, SRC_FP8), oracle_pins_fp8.FP8_PINS)
    assert caught is not None, f"no pin catches the planted mistake {name!r}"


def test_unmutated_copy_passes():
    src = open(SRC).read()
    mod = types.ModuleType("oracle_copy")
    exec(compile(src, "oracle_copy", "exec"), mod.__dict__)
    assert _some_pin_fails(mod) is None
    mod8 = types.ModuleType("oracle_fp8_copy")
    mod8.__package__ = "oracle"
    exec(compile(open(SRC_FP8).read(), "oracle_fp8_copy", "exec"), mod8.__dict__)
    assert _some_pin_fails(mod8, oracle_pins_fp8.FP8_PINS) is None
