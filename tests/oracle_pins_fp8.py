"""Checks that pin the FP8 part of the oracle (``oracle/fp8.py``) to facts that
do not come from its own code.

Each ``pin_*`` takes the FP8 oracle module (so that the mutation test can run
the same checks against a deliberately broken copy) and raises AssertionError
on a disagreement with:
  * PyTorch's float8_e4m3fn type: its bit patterns give the value of every
    code, and its CPU cast is a round-to-nearest-even conversion,
  * closed forms of the e4m3 format (largest value, smallest subnormal, ties),
  * the defining inequality of the scale exponent,
  * the round-trip error bound of the format and the locality of tile scales,
  * exact attention, when every input already lies on the scaled e4m3 grid,
  * an emulation (with PyTorch's cast) of rounding the softmax numerators.
"""

from __future__ import annotations

import math

import numpy as np
import torch


def _torch_grid():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    return codes, vals


def _torch_round(x):
    """e4m3 rounding by PyTorch's cast (values of magnitude <= 448 only; the
    cast gives NaN, not 448, above the largest finite value)."""
    x = np.asarray(x, dtype=np.float32)
    return torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).double().numpy()


def pin_e4m3_code_table(f):
    codes, vals = _torch_grid()
    fin = ~np.isnan(vals)
    dec = f.e4m3_decode(codes)
    assert np.array_equal(np.isnan(dec), ~fin), "NaN codes"
    assert np.array_equal(dec[fin], vals[fin]), "decoded values"
    assert np.array_equal(np.signbit(dec[fin]), np.signbit(vals[fin])), "sign of zero"
    assert np.array_equal(f.e4m3_round(vals[fin]), vals[fin]), "grid points are fixed points"
    assert np.array_equal(f.e4m3_encode(vals[fin]), codes[fin]), "encode(decode(c)) == c"


def pin_e4m3_rounding_matches_torch(f, seed=20):
    _, vals = _torch_grid()
    g = np.unique(np.abs(vals[~np.isnan(vals)]))
    mids = (g[1:] + g[:-1]) / 2  # every tie between neighbouring grid values
    rng = np.random.default_rng(seed)
    rnd = np.float32(2.0) ** rng.uniform(-13, math.log2(448), 20000).astype(np.float32)
    xs = np.concatenate([mids, -mids, rnd, -rnd, g, -g]).astype(np.float32)
    xs = xs[np.abs(xs) <= 448]
    got = f.e4m3_round(xs.astype(np.float64))
    want = _torch_round(xs)
    assert np.array_equal(got, want), f"{np.sum(got != want)} roundings differ from torch"
    assert np.array_equal(np.signbit(got), np.signbit(want)), "sign of rounded zeros"


def pin_e4m3_closed_forms(f):
    cases = {
        448.0: 448.0, 464.0: 448.0, 1000.0: 448.0, -1000.0: -448.0, 1e30: 448.0,
        2.0 ** -9: 2.0 ** -9, 2.0 ** -10: 0.0, 1.5 * 2.0 ** -10: 2.0 ** -9, 3 * 2.0 ** -10: 2.0 ** -8,
        2.0 ** -6: 2.0 ** -6, 1.0625: 1.0, 1.1875: 1.25, 240.0: 240.0, 248.0: 256.0, 0.0: 0.0,
    }
    for x, y in cases.items():
        r = float(f.e4m3_round(np.array([x]))[0])
        assert r == y, f"e4m3_round({x}) = {r}, expected {y}"
    enc = {448.0: 0x7E, 1.0: 0x38, 2.0 ** -9: 0x01, -2.0: 0xC0, 2.0 ** -6: 0x08, 0.0: 0x00}
    for x, c in enc.items():
        got = int(f.e4m3_encode(np.array([x]))[0])
        assert got == c, f"e4m3_encode({x}) = {got:#x}, expected {c:#x}"


def pin_scale_exponent(f, seed=21):
    rng = np.random.default_rng(seed)
    amax = 2.0 ** rng.uniform(-100, 100, 5000)
    amax = np.concatenate([amax, [448.0, 449.0, 1.0, 1.75, 1.7500001, 224.0, 3.0, 2.0 ** 100]])
    e = f.scale_exponent(amax)
    assert np.issubdtype(e.dtype, np.integer)
    assert np.all(amax * 2.0 ** e <= 448.0), "amax * 2^e exceeds 448"
    assert np.all(amax * 2.0 ** (e + 1) > 448.0), "a larger exponent would still fit"
    fixed = {0.0: 0, 448.0: 0, 449.0: -1, 1.0: 8, 1.75: 8, 2.0 ** -130: 126}
    for a, want in fixed.items():
        assert int(f.scale_exponent(np.array([a]))[0]) == want, a


def pin_quantize_tiles(f, seed=22):
    rng = np.random.default_rng(seed)
    B, N, H, d = 2, 300, 3, 64  # three row tiles, the last one ragged (44 rows)
    x = rng.standard_normal((B, N, H, d)) * np.exp(rng.uniform(-4, 4, (B, N, H, 1)))
    x = x.astype(np.float32).astype(np.float64)
    codes, exps, deq = f.quantize_row_tiles(x)
    assert codes.shape == x.shape and exps.shape == (B, H, 3) and codes.dtype == np.uint8
    for b in range(B):
        for h in range(H):
            for t in range(3):
                blk = x[b, 128 * t:128 * (t + 1), h]
                e = exps[b, h, t]
                top = np.abs(blk).max() * 2.0 ** e
                assert 224.0 < top <= 448.0, (b, h, t, top)
                # format round trip: half a step, relative or absolute (subnormal)
                err = np.abs(deq[b, 128 * t:128 * (t + 1), h] - blk)
                bound = np.maximum(2.0 ** -4 * np.abs(blk), 2.0 ** -10 * 2.0 ** -float(e))
                assert np.all(err <= bound), (b, h, t)
    dec = f.e4m3_decode(codes) * 2.0 ** -np.repeat(exps, 128, axis=2)[:, :, :N].transpose(0, 2, 1)[..., None]
    assert np.array_equal(dec, deq), "codes and exponents do not give the dequantised values"
    # a huge value in the first row of tile 1 of (b=1, h=2) moves that tile only
    y = x.copy()
    y[1, 128, 2, 5] = 1e4
    c2, e2, _ = f.quantize_row_tiles(y)
    changed = np.argwhere(e2 != exps)
    assert changed.tolist() == [[1, 2, 1]], changed.tolist()
    rows = np.unique(np.argwhere(c2 != codes)[:, [0, 1, 2]], axis=0)
    assert set(map(tuple, rows[:, [0, 2]])) == {(1, 2)} and rows[:, 1].min() >= 128 \
        and rows[:, 1].max() < 256


def pin_quantize_v_transposed(f, seed=23):
    rng = np.random.default_rng(seed)
    B, N, H, d = 2, 37, 2, 16
    v = rng.standard_normal((B, N, H, d)).astype(np.float32).astype(np.float64)
    v[0, 36, 1, 3] = 9.0
    codes, exps, deq = f.quantize_per_head_transposed(v)
    assert codes.shape == (B, H, d, 48) and exps.shape == (B, H)
    assert np.all(codes[..., 37:] == 0), "padding keys must be zero"
    for b in range(B):
        for h in range(H):
            e = exps[b, h]
            assert 224.0 < np.abs(v[b, :, h]).max() * 2.0 ** e <= 448.0
            back = f.e4m3_decode(codes[b, h, :, :N]).T * 2.0 ** -float(e)
            assert np.array_equal(back, deq[b, :, h])
            assert np.all(np.abs(back - v[b, :, h]) <=
                          np.maximum(2.0 ** -4 * np.abs(v[b, :, h]), 2.0 ** -10 * 2.0 ** -float(e)))
    assert exps[0, 1] == 5  # amax 9: 9 * 2^5 = 288 <= 448 < 576


def pin_fp8_attention_on_grid_inputs(f, seed=24):
    """Inputs whose every tile holds a +-2 and otherwise values of
    {0, +-0.25, +-0.5, +-1, +-1.5}: the exponent is 7 everywhere and x * 128 is
    on the e4m3 grid, so quantisation is exact and FP8 attention must equal
    exact attention on the original inputs."""
    import oracle
    rng = np.random.default_rng(seed)
    B, N, Hq, Hkv, d = 1, 200, 4, 2, 32
    pool = np.array([0, 0.25, -0.25, 0.5, -0.5, 1, -1, 1.5, -1.5])

    def mk(H):
        x = rng.choice(pool, size=(B, N, H, d))
        x[:, ::128, :, 0] = 2.0  # first row of every 128-row tile
        return x

    q, k, v = mk(Hq), mk(Hkv), mk(Hkv)
    for causal, window in [(False, -1), (True, -1), (False, 20)]:
        O, L, qz = f.attention_fp8(q, k, v, causal=causal, window=window)
        assert np.all(qz["q_exp"] == 7) and np.all(qz["k_exp"] == 7) and np.all(qz["v_exp"] == 7)
        O2, L2 = oracle.attention(q, k, v, causal=causal, window=window)
        assert np.array_equal(O, O2) and np.array_equal(L, L2), (causal, window)


def _emulate_rounded_p(q, k, v, causal, window, lag):
    """O with the softmax numerators rounded to e4m3 by PyTorch's cast, in
    units where the row maximum is 2^lag, divided by the unrounded sum."""
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    scale = 1.0 / math.sqrt(d)
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    vis = np.ones((N, N), bool)
    if causal:
        vis &= j <= i
    if window >= 0:
        vis &= (np.abs(i - j) <= window) if not causal else (i - j <= window)
    O = np.zeros((B, N, Hq, d))
    for b in range(B):
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            S = np.where(vis, scale * q[b, :, h] @ k[b, :, hk].T, -np.inf)
            p = np.exp(S - S.max(axis=1, keepdims=True)) * 2.0 ** lag
            O[b, :, h] = (_torch_round(p) @ v[b, :, hk]) / p.sum(axis=1, keepdims=True)
    return O


def pin_p_rounding_bound(f, seed=25):
    """The error of rounding P to e4m3, emulated with PyTorch's cast, stays
    within a few bound units and its RMS is a sizeable fraction of the bound."""
    import oracle
    rng = np.random.default_rng(seed)
    B, N, H, d = 1, 300, 2, 32
    q0, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    # (query scale, causal, window, lag): a larger query scale spreads the
    # scores, so that most numerators fall below the smallest normal e4m3
    for qs, causal, window, lag in [(1.0, False, -1, 0.0), (1.0, True, -1, 3.7),
                                    (1.0, False, 40, 7.5), (8.0, False, -1, 0.0)]:
        q = q0 * qs
        O, _ = oracle.attention(q, k, v, causal=causal, window=window)
        bound = f.p_rounding_bound(q, k, v, causal=causal, window=window)
        err = np.abs(_emulate_rounded_p(q, k, v, causal, window, lag) - O)
        ratio = err / np.maximum(bound, 1e-300)
        assert ratio.max() <= 3.0, (causal, window, lag, ratio.max())
        rms = float(np.sqrt(np.mean(ratio ** 2)))
        assert 0.05 <= rms <= 1.0, (causal, window, lag, rms)
    sub = f.p_rounding_bound(q0, k, v, causal=True, rows=[0, 5, 299])
    full = f.p_rounding_bound(q0, k, v, causal=True)
    assert np.allclose(sub, full[:, [0, 5, 299]], rtol=1e-12, atol=0), "row subset"


FP8_PINS = [
    pin_e4m3_code_table, pin_e4m3_rounding_matches_torch, pin_e4m3_closed_forms,
    pin_scale_exponent, pin_quantize_tiles, pin_quantize_v_transposed,
    pin_fp8_attention_on_grid_inputs, pin_p_rounding_bound,
]
