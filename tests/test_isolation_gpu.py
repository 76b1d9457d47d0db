"""Rows outside a sequence never reach its results.

A key tile that runs past a sequence's end holds the next sequence's rows (or
the rows after the last sequence).  Their scores are masked, so their weights
are exactly 0, but 0 times a non-finite value is not 0.  These tests plant NaN
in one sequence, or past the last sequence, and check that every other
sequence's O, LSE and gradients still match the float64 oracle, which only
ever sees the sequence itself ("FlashAttention" learn page, FAQ: the output is
that of standard attention, sequence by sequence).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3
NAN = float("nan")


@pytest.fixture(scope="module")
def fa():
    from exact_transformer_attention_flashattention_b300 import binding
    return binding


def _check(O, L, O_ref, L_ref, what):
    O = O.detach().double().cpu().numpy()
    L = L.detach().double().cpu().numpy()
    assert np.isfinite(O).all() and np.isfinite(L).all(), f"{what}: non-finite result"
    dO = np.abs(O - O_ref)
    dL = np.abs(L - L_ref)
    assert dO.max() <= O_MAX and dO.mean() <= O_MEAN, (what, dO.max(), dO.mean())
    assert dL.max() <= LSE_MAX, (what, dL.max())


DENSE = [
    # B, Hq, Hkv, N, d, causal, window
    (2, 2, 2, 300, 128, True, -1),
    (2, 2, 2, 300, 64, False, -1),
    (3, 4, 2, 200, 128, False, 50),
    (2, 2, 1, 129, 64, True, 100),
    (2, 2, 2, 300, 64, False, 100),   # short non-causal window at d = 64
]


@pytest.mark.parametrize("case", DENSE, ids=lambda c: "-".join(map(str, c)))
def test_dense_prefill_ignores_nan_in_next_batch(fa, case):
    B, Hq, Hkv, N, d, causal, window = case
    q, k, v = prefill_inputs(B, Hq, Hkv, N, d, seed=2000 + N + d)
    for t in (q, k, v):
        t[B - 1] = NAN  # the last sequence is all NaN
    O, L = fa.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window,
                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.attention(q[:B - 1], k[:B - 1], v[:B - 1], causal=causal,
                                    window=window, scale=1.0 / math.sqrt(d))
    _check(O[:B - 1], L[:B - 1], O_ref, L_ref, str(case))


def test_varlen_prefill_ignores_nan_neighbours_and_tail(fa):
    lens = [300, 200, 129, 77]
    Hq, Hkv, d = 4, 2, 128
    extra = 70
    g = torch.Generator("cpu").manual_seed(41)
    T = sum(lens) + extra
    q, k, v = (torch.randn(T, h, d, generator=g).bfloat16() for h in (Hq, Hkv, Hkv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    # sequence 1 is all NaN, and so are the rows after the last sequence
    for t in (q, k, v):
        t[cu[1]:cu[2]] = NAN
        t[cu[-1]:] = NAN
    for causal, window in [(True, -1), (False, -1), (False, 64)]:
        O, L = fa.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.tensor(cu).cuda(),
                                  max(lens), causal=causal, window=window,
                                  out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        for s in (0, 2, 3):
            a, e = int(cu[s]), int(cu[s + 1])
            O_ref, L_ref = oracle.attention(q[None, a:e], k[None, a:e], v[None, a:e],
                                            causal=causal, window=window,
                                            scale=1.0 / math.sqrt(d))
            _check(O[a:e], L[:, a:e], O_ref[0], L_ref[0], f"seq {s} {causal} {window}")


def test_backward_ignores_nan_in_next_batch(fa):
    B, H, N, d = 2, 2, 300, 128
    q, k, v = prefill_inputs(B, H, H, N, d, seed=77)
    dO = torch.randn(B, N, H, d, generator=torch.Generator("cpu").manual_seed(78)).bfloat16()
    for t in (q, k, v, dO):
        t[1] = NAN
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    O, L = fa.attn_fwd(qd, kd, vd, causal=True)
    dq, dk, dv = fa.attn_bwd(qd, kd, vd, O, L, dOd, causal=True)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    rq, rk, rv = oracle.attention_backward(q[:1], k[:1], v[:1], dO[:1], causal=True,
                                           scale=1.0 / math.sqrt(d))
    for got, ref, name in ((dv[:1], rv, "dV"), (dk[:1], rk, "dK"), (dq[:1], rq, "dQ")):
        got = got.double().cpu().numpy()
        assert np.isfinite(got).all(), name
        err = np.abs(got - ref)
        assert err.max() <= 2e-2 * np.abs(ref).max(), name
        assert err.mean() <= 1e-2 * np.abs(ref).mean(), name
