"""GPU parity of the attention backward (dQ, dK, dV) against the float64 oracle.

The kernels recompute P from the forward's LSE; the comparison uses the
forward's own O and LSE from the library, on the same seeded bf16 inputs.
Tolerance: gradients are sums over up to N terms of bf16-rounded products, so
the bound is scaled by the gradient's own size: max-abs error <= 2e-2 of the
largest |gradient| and mean-abs error <= 1e-2 of its mean |gradient|
(reading: the pages give no backward tolerance; bf16 P and dS carry a relative
rounding of 2^-9 each)."""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_transformer_attention_flashattention_b300 import binding
    return binding


def _rel_close(got, ref, what):
    got = got.double().cpu().numpy()
    err = np.abs(got - ref)
    big = np.abs(ref).max()
    assert np.isfinite(got).all(), what
    assert err.max() <= 2e-2 * big, f"{what}: max err {err.max():.3e} vs max |ref| {big:.3e}"
    assert err.mean() <= 1e-2 * max(np.abs(ref).mean(), 1e-30), \
        f"{what}: mean err {err.mean():.3e} vs mean |ref| {np.abs(ref).mean():.3e}"


CASES = [
    # B, Hq, Hkv, N, d, causal, window
    (1, 2, 2, 256, 64, False, -1),
    (2, 4, 2, 300, 128, True, -1),
    (1, 2, 1, 200, 64, False, 50),
    (1, 4, 4, 640, 128, True, 128),
    (1, 8, 2, 384, 128, False, -1),
    # d = 64 with five key tiles per query tile: the dQ kernel's K/V ring
    # wraps into the stage where Q and dO arrived
    (1, 2, 2, 640, 64, False, -1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_matches_oracle(fa, case):
    B, Hq, Hkv, N, d, causal, window = case
    q, k, v = prefill_inputs(B, Hq, Hkv, N, d, seed=500 + N + d)
    g = torch.Generator("cpu").manual_seed(501 + N)
    dO = torch.randn(B, N, Hq, d, generator=g).bfloat16()
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    O, L = fa.attn_fwd(qd, kd, vd, causal=causal, window=window, scale=scale)
    dq, dk, dv = fa.attn_bwd(qd, kd, vd, O, L, dOd, causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    rq, rk, rv = oracle.attention_backward(q, k, v, dO, causal=causal, window=window,
                                           scale=scale)
    _rel_close(dv, rv, "dV")
    _rel_close(dk, rk, "dK")
    _rel_close(dq, rq, "dQ")


def test_backward_is_deterministic(fa):
    q, k, v = (t.cuda() for t in prefill_inputs(1, 4, 2, 500, 128, seed=9))
    dO = torch.randn_like(q)
    O, L = fa.attn_fwd(q, k, v, causal=True)
    a = fa.attn_bwd(q, k, v, O, L, dO, causal=True)
    b = fa.attn_bwd(q, k, v, O, L, dO, causal=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_backward_full_size_sampled_heads(fa):
    """The benchmarked backward launch (causal, B=4, H=16, N=4096, d=128,
    heaviest-first order) at full size; the oracle recomputes two whole heads
    (with Hq = Hkv a head's dQ, dK, dV depend on that head alone)."""
    from exact_transformer_attention_flashattention_b300.inputs import WORKLOADS
    w = WORKLOADS["causal_prefill_4k"]
    q, k, v = prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
    dO = torch.randn(w.B, w.N, w.Hq, w.d, generator=torch.Generator("cpu").manual_seed(11)
                     ).bfloat16()
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    O, L = fa.attn_fwd(qd, kd, vd, causal=True, scale=w.scale)
    dq, dk, dv = fa.attn_bwd(qd, kd, vd, O, L, dOd, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    for b, h in [(0, 0), (w.B - 1, w.Hq - 1)]:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        rq, rk, rv = oracle.attention_backward(q[sl], k[sl], v[sl], dO[sl], causal=True,
                                               scale=w.scale)
        _rel_close(dv[sl], rv, f"dV b={b} h={h}")
        _rel_close(dk[sl], rk, f"dK b={b} h={h}")
        _rel_close(dq[sl], rq, f"dQ b={b} h={h}")
