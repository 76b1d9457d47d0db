"""GPU parity of the FP8 (e4m3) path against the float64 oracle (oracle.fp8).

* Quantisation (codes, exponents, the transposed padded V) is byte work:
  bit-exact, except that a zero may carry either sign.
* Attention: the oracle is exact attention on the dequantised inputs; the
  kernel also rounds the softmax numerators to e4m3, which the oracle bounds
  (``p_rounding_bound``, the error's standard-deviation scale).  Tolerance:
  every element within 6 bound units plus the f32 accumulation slack, the RMS
  of err / bound at most 1; LSE (from the unrounded numerators) within 1e-3.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8 as f8
from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs

pytestmark = pytest.mark.gpu

LSE_MAX = 1e-3
BOUND_UNITS, RMS_UNITS, F32_SLACK = 6.0, 1.0, 1e-5


@pytest.fixture(scope="module")
def fa():
    from exact_transformer_attention_flashattention_b300 import binding
    assert torch.cuda.is_available()
    return binding


def _spread_inputs(B, Hq, Hkv, N, d, seed):
    """N(0,1) bf16 inputs with every row scaled by exp(U(-3, 3)), so that tiles
    get different exponents."""
    q, k, v = prefill_inputs(B, Hq, Hkv, N, d, seed)
    g = torch.Generator("cpu").manual_seed(seed + 7)
    out = []
    for x in (q, k, v):
        s = torch.exp(torch.rand(x.shape[:3] + (1,), generator=g) * 6 - 3)
        out.append((x.float() * s).bfloat16())
    return out


def _codes_equal(got, want):
    """Byte equality, a zero of either sign counting as equal."""
    got = np.asarray(got, dtype=np.uint8)
    want = np.asarray(want, dtype=np.uint8)
    zero = ((got & 0x7F) == 0) & ((want & 0x7F) == 0)
    return np.all((got == want) | zero)


QUANT_CASES = [
    # B, Hq, Hkv, N, spread
    (2, 4, 2, 300, True),    # ragged last tile, grouped heads
    (1, 2, 1, 1, False),     # a single token
    (1, 8, 2, 1000, True),   # N not a multiple of 16: padded V keys
    (1, 2, 2, 128, False),   # exactly one tile
]


@pytest.mark.parametrize("case", QUANT_CASES, ids=lambda c: "-".join(map(str, c)))
def test_quantize_bit_exact(fa, case):
    B, Hq, Hkv, N, spread = case
    d = 128
    q, k, v = (_spread_inputs if spread else prefill_inputs)(B, Hq, Hkv, N, d, seed=N + Hq)
    qz = fa.attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    ref = f8.quantize_inputs(q, k, v)
    for name in ("q_exp", "k_exp", "v_exp"):
        assert np.array_equal(qz[name].cpu().numpy(), ref[name]), name
    for name in ("q8", "k8", "v8t"):
        got = qz[name].cpu().numpy()
        assert got.shape == ref[name].shape, (name, got.shape, ref[name].shape)
        assert _codes_equal(got, ref[name]), f"{name}: {np.sum(got != ref[name])} codes differ"
    assert np.all(qz["v8t"].cpu().numpy()[..., N:] == 0), "padding keys must be zero"


def _check_attention(O, L, qd, kd, vd, causal, window, scale, rows=None, bf16_out=False):
    """O [B, R, Hq, d] and L [B, Hq, R] from the GPU for query rows `rows`
    (all when None) against the oracle on the dequantised inputs."""
    B, N, Hq, d = qd.shape
    rows = np.arange(N) if rows is None else np.asarray(rows)
    O_ref = np.zeros((B, len(rows), Hq, d))
    L_ref = np.zeros((B, Hq, len(rows)))
    for b in range(B):
        for h in range(Hq):
            O_ref[b, :, h], L_ref[b, h] = oracle.attention_rows(qd, kd, vd, b, h, rows, causal=causal,
                                                                window=window, scale=scale)
    bound = f8.p_rounding_bound(qd, kd, vd, causal=causal, window=window, scale=scale, rows=rows)
    O = O.double().cpu().numpy()
    L = L.double().cpu().numpy()
    assert np.all(np.isfinite(O))
    err = np.abs(O - O_ref)
    slack = F32_SLACK + (2.0 ** -8 * np.abs(O_ref) if bf16_out else 0.0)
    ratio = np.maximum(err - slack, 0.0) / np.maximum(bound, 1e-30)
    assert ratio.max() <= BOUND_UNITS, f"max err / bound {ratio.max():.2f}"
    rms = float(np.sqrt(np.mean((err / np.maximum(bound, 1e-30)) ** 2)))
    assert rms <= RMS_UNITS, f"RMS err / bound {rms:.2f}"
    both = np.isneginf(L) & np.isneginf(L_ref)
    dL = np.where(both, 0.0, np.abs(L - L_ref))
    assert np.all(np.isfinite(dL)) and dL.max() <= LSE_MAX, dL.max()


ATTN_CASES = [
    # B, Hq, Hkv, N, causal, window, spread, bf16 out
    (1, 4, 2, 700, True, -1, False, False),
    (2, 2, 2, 300, False, -1, True, False),
    (1, 2, 1, 777, False, 100, False, True),
    (1, 2, 2, 1000, True, 200, True, False),
    (1, 1, 1, 1, True, -1, False, False),      # a single token: O = v exactly up to rounding
    (1, 2, 2, 257, False, -1, False, True),
    (1, 2, 2, 300, False, 0, False, False),    # window 0: O_i = v_i (P = 1 is exact in e4m3)
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: "-".join(map(str, c)))
def test_fwd_fp8_matches_oracle(fa, case):
    B, Hq, Hkv, N, causal, window, spread, bf16_out = case
    d = 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = (_spread_inputs if spread else prefill_inputs)(B, Hq, Hkv, N, d, seed=3 * N + Hq)
    qz = fa.attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
    O, L = fa.attn_fwd_fp8(qz, causal=causal, window=window, scale=scale,
                           out_dtype=torch.bfloat16 if bf16_out else torch.float32)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    ref = f8.quantize_inputs(q, k, v)
    _check_attention(O, L, ref["q"], ref["k"], ref["v"], causal, window, scale, bf16_out=bf16_out)


def test_fwd_fp8_rescale_every_tile(fa):
    """Key rows of tile t scaled by 1 + 4t and scale 0.5: each key tile raises
    most rows' maximum by far more than the 2^8 rescale threshold, so the
    running O is rescaled on every tile (before the first half of P·V of that
    tile may add into it)."""
    B, H, N, d = 1, 2, 640, 128
    q, k, v = prefill_inputs(B, H, H, N, d, seed=21)
    ramp = (1.0 + 4.0 * (torch.arange(N) // 128)).view(1, N, 1, 1)
    k = (k.float() * ramp).bfloat16()
    for causal in (False, True):
        qz = fa.attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
        O, L = fa.attn_fwd_fp8(qz, causal=causal, scale=0.5, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        ref = f8.quantize_inputs(q, k, v)
        _check_attention(O, L, ref["q"], ref["k"], ref["v"], causal, -1, 0.5, bf16_out=False)


def test_fp8_full_size_sampled(fa):
    """The causal N=4096, d=128 workload shape (B=4, 16 heads) in the launch
    configuration the benchmark times: quantisation bit-exact in full, attention
    on sampled rows (first, tile edges, last) of every head."""
    B, H, N, d = 4, 16, 4096, 128
    q, k, v = prefill_inputs(B, H, H, N, d, seed=1)
    qz = fa.attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
    O, L = fa.attn_fwd_fp8(qz, causal=True, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    ref = f8.quantize_inputs(q, k, v)
    for name in ("q_exp", "k_exp", "v_exp"):
        assert np.array_equal(qz[name].cpu().numpy(), ref[name]), name
    for name in ("q8", "k8", "v8t"):
        assert _codes_equal(qz[name].cpu().numpy(), ref[name]), name
    rows = np.array([0, 127, 128, 255, 256, 2047, 2048, 4095])
    _check_attention(O[:, rows], L[:, :, rows], ref["q"], ref["k"], ref["v"], True, -1,
                     1.0 / math.sqrt(d), rows=rows, bf16_out=True)


def test_fp8_repeatable(fa):
    q, k, v = prefill_inputs(1, 4, 2, 1000, 128, seed=9)
    qz1 = fa.attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
    O1, L1 = fa.attn_fwd_fp8(qz1, causal=True)
    qz2 = fa.attn_fp8_quantize(q.cuda(), k.cuda(), v.cuda())
    O2, L2 = fa.attn_fwd_fp8(qz2, causal=True)
    torch.cuda.synchronize()
    for name in qz1:
        assert torch.equal(qz1[name], qz2[name]), name
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
