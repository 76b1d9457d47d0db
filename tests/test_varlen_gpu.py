"""GPU parity of the variable-length prefill (sequences packed back to back,
cu_seqlens on the device) against the float64 oracle, sequence by sequence."""

import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def fa():
    from exact_transformer_attention_flashattention_b300 import binding
    return binding


def _inputs(lens, Hq, Hkv, d, seed, extra_rows=0):
    g = torch.Generator("cpu").manual_seed(seed)
    T = sum(lens) + extra_rows
    q = torch.randn(T, Hq, d, generator=g).bfloat16()
    k = torch.randn(T, Hkv, d, generator=g).bfloat16()
    v = torch.randn(T, Hkv, d, generator=g).bfloat16()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return q, k, v, cu


def _check(O, L, O_ref, L_ref, rows):
    O = O.float().cpu().numpy()[rows]
    L = L.cpu().numpy()[:, rows]
    dO = np.abs(O - O_ref[rows])
    dL = np.abs(L - L_ref[:, rows])
    assert np.isfinite(O).all()
    assert dO.max() <= O_MAX and dO.mean() <= O_MEAN, (dO.max(), dO.mean())
    assert dL.max() <= LSE_MAX, dL.max()


CASES = [
    # lens, Hq, Hkv, d, causal, window, fp32
    ([1, 255, 256, 257, 1000, 3], 4, 2, 128, True, -1, False),
    ([700, 5, 300], 2, 2, 64, False, 100, True),
    ([129, 0, 512], 4, 4, 128, False, -1, True),
    ([2000, 17, 1, 640], 8, 2, 64, True, 128, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{len(c[0])}seqs-d{c[3]}-c{int(c[4])}-w{c[5]}")
def test_varlen_matches_oracle(fa, case):
    lens, Hq, Hkv, d, causal, window, fp32 = case
    q, k, v, cu = _inputs(lens, Hq, Hkv, d, seed=sum(lens) + d)
    O, L = fa.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max(lens), causal=causal,
                              window=window, out_dtype=torch.float32 if fp32 else torch.bfloat16)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.attention_varlen(q, k, v, cu.tolist(), causal=causal, window=window,
                                           scale=1.0 / math.sqrt(d))
    _check(O, L, O_ref, L_ref, np.arange(q.shape[0]))


def test_varlen_equal_lengths_equal_dense_bitwise(fa):
    B, N, H, d = 3, 700, 4, 128
    g = torch.Generator("cpu").manual_seed(3)
    q, k, v = (torch.randn(B, N, H, d, generator=g).bfloat16().cuda() for _ in range(3))
    O, L = fa.attn_fwd(q, k, v, causal=True)
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32).cuda()
    Ov, Lv = fa.attn_fwd_varlen(q.view(B * N, H, d), k.view(B * N, H, d), v.view(B * N, H, d),
                                cu, N, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(Ov.view(B, N, H, d), O)
    assert torch.equal(Lv.view(H, B, N).permute(1, 0, 2), L)


def test_varlen_leaves_rows_outside_sequences_untouched(fa):
    lens = [300, 200]
    q, k, v, cu = _inputs(lens, 2, 2, 64, seed=5, extra_rows=70)
    T = q.shape[0]
    out = torch.full((T, 2, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((2, T), 7.0, dtype=torch.float32, device="cuda")
    fa.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), 300, causal=True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(out[500:] == 7.0) and torch.all(lse[:, 500:] == 7.0)
    O_ref, L_ref = oracle.attention_varlen(q, k, v, cu.tolist(), causal=True, scale=0.125)
    _check(out, lse, O_ref, L_ref, np.arange(500))


def test_varlen_many_sequences_sampled(fa):
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 2049, size=64).tolist()
    q, k, v, cu = _inputs(lens, 4, 2, 128, seed=12)
    O, L = fa.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max(lens), causal=True)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert torch.isfinite(O.float()).all()
    for s in [0, 1, 31, 62, 63]:
        a, e = int(cu[s]), int(cu[s + 1])
        O_ref, L_ref = oracle.attention(q[None, a:e], k[None, a:e], v[None, a:e], causal=True,
                                        scale=1.0 / math.sqrt(128))
        dO = np.abs(O[a:e].float().cpu().numpy() - O_ref[0])
        dL = np.abs(L[:, a:e].cpu().numpy() - L_ref[0])
        assert dO.max() <= O_MAX and dO.mean() <= O_MEAN and dL.max() <= LSE_MAX, s
