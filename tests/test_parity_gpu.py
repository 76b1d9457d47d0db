"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (bf16 inputs, f32 accumulation): O max-abs <= 1e-2 and mean-abs
<= 1e-3, LSE max-abs <= 1e-3, element by element on the same seeded inputs.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_transformer_attention_flashattention_b300.inputs import (WORKLOADS, decode_inputs,
                                                                    prefill_inputs)

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def fa():
    import exact_transformer_attention_flashattention_b300 as pkg
    from exact_transformer_attention_flashattention_b300 import binding
    assert torch.cuda.is_available()
    return binding


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(O, LSE, O_ref, L_ref, what=""):
    O, LSE = _np(O), _np(LSE)
    assert O.shape == O_ref.shape, (O.shape, O_ref.shape)
    assert np.all(np.isfinite(O)), f"{what}: non-finite O"
    dO = np.abs(O - O_ref)
    both_ninf = np.isneginf(LSE) & np.isneginf(L_ref)
    dL = np.where(both_ninf, 0.0, np.abs(LSE - L_ref))
    assert dO.max() <= O_MAX, f"{what}: O max abs err {dO.max():.3e}"
    assert dO.mean() <= O_MEAN, f"{what}: O mean abs err {dO.mean():.3e}"
    assert np.all(np.isfinite(dL)) and dL.max() <= LSE_MAX, f"{what}: LSE max abs err {dL.max()}"


# ------------------------------------------------------------------ prefill
PREFILL_CASES = [
    # B, Hq, Hkv, N, d, causal, window, fp32 out, scale (None = 1/sqrt(d))
    (1, 2, 2, 256, 64, False, -1, True, None),      # the tiny non-causal workload's shape
    (2, 4, 2, 300, 128, True, -1, False, None),     # ragged tail, grouped heads
    (2, 4, 2, 300, 64, False, -1, False, None),
    (1, 2, 1, 777, 128, False, 100, True, None),    # local window
    (1, 2, 2, 1000, 64, True, 200, True, None),     # causal + window
    (1, 1, 1, 1, 128, True, -1, True, None),        # a single token
    (1, 1, 1, 1, 64, False, -1, False, None),
    (1, 2, 2, 129, 128, False, -1, True, None),
    (1, 2, 2, 255, 128, True, -1, True, None),
    (1, 2, 2, 257, 64, True, -1, False, None),
    (1, 2, 2, 300, 128, False, 0, True, None),      # window 0: O_i = v_i
    (1, 2, 2, 300, 64, False, 5000, False, None),   # window wider than the sequence
    (1, 2, 2, 513, 128, False, -1, True, 0.0),      # scale 0: plain mean of V
    (3, 6, 3, 640, 128, True, -1, False, None),     # several tiles and blocks
    # large scores (peaked rows, rescaling exercised); f32 O, because bf16
    # rounding of |O| up to ~4 alone costs 2^-9 * 4 = 0.008 of the 0.01 budget
    (1, 4, 4, 1536, 128, False, -1, True, 0.5),
    # short non-causal windows at d = 64 (the two-stream band schedule)
    (2, 4, 2, 300, 64, False, 50, True, None),
    (1, 2, 2, 129, 64, False, 0, False, None),
    (2, 2, 1, 1000, 64, False, 256, True, None),
    (1, 3, 3, 1025, 64, False, 128, False, None),
    (3, 2, 2, 640, 64, False, 128, True, 0.5),
    (1, 1, 1, 1, 64, False, 64, True, None),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "-".join(map(str, c)))
def test_prefill_matches_oracle(fa, case):
    B, Hq, Hkv, N, d, causal, window, fp32, scale = case
    q, k, v = prefill_inputs(B, Hq, Hkv, N, d, seed=1000 + N + d)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O, L = fa.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, scale=scale,
                       out_dtype=torch.float32 if fp32 else torch.bfloat16)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.attention(q, k, v, causal=causal, window=window, scale=scale)
    assert_close(O, L, O_ref, L_ref, str(case))


def test_tiny_noncausal_workload(fa):
    w = WORKLOADS["tiny_noncausal"]
    q, k, v = prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
    O, L = fa.attn_fwd(q.cuda(), k.cuda(), v.cuda(), out_dtype=torch.float32)
    O_ref, L_ref = oracle.attention(q, k, v, scale=w.scale)
    assert_close(O, L, O_ref, L_ref, w.name)


def _sampled_rows(N, rng, n=40):
    fixed = [0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rnd = rng.integers(0, N, size=n).tolist()
    return sorted(set(r for r in fixed + rnd if 0 <= r < N))


@pytest.mark.parametrize("name", ["causal_prefill_4k", "window_encoder_8k"])
def test_full_size_prefill_sampled_rows(fa, name):
    """The benchmarked launch configuration at full size, checked on sampled
    rows of sampled heads (every row of those heads is also finite)."""
    w = WORKLOADS[name]
    q, k, v = prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
    O, L = fa.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, window=w.window,
                       scale=w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()
    rng = np.random.default_rng(7)
    heads = [(0, 0), (w.B - 1, w.Hq - 1), (int(rng.integers(w.B)), int(rng.integers(w.Hq)))]
    for b, h in heads:
        rows = _sampled_rows(w.N, rng)
        O_ref, L_ref = oracle.attention_rows(q, k, v, b, h, rows, causal=w.causal,
                                             window=w.window, scale=w.scale)
        assert_close(O[b, rows, h], L[b, h, rows], O_ref, L_ref, f"{name} b={b} h={h}")


def test_prefill_is_deterministic(fa):
    q, k, v = (t.cuda() for t in prefill_inputs(2, 4, 4, 1000, 128, seed=5))
    a = fa.attn_fwd(q, k, v, causal=True)
    b = fa.attn_fwd(q, k, v, causal=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("d,causal,window,dtype", [
    (128, True, -1, torch.bfloat16),
    (64, False, 128, torch.bfloat16),   # short window at d = 64: O leaves by TMA store
    (64, False, 128, torch.float32),
], ids=["d128-causal", "d64-window-bf16", "d64-window-f32"])
def test_prefill_writes_only_its_outputs(fa, d, causal, window, dtype):
    """Guard regions around O and LSE keep their sentinel values.  N = 300
    leaves the last 128-row tile 84 rows short; each guard holds a whole tile,
    so that a write past the end would land inside the allocation."""
    B, H, N = 1, 2, 300
    G, GL = 128 * H * d, 4096
    q, k, v = (t.cuda() for t in prefill_inputs(B, H, H, N, d, seed=9))
    o_buf = torch.full((G + B * N * H * d + G,), 7.0, dtype=dtype, device="cuda")
    l_buf = torch.full((GL + B * H * N + GL,), 7.0, dtype=torch.float32, device="cuda")
    O = o_buf[G:G + B * N * H * d].view(B, N, H, d)
    L = l_buf[GL:GL + B * H * N].view(B, H, N)
    fa.attn_fwd(q, k, v, causal=causal, window=window, out=O, lse=L)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for buf, g in ((o_buf, G), (l_buf, GL)):
        assert torch.all(buf[:g] == 7.0) and torch.all(buf[-g:] == 7.0)
    O_ref, L_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal, window=window,
                                    scale=1.0 / math.sqrt(d))
    assert_close(O, L, O_ref, L_ref, f"d={d} window={window} {dtype}")


# ------------------------------------------------------------------ decode
DECODE_CASES = [
    # B, Hq, Hkv, Lmax, d, num_splits, kv_len list (None: drawn), fp32
    (3, 8, 2, 1000, 128, 7, [1000, 1, 65], True),
    (4, 8, 2, 700, 128, 4, [0, 63, 64, 700], False),
    (2, 4, 4, 300, 64, 3, [300, 129], True),          # one query head per kv head
    (2, 8, 4, 520, 64, 2, [520, 7], True),            # two heads per group
    (2, 16, 2, 900, 128, 5, [900, 333], True),        # eight heads per group
    (2, 12, 2, 400, 128, 3, [400, 150], True),        # six heads per group: 3 CTAs of 2
    (1, 4, 1, 4096, 128, 1, [4096], True),            # a single split
    (1, 8, 2, 2048, 64, 64, [2000], False),           # many small splits
    (2, 8, 2, 6400, 128, 100, [6400, 777], True),     # > 64 splits: two-level merge
    (1, 4, 2, 9000, 64, 300, [8999], False),          # two levels, five segments, d=64
]


def _decode_case_inputs(B, Hq, Hkv, L, d, lens, seed):
    q, kc, vc, _ = decode_inputs(B, Hq, Hkv, L, d, seed)
    kv_len = torch.tensor(lens, dtype=torch.int32)
    for b, n in enumerate(lens):
        kc[b, n:] = float("nan")
        vc[b, n:] = float("nan")
    return q, kc, vc, kv_len


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "-".join(map(str, c[:6])))
def test_decode_matches_oracle(fa, case):
    B, Hq, Hkv, L, d, S, lens, fp32 = case
    q, kc, vc, kv_len = _decode_case_inputs(B, Hq, Hkv, L, d, lens, seed=77 + L)
    scale = 1.0 / math.sqrt(d)
    ws = torch.empty(fa.attn_decode_workspace_size(B, Hq, S, d), dtype=torch.uint8,
                     device="cuda")
    O, LSE = fa.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kv_len.cuda(), S,
                                    scale=scale, workspace=ws,
                                    out_dtype=torch.float32 if fp32 else torch.bfloat16)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.decode(q, kc, vc, kv_len, scale=scale)
    assert_close(O, LSE, O_ref, L_ref, str(case))
    # the split partials themselves follow the split definition
    chunk = fa.attn_decode_chunk(L, S)
    m, l, o = fa.split_partials_view(ws, B, Hq, S, d)
    M_ref, Lr, Or = oracle.split_partials(q, kc, vc, kv_len, chunk, S, scale=scale)
    m, l, o = _np(m).reshape(B, Hq, S), _np(l).reshape(B, Hq, S), _np(o).reshape(B, Hq, S, d)
    empty = np.isneginf(M_ref)
    assert np.array_equal(np.isneginf(m), empty)
    assert np.all(l[empty] == 0.0)
    ok = ~empty
    # compare the normalised partials (o/l and m + ln l), which do not depend on
    # which stale maximum a kernel kept
    assert np.max(np.abs(o[ok] / l[ok][:, None] - Or[ok] / Lr[ok][:, None])) <= O_MAX
    assert np.max(np.abs((m[ok] + np.log(l[ok])) - (M_ref[ok] + np.log(Lr[ok])))) <= LSE_MAX


def test_gqa_decode_batch_workload(fa):
    w = WORKLOADS["gqa_decode_batch32"]
    q, kc, vc, kv_len = decode_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.kv_len_lo,
                                      w.kv_len_hi)
    assert fa.attn_decode_chunk(w.N, w.num_splits) == 512
    O, LSE = fa.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kv_len.cuda(), w.num_splits,
                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.decode(q, kc, vc, kv_len, scale=w.scale)
    assert_close(O, LSE, O_ref, L_ref, w.name)


def test_million_token_decode_workload(fa):
    """Full size (4 GiB of K/V, 2048 splits); the oracle checks six heads."""
    w = WORKLOADS["decode_1m"]
    q, kc, vc, kv_len = decode_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
    assert fa.attn_decode_chunk(w.N, w.num_splits) == 512
    O, LSE = fa.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kv_len.cuda(), w.num_splits,
                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert torch.isfinite(O).all() and torch.isfinite(LSE).all()
    heads = [(0, 0), (0, 3), (0, 4), (0, 17), (0, 30), (0, 31)]
    O_ref, L_ref = oracle.decode(q, kc, vc, kv_len, scale=w.scale, heads=heads)
    idx = tuple(np.array(heads).T)
    assert_close(O[idx], LSE[idx], O_ref[idx], L_ref[idx], w.name)


@pytest.mark.parametrize("rows,S,d", [(7, 1, 128), (33, 5, 64), (32, 2048, 128), (5, 300, 64)])
def test_lse_tree_combine_matches_oracle(fa, rows, S, d):
    rng = np.random.default_rng(rows * S + d)
    m = rng.normal(0, 3, size=(rows, S))
    m[rng.random((rows, S)) < 0.2] = -np.inf  # empty splits (identity partials)
    m[0, :] = -np.inf                         # a row with nothing at all
    l = np.where(np.isneginf(m), 0.0, rng.uniform(0.5, 50, size=(rows, S)))
    o = rng.normal(0, 5, size=(rows, S, d)) * (l[..., None] > 0)
    O_ref, L_ref = oracle.combine_rows(m, l, o)
    t = lambda a: torch.tensor(a, dtype=torch.float32, device="cuda")
    # o values of empty partials are never read: poison them
    o_dev = t(o)
    o_dev[t(np.isneginf(m)).bool()] = float("nan")
    O, L = fa.lse_tree_combine(t(m), t(l), o_dev)
    assert_close(O, L, O_ref, L_ref, f"combine {rows}x{S}x{d}")


def test_device_status_clean(fa):
    assert fa.device_status() == 0
