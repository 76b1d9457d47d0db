"""CPU tests of the seeded input generators and the algorithmic-work counts the
benchmark divides by: the five workloads have the stated shapes, the draws are
reproducible, ragged lengths stay in range with NaN padding beyond them, and
the flop and byte counts match closed forms."""

import math

import pytest
import torch

from exact_transformer_attention_flashattention_b300.inputs import (WORKLOADS, decode_inputs,
                                                                    decode_kv_bytes,
                                                                    prefill_flops,
                                                                    prefill_inputs,
                                                                    visible_pairs)


def test_workload_shapes():
    w = WORKLOADS
    assert (w["tiny_noncausal"].B, w["tiny_noncausal"].Hq, w["tiny_noncausal"].N,
            w["tiny_noncausal"].d, w["tiny_noncausal"].o_fp32) == (1, 2, 256, 64, True)
    c = w["causal_prefill_4k"]
    assert (c.B, c.Hq, c.Hkv, c.N, c.d, c.causal, c.window) == (4, 16, 16, 4096, 128, True, -1)
    e = w["window_encoder_8k"]
    assert (e.B, e.Hq, e.N, e.d, e.causal, e.window) == (8, 12, 8192, 64, False, 128)
    g = w["gqa_decode_batch32"]
    assert (g.B, g.Hq, g.Hkv, g.d, g.kv_len_lo, g.kv_len_hi) == (32, 32, 8, 128, 1024, 8192)
    assert math.ceil(g.N / g.num_splits) == 512  # chunks of 512 keys
    m = w["decode_1m"]
    assert (m.B, m.Hq, m.Hkv, m.N, m.d, m.num_splits) == (1, 32, 8, 1 << 20, 128, 2048)
    assert m.N // m.num_splits == 512
    assert [x.seed for x in w.values()] == [0, 1, 2, 3, 4]


def test_prefill_draws_are_reproducible_and_bf16():
    a = prefill_inputs(1, 2, 1, 33, 64, seed=7)
    b = prefill_inputs(1, 2, 1, 33, 64, seed=7)
    c = prefill_inputs(1, 2, 1, 33, 64, seed=8)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    assert a[0].shape == (1, 33, 2, 64) and a[1].shape == (1, 33, 1, 64)
    # i.i.d. N(0, 1): sample moments of the first tensor
    q = a[0].float()
    assert abs(q.mean().item()) < 0.1 and abs(q.std().item() - 1.0) < 0.1


def test_ragged_decode_lengths_and_nan_padding():
    q, k, v, kv_len = decode_inputs(6, 4, 2, 300, 64, seed=3, kv_len_lo=10, kv_len_hi=300)
    assert kv_len.dtype == torch.int32 and kv_len.shape == (6,)
    assert int(kv_len.min()) >= 10 and int(kv_len.max()) <= 300
    for b in range(6):
        n = int(kv_len[b])
        assert torch.isfinite(k[b, :n].float()).all() and torch.isfinite(v[b, :n].float()).all()
        assert torch.isnan(k[b, n:].float()).all() and torch.isnan(v[b, n:].float()).all()
    _, _, _, full = decode_inputs(2, 4, 2, 50, 64, seed=3)
    assert full.tolist() == [50, 50]


@pytest.mark.parametrize("N,causal,window,expect", [
    (7, False, -1, 49),
    (7, True, -1, 28),              # N(N+1)/2
    (10, False, 0, 10),             # the diagonal
    (10, False, 2, 10 + 2 * (9 + 8)),
    (10, True, 2, 10 + 9 + 8),
    (10, False, 100, 100),          # wider than the sequence
])
def test_visible_pairs_closed_forms(N, causal, window, expect):
    assert visible_pairs(N, causal, window) == expect


def test_headline_work_counts():
    assert prefill_flops(4, 16, 4096, 128, True, -1) == 4 * 128 * (4096 * 4097 // 2) * 4 * 16
    assert prefill_flops(4, 16, 4096, 128, True, -1) == pytest.approx(2.749e11, rel=1e-3)
    # band |i - j| <= 128 over 8192 rows: 257 per interior row, minus the two edges
    per_head = 8192 * 257 - 2 * (128 * 129 // 2)
    assert visible_pairs(8192, False, 128) == per_head
    assert decode_kv_bytes([1 << 20], 8, 128) == 4294967296


def test_alternating_layer_groups():
    """Layer l is global when l % 3 == 0; each group is one global layer and the
    local layers up to the next global one (two calls per group)."""
    from exact_transformer_attention_flashattention_b300.alternating import layer_groups
    assert layer_groups(6) == [(0, 1, 3), (3, 4, 6)]
    assert layer_groups(5) == [(0, 1, 3), (3, 4, 5)]
    assert layer_groups(1) == [(0, 1, 1)]
    assert layer_groups(4, global_every=1) == [(0, 1, 1), (1, 2, 2), (2, 3, 3), (3, 4, 4)]
    for L in range(1, 12):
        glob = [g for g, _, _ in layer_groups(L)]
        assert glob == [l for l in range(L) if l % 3 == 0]
        covered = sorted(glob + [l for _, a, e in layer_groups(L) for l in range(a, e)])
        assert covered == list(range(L))
