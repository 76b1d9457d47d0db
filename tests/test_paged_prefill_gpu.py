"""GPU parity of the paged-KV prefill: K and V live in a shuffled pool of
fixed-size pages addressed through a block table.  The result must match the
float64 oracle on the keys gathered back into contiguous K and V, and equal
bit for bit the dense prefill of that gathered K and V."""

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


def _pool(B, N, Hkv, d, page, seed, extra_pages=3):
    """A shuffled pool with every sequence's pages; table entries past a
    sequence's N keys are -1 (never read)."""
    rng = np.random.default_rng(seed)
    g = torch.Generator("cpu").manual_seed(seed)
    pps = (N + page - 1) // page + 1  # one spare table column per sequence
    P = B * pps + extra_pages
    k_pages = torch.randn(P, page, Hkv, d, generator=g).bfloat16()
    v_pages = torch.randn(P, page, Hkv, d, generator=g).bfloat16()
    table = torch.tensor(rng.permutation(P)[:B * pps].reshape(B, pps), dtype=torch.int32)
    used = (N + page - 1) // page
    table[:, used:] = -1
    kc = k_pages[table[:, :used].long()].reshape(B, used * page, Hkv, d)[:, :N].contiguous()
    vc = v_pages[table[:, :used].long()].reshape(B, used * page, Hkv, d)[:, :N].contiguous()
    return k_pages, v_pages, table, kc, vc


CASES = [
    # B, Hq, Hkv, N, d, page, causal, window, fp32
    (3, 4, 2, 300, 128, 64, True, -1, False),
    (2, 2, 2, 700, 64, 128, False, 100, True),
    (2, 8, 2, 513, 128, 256, False, -1, True),
    (1, 2, 1, 1000, 64, 192, True, 200, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_paged_prefill_matches_oracle_and_dense(fa, case):
    B, Hq, Hkv, N, d, page, causal, window, fp32 = case
    g = torch.Generator("cpu").manual_seed(N + d)
    q = torch.randn(B, N, Hq, d, generator=g).bfloat16()
    k_pages, v_pages, table, kc, vc = _pool(B, N, Hkv, d, page, seed=N + page)
    dt = torch.float32 if fp32 else torch.bfloat16
    O, L = fa.attn_fwd_paged(q.cuda(), k_pages.cuda(), v_pages.cuda(), table.cuda(),
                             causal=causal, window=window, out_dtype=dt)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.attention(q, kc, vc, causal=causal, window=window,
                                    scale=1.0 / math.sqrt(d))
    dO = np.abs(O.double().cpu().numpy() - O_ref)
    dL = np.abs(L.double().cpu().numpy() - L_ref)
    assert np.isfinite(dO).all()
    assert dO.max() <= O_MAX and dO.mean() <= O_MEAN and dL.max() <= LSE_MAX
    Od, Ld = fa.attn_fwd(q.cuda(), kc.cuda(), vc.cuda(), causal=causal, window=window,
                         out_dtype=dt)
    assert torch.equal(O, Od) and torch.equal(L, Ld)


def test_paged_prefill_flags_a_block_table_entry_out_of_range(fa):
    B, H, N, d, page = 2, 2, 256, 128, 64
    g = torch.Generator("cpu").manual_seed(9)
    q = torch.randn(B, N, H, d, generator=g).bfloat16()
    k_pages, v_pages, table, kc, vc = _pool(B, N, H, d, page, seed=9)
    table[1, 1] = k_pages.shape[0] + 5  # a page of sequence 1 out of range
    O, L = fa.attn_fwd_paged(q.cuda(), k_pages.cuda(), v_pages.cuda(), table.cuda(),
                             causal=True, out_dtype=torch.float32)
    assert fa.device_status() == fa.ERR_INVALID
    assert fa.device_status() == 0
    # sequence 0 is untouched by the bad entry
    O_ref, L_ref = oracle.attention(q[:1], kc[:1], vc[:1], causal=True, scale=1.0 / math.sqrt(d))
    assert np.abs(O[:1].double().cpu().numpy() - O_ref).max() <= O_MAX
    assert np.abs(L[:1].double().cpu().numpy() - L_ref).max() <= LSE_MAX
