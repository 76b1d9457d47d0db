"""GPU parity of the paged-KV split decode: the cache lives in a shuffled pool
of fixed-size pages addressed through a block table; the result must equal the
float64 oracle on the same keys gathered back into a contiguous cache, and the
contiguous decode of that gathered cache."""

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


@pytest.mark.parametrize("B,Hq,Hkv,d,page,pps,lens,S", [
    (3, 8, 2, 128, 64, 10, [640, 1, 333], 4),
    (4, 32, 8, 128, 256, 8, [2048, 1500, 256, 7], 8),
    (2, 4, 4, 64, 128, 5, [600, 129], 3),
])
def test_paged_decode_matches_oracle(fa, B, Hq, Hkv, d, page, pps, lens, S):
    rng = np.random.default_rng(B * 100 + page)
    g = torch.Generator("cpu").manual_seed(int(page + d))
    P = B * pps + 3  # pool larger than needed; pages handed out in random order
    k_pages = torch.randn(P, page, Hkv, d, generator=g).bfloat16()
    v_pages = torch.randn(P, page, Hkv, d, generator=g).bfloat16()
    q = torch.randn(B, Hq, d, generator=g).bfloat16()
    table = torch.tensor(rng.permutation(P)[:B * pps].reshape(B, pps), dtype=torch.int32)
    kv_len = torch.tensor(lens, dtype=torch.int32)
    # the same keys gathered into a contiguous [B, pps*page, Hkv, d] cache
    kc = k_pages[table.long()].reshape(B, pps * page, Hkv, d)
    vc = v_pages[table.long()].reshape(B, pps * page, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    O, L = fa.attn_decode_splitkv_paged(q.cuda(), k_pages.cuda(), v_pages.cuda(), table.cuda(),
                                        kv_len.cuda(), S, scale=scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.decode(q, kc, vc, kv_len, scale=scale)
    dO = np.abs(O.double().cpu().numpy() - O_ref)
    dL = np.abs(L.double().cpu().numpy() - L_ref)
    assert dO.max() <= O_MAX and dO.mean() <= O_MEAN and dL.max() <= LSE_MAX
    O1, L1 = fa.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kv_len.cuda(), S,
                                    scale=scale, out_dtype=torch.float32)
    assert torch.equal(O, O1) and torch.equal(L, L1)


def test_paged_decode_flags_a_block_table_entry_out_of_range(fa):
    """An entry outside [0, num_pages) is checked by the kernel: never
    dereferenced, its keys left out, and the next status read reports an
    invalid input.  The other sequence is unaffected."""
    B, Hq, Hkv, d, page, pps = 2, 8, 2, 128, 64, 4
    g = torch.Generator("cpu").manual_seed(5)
    P = B * pps
    k_pages = torch.randn(P, page, Hkv, d, generator=g).bfloat16()
    v_pages = torch.randn(P, page, Hkv, d, generator=g).bfloat16()
    q = torch.randn(B, Hq, d, generator=g).bfloat16()
    table = torch.arange(P, dtype=torch.int32).reshape(B, pps)
    table[1, 2] = P + 1000  # sequence 1's third page is out of range
    kv_len = torch.tensor([256, 256], dtype=torch.int32)
    O, L = fa.attn_decode_splitkv_paged(q.cuda(), k_pages.cuda(), v_pages.cuda(), table.cuda(),
                                        kv_len.cuda(), 2, out_dtype=torch.float32)
    assert fa.device_status() == fa.ERR_INVALID
    assert fa.device_status() == 0  # read and cleared
    scale = 1.0 / math.sqrt(d)
    kc = k_pages[table[:1].long()].reshape(1, pps * page, Hkv, d)
    vc = v_pages[table[:1].long()].reshape(1, pps * page, Hkv, d)
    O_ref, L_ref = oracle.decode(q[:1], kc, vc, kv_len[:1], scale=scale)
    assert np.abs(O[:1].double().cpu().numpy() - O_ref).max() <= O_MAX
    assert np.abs(L[:1].double().cpu().numpy() - L_ref).max() <= LSE_MAX
    # sequence 1: its result is that of the keys of its three valid pages
    keep = torch.tensor([0, 1, 3])
    kc1 = k_pages[table[1, keep].long()].reshape(1, 3 * page, Hkv, d)
    vc1 = v_pages[table[1, keep].long()].reshape(1, 3 * page, Hkv, d)
    O1, L1 = oracle.decode(q[1:], kc1, vc1, torch.tensor([3 * page]), scale=scale)
    assert np.abs(O[1:].double().cpu().numpy() - O1).max() <= O_MAX
