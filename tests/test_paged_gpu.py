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
