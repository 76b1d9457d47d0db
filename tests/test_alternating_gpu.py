"""GPU parity of the alternating global / local layer stack (ModernBERT
paragraph of the Arabic context-length thread): every layer against the
float64 oracle with its own mask, and each group run as exactly two calls
that equal per-layer calls bit for bit."""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_transformer_attention_flashattention_b300.inputs import layer_stack_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    from exact_transformer_attention_flashattention_b300 import alternating, binding
    return alternating, binding


@pytest.mark.parametrize("L,B,Hq,Hkv,N,d", [(5, 2, 4, 2, 300, 64), (3, 1, 2, 2, 700, 128)])
def test_alternating_stack_matches_oracle(mods, L, B, Hq, Hkv, N, d):
    alt, fa = mods
    q, k, v = layer_stack_inputs(L, B, Hq, Hkv, N, d, seed=L * 100 + N)
    O, LSE = alt.alternating_attention(q.cuda(), k.cuda(), v.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for layer in range(L):
        window = -1 if layer % 3 == 0 else 64
        O_ref, L_ref = oracle.attention(q[layer], k[layer], v[layer], window=window,
                                        scale=1.0 / math.sqrt(d))
        dO = np.abs(O[layer].double().cpu().numpy() - O_ref)
        dL = np.abs(LSE[layer].double().cpu().numpy() - L_ref)
        assert dO.max() <= 1e-2 and dO.mean() <= 1e-3 and dL.max() <= 1e-3, layer
        # the stacked call equals a call on this layer alone
        Ol, Ll = fa.attn_fwd(q[layer].cuda(), k[layer].cuda(), v[layer].cuda(), window=window,
                             out_dtype=torch.float32)
        assert torch.equal(Ol, O[layer]) and torch.equal(Ll, LSE[layer]), layer
