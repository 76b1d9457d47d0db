"""Cross-device tree decoding emulated on one GPU: every shard of the KV
sequence axis is decoded by the library's split-KV kernels as if on its own
device, and the per-shard (O_r, LSE_r) are merged by the logsumexp tree kernel
("Tree Attention" page, abstract).  Checked against the float64 oracle and
against the single-device decode, with the parity tolerances."""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_transformer_attention_flashattention_b300.inputs import decode_inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3


def _close(O, L, O_ref, L_ref):
    O = O.double().cpu().numpy()
    L = L.double().cpu().numpy()
    dO = np.abs(O - O_ref)
    both = np.isneginf(L) & np.isneginf(L_ref)
    dL = np.where(both, 0.0, np.abs(L - L_ref))
    assert dO.max() <= O_MAX and dO.mean() <= O_MEAN, (dO.max(), dO.mean())
    assert np.isfinite(dL).all() and dL.max() <= LSE_MAX, dL.max()


@pytest.mark.parametrize("world,B,L,lo,hi", [(2, 4, 3000, 1, 3000), (4, 8, 2048, 100, 2048),
                                             (7, 2, 5000, 4000, 5000)])
def test_tree_decode_matches_oracle_and_single_device(world, B, L, lo, hi):
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300 import tree_decode as td
    Hq, Hkv, d = 32, 8, 128
    q, kc, vc, kv_len = decode_inputs(B, Hq, Hkv, L, d, seed=50 + world, kv_len_lo=lo,
                                      kv_len_hi=hi)
    qd, kd, vd, lend = q.cuda(), kc.cuda(), vc.cuda(), kv_len.cuda()
    shards = []
    for a, b in td.shard_bounds(L, world):
        k_s, v_s = td.shard_cache(kd, vd, a, b)
        shards.append((k_s, v_s, td.shard_kv_len(lend, a, b)))
    O, LSE = td.tree_decode_emulated(qd, shards, num_splits=4, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.decode(q, kc, vc, kv_len, scale=1.0 / math.sqrt(d))
    _close(O, LSE, O_ref, L_ref)
    O1, L1 = fa.attn_decode_splitkv(qd, kd, vd, lend, 8, out_dtype=torch.float32)
    assert (O - O1).abs().max().item() <= O_MAX
    assert (LSE - L1).abs().max().item() <= LSE_MAX
