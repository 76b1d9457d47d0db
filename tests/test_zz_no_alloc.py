"""The allocation-free decode entry point, checked on the GPU.

attn_decode_splitkv_noalloc serves callers that must not allocate device
memory while they run decode: for instance a plugin whose host framework owns
all device memory, or a latency-critical loop that cannot afford cudaMalloc's
device-wide synchronisation.  It keeps its split partials in a 40 MiB array
built into the library instead of a caller workspace.  This file is named so
that pytest collects it last; it must pass on its own in a fresh process and
after the rest of the suite.
"""

import math

import pytest
import torch

from exact_transformer_attention_flashattention_b300.inputs import decode_inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3  # the tolerances of the parity tests
SCRATCH_BYTES = 40 << 20


@pytest.fixture(scope="module")
def fa():
    from exact_transformer_attention_flashattention_b300 import binding
    return binding


def _compare(a, b):
    (Oa, La), (Ob, Lb) = a, b
    dO = (Oa.double() - Ob.double()).abs()
    assert dO.max().item() <= O_MAX and dO.mean().item() <= O_MEAN
    both_ninf = torch.isneginf(La) & torch.isneginf(Lb)
    dL = torch.where(both_ninf, torch.zeros_like(La), (La - Lb).abs())
    assert torch.isfinite(dL).all() and dL.max().item() <= LSE_MAX


def _case(B, Hq, Hkv, L, d, lo, hi, seed):
    q, kc, vc, kv_len = decode_inputs(B, Hq, Hkv, L, d, seed, lo, hi)
    return q.cuda(), kc.cuda(), vc.cuda(), kv_len.cuda()


def test_noalloc_matches_workspace_entry_point_twice(fa):
    """Two calls in a row, of different shapes, through the C ABI; each equals
    attn_decode_splitkv with a caller workspace on the same inputs."""
    cases = [
        ((4, 32, 8, 4096, 128, 100, 4096, 21), 8, torch.float32),
        ((2, 8, 2, 1500, 64, 0, 0, 22), 3, torch.bfloat16),
    ]
    for (B, Hq, Hkv, L, d, lo, hi, seed), S, dt in cases:
        q, kc, vc, kv_len = _case(B, Hq, Hkv, L, d, lo, hi, seed)
        scale = 1.0 / math.sqrt(d)
        ref = fa.attn_decode_splitkv(q, kc, vc, kv_len, S, scale=scale, out_dtype=dt)
        got = fa.attn_decode_splitkv_noalloc(q, kc, vc, kv_len, S, scale=scale, out_dtype=dt)
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        _compare(got, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch(fa):
    B, Hq, d = 1, 64, 128
    S = 2048  # 64 heads x 2048 splits x (128 + 2) floats > 40 MiB
    assert fa.attn_decode_workspace_size(B, Hq, S, d) > SCRATCH_BYTES
    q, kc, vc, kv_len = _case(B, Hq, 8, 4096, d, 0, 0, 23)
    with pytest.raises(fa.B300AttnError) as err:
        fa.attn_decode_splitkv_noalloc(q, kc, vc, kv_len, S)
    assert err.value.status == fa.ERR_WORKSPACE
    assert "built-in scratch" in str(err.value)
