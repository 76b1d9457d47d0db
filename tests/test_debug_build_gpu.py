"""The debug build (libb300attn_debug.so, compiled with -DB300ATTN_DEBUG) on
the GPU.

On valid inputs its results are bit-identical to the release build's and no
device-side check fails.  Two kinds of caller data that the release build
clamps silently are reported by attn_device_status: a decode kv_len entry
above max_kv_len, and cu_seqlens that decrease.  Both stay memory-safe in
either build (the kernels clamp them); the debug build only adds the report.
"""

import contextlib

import pytest
import torch

from exact_transformer_attention_flashattention_b300 import binding as fa
from exact_transformer_attention_flashattention_b300 import build
from exact_transformer_attention_flashattention_b300.inputs import decode_inputs, prefill_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    return {"release": fa._lib, "debug": fa.load_library(build.build(debug=True))}


@contextlib.contextmanager
def using(lib):
    old = fa._lib
    fa._lib = lib
    try:
        yield
    finally:
        fa._lib = old


def _run_all():
    """One call of each path on small valid inputs; every output tensor."""
    out = []
    q, k, v = (t.cuda() for t in prefill_inputs(2, 4, 2, 300, 128, seed=31))
    out += fa.attn_fwd(q, k, v, causal=True)
    q6, k6, v6 = (t.cuda() for t in prefill_inputs(2, 4, 2, 300, 64, seed=32))
    out += fa.attn_fwd(q6, k6, v6, window=64)                  # band kernel
    out += fa.attn_fwd(q6, k6, v6)                             # non-causal, d = 64
    T = 2 * 300
    cu = torch.tensor([0, 300, T], dtype=torch.int32, device="cuda")
    out += fa.attn_fwd_varlen(q.reshape(T, 4, 128), k.reshape(T, 2, 128), v.reshape(T, 2, 128),
                              cu, 300, causal=True)
    O, L = fa.attn_fwd(q, k, v, causal=True)
    dO = torch.randn(q.shape, generator=torch.Generator("cpu").manual_seed(36)).to(q)
    out += fa.attn_bwd(q, k, v, O, L, dO, causal=True)
    qz = fa.attn_fp8_quantize(q, k, v)
    out += list(qz.values())
    out += fa.attn_fwd_fp8(qz, causal=True)
    qd, kc, vc, _ = decode_inputs(2, 8, 2, 700, 128, 33)
    kv_len = torch.tensor([700, 333], dtype=torch.int32, device="cuda")
    out += fa.attn_decode_splitkv(qd.cuda(), kc.cuda(), vc.cuda(), kv_len, 4)
    torch.cuda.synchronize()
    return out


def test_debug_build_matches_release_and_reports_nothing(libs):
    results = {}
    for name, lib in libs.items():
        with using(lib):
            results[name] = _run_all()
            assert fa.device_status() == 0, (name, fa.last_error())
    for a, b in zip(results["release"], results["debug"]):
        assert torch.equal(a, b)


def _decode_with_long_kv_len(lib):
    q, kc, vc, _ = decode_inputs(1, 8, 2, 512, 128, 34)
    kv_len = torch.tensor([512 + 7], dtype=torch.int32, device="cuda")  # above max_kv_len
    with using(lib):
        O, L = fa.attn_decode_splitkv(q.cuda(), kc.cuda(), vc.cuda(), kv_len, 2)
        torch.cuda.synchronize()
        return fa.device_status(), fa.last_error(), O


def test_debug_build_reports_kv_len_above_max(libs):
    rel, _, o_rel = _decode_with_long_kv_len(libs["release"])
    dbg, msg, o_dbg = _decode_with_long_kv_len(libs["debug"])
    assert rel == 0                        # the release build clamps to max_kv_len
    assert dbg == fa.ERR_INVALID and "debug build" in msg and "0x1" in msg
    assert torch.equal(o_rel, o_dbg)       # both computed the clamped decode


def test_debug_build_reports_decreasing_cu_seqlens(libs):
    q, k, v = (t.cuda() for t in prefill_inputs(1, 2, 2, 300, 64, seed=35))
    cu = torch.tensor([0, 200, 150, 300], dtype=torch.int32, device="cuda")  # 200 > 150
    status = {}
    for name, lib in libs.items():
        with using(lib):
            fa.attn_fwd_varlen(q[0], k[0], v[0], cu, 200)
            torch.cuda.synchronize()
            status[name] = (fa.device_status(), fa.last_error())
    assert status["release"][0] == 0
    assert status["debug"][0] == fa.ERR_INVALID and "0x2" in status["debug"][1]
