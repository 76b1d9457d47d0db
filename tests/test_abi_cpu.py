"""CPU tests of the C ABI: the library loads, exports every function the header
declares, and rejects bad arguments on the host before touching the GPU."""

import ctypes
import os
import re

import pytest

from exact_transformer_attention_flashattention_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "b300attn.h")

INVALID, UNSUPPORTED, WORKSPACE = -1, -2, -3
FAKE = 0x10000  # a 16-byte aligned non-NULL value; validation fails before any use


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text,
                                 flags=re.M)))


@pytest.fixture(scope="module")
def binding():
    build.build()
    from exact_transformer_attention_flashattention_b300 import binding as b
    return b


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("attn_fwd", "attn_decode_splitkv", "lse_tree_combine"):
        assert required in names


def test_library_exports_every_declared_symbol(binding):
    lib = ctypes.CDLL(binding.LIB_PATH)
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in the header but not exported"
        assert name in binding.SIGNATURES, f"{name} has no ctypes signature in the binding"


def test_version(binding):
    assert binding.lib().attn_version() >= 100


def _fwd(lib, B=1, Hq=2, Hkv=2, N=16, d=64, causal=0, window=-1, scale=0.125, o_dtype=0,
         ptr=FAKE, misalign=0):
    p = ptr + misalign if ptr else None
    return lib.attn_fwd(p, ptr, ptr, ptr, ptr, B, Hq, Hkv, N, d, causal, window, scale, None,
                        o_dtype)


def test_prefill_validation(binding):
    lib = binding.lib()
    assert _fwd(lib, B=-1) == INVALID
    assert _fwd(lib, N=-5) == INVALID
    assert _fwd(lib, Hq=3, Hkv=2) == INVALID
    assert _fwd(lib, Hkv=0) == INVALID
    assert _fwd(lib, d=96) == UNSUPPORTED
    assert "d=96" in binding.last_error()
    assert _fwd(lib, d=256) == UNSUPPORTED
    assert _fwd(lib, ptr=0) == INVALID
    assert _fwd(lib, misalign=8) == INVALID
    assert _fwd(lib, causal=2) == INVALID
    assert _fwd(lib, scale=float("nan")) == INVALID
    assert _fwd(lib, scale=float("inf")) == INVALID
    assert _fwd(lib, scale=-1.0) == INVALID
    assert _fwd(lib, o_dtype=7) == INVALID


def test_prefill_empty_is_a_noop(binding):
    lib = binding.lib()
    assert _fwd(lib, B=0, ptr=0) == 0
    assert _fwd(lib, N=0, ptr=0) == 0
    assert _fwd(lib, Hq=0, ptr=0) == 0


def test_decode_chunk_and_workspace(binding):
    assert binding.attn_decode_chunk(1 << 20, 2048) == 512
    assert binding.attn_decode_chunk(8192, 16) == 512
    assert binding.attn_decode_chunk(1000, 3) == 384  # ceil(1000/3)=334 -> multiple of 64
    assert binding.attn_decode_chunk(1, 1) == 64
    with pytest.raises(binding.B300AttnError):
        binding.attn_decode_chunk(0, 4)
    rows = 32 * 32 * 16
    assert binding.attn_decode_workspace_size(32, 32, 16, 128) == 2 * rows * 4 + rows * 128 * 4
    # 15 rows: m and l take 60 B each, padded to 256; o takes 15*64*4 = 3840 B
    assert binding.attn_decode_workspace_size(1, 3, 5, 64) == 2 * 256 + 3840
    assert binding.attn_decode_workspace_size(1, 1, 0, 64) == 0


def _dec(lib, B=2, Hq=4, Hkv=2, L=100, d=128, S=4, ws=FAKE, ws_bytes=1 << 30, ptr=FAKE,
         scale=0.1, o_dtype=0):
    return lib.attn_decode_splitkv(ptr, ptr, ptr, ptr, ptr, ptr, B, Hq, Hkv, L, d, scale, S, ws,
                                   ws_bytes, None, o_dtype)


def test_decode_validation(binding):
    lib = binding.lib()
    assert _dec(lib, B=-1) == INVALID
    assert _dec(lib, Hq=3) == INVALID
    assert _dec(lib, d=80) == UNSUPPORTED
    assert _dec(lib, S=0) == INVALID
    assert _dec(lib, S=70000) == INVALID
    assert _dec(lib, L=0) == INVALID
    assert _dec(lib, ptr=0) == INVALID
    assert _dec(lib, ws=0) == WORKSPACE
    assert _dec(lib, ws_bytes=16) == WORKSPACE
    assert "workspace" in binding.last_error()
    assert _dec(lib, ws=FAKE + 16) == INVALID  # not 256-byte aligned
    assert _dec(lib, scale=float("nan")) == INVALID
    assert _dec(lib, B=0, ptr=0, ws=0) == 0


def test_combine_validation(binding):
    lib = binding.lib()
    assert lib.lse_tree_combine(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 128, None, 0) == INVALID
    assert lib.lse_tree_combine(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 0, 128, None, 0) == INVALID
    assert lib.lse_tree_combine(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 32, None, 0) == UNSUPPORTED
    assert lib.lse_tree_combine(None, FAKE, FAKE, FAKE, FAKE, 4, 4, 64, None, 0) == INVALID
    assert lib.lse_tree_combine(None, None, None, None, None, 0, 4, 64, None, 0) == 0


def test_varlen_validation(binding):
    lib = binding.lib()

    def call(S=2, T=100, maxlen=60, Hq=2, Hkv=2, d=64, ptr=FAKE, cu=FAKE, causal=0):
        return lib.attn_fwd_varlen(ptr, ptr, ptr, ptr, ptr, cu, S, T, maxlen, Hq, Hkv, d, causal,
                                   -1, 0.125, None, 0)
    assert call(S=-1) == INVALID
    assert call(S=4097) == UNSUPPORTED
    assert "4096" in binding.last_error()
    assert call(d=96) == UNSUPPORTED
    assert call(Hq=3) == INVALID
    assert call(cu=0) == INVALID
    assert call(cu=FAKE + 2) == INVALID  # not 4-byte aligned
    assert call(ptr=FAKE + 8) == INVALID
    assert call(causal=3) == INVALID
    assert call(S=0, ptr=0, cu=0) == 0
    assert call(T=0, ptr=0, cu=0) == 0


def test_backward_validation(binding):
    lib = binding.lib()
    assert binding.lib().attn_bwd_workspace_size(2, 4, 300) == (2 * 4 * 300 * 4 + 255) // 256 * 256

    def call(B=1, Hq=2, Hkv=2, N=16, d=64, ptr=FAKE, ws=FAKE, ws_bytes=1 << 20, causal=0,
             o_dtype=0):
        return lib.attn_bwd(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ws, ws_bytes, B, Hq, Hkv,
                            N, d, causal, -1, 0.125, None, o_dtype)
    assert call(B=-1) == INVALID
    assert call(Hq=3) == INVALID
    assert call(d=80) == UNSUPPORTED
    assert call(ptr=0) == INVALID
    assert call(ptr=FAKE + 4) == INVALID
    assert call(ws=0) == WORKSPACE
    assert call(ws_bytes=8) == WORKSPACE
    assert call(ws=FAKE + 16) == INVALID
    assert call(causal=5) == INVALID
    assert call(o_dtype=3) == INVALID
    assert call(N=0, ptr=0, ws=0) == 0


def test_bench_and_tests_call_only_existing_binding_functions(binding):
    """Every `fa.<name>` used by bench.py, the smoke check and the tests exists."""
    import re
    files = [os.path.join(ROOT, "bench.py"), os.path.join(ROOT, "__graft_entry__.py")]
    files += [os.path.join(ROOT, "tests", f) for f in os.listdir(os.path.join(ROOT, "tests"))
              if f.endswith(".py")]
    for f in files:
        for name in set(re.findall(r"\bfa\.(\w+)", open(f).read())):
            assert hasattr(binding, name), f"{os.path.basename(f)} uses missing fa.{name}"


def test_paged_decode_validation(binding):
    lib = binding.lib()

    def call(B=2, page=64, P=8, pps=4, ptr=FAKE, table=FAKE, ws=FAKE, S=2, d=128):
        return lib.attn_decode_splitkv_paged(ptr, ptr, ptr, table, ptr, ptr, ptr, B, 4, 2, page,
                                             P, pps, d, 0.1, S, ws, 1 << 30, None, 0)
    assert call(page=100) == UNSUPPORTED
    assert call(page=0) == UNSUPPORTED
    assert call(P=0) == INVALID
    assert call(pps=0) == INVALID
    assert call(table=0) == INVALID
    assert call(table=FAKE + 2) == INVALID
    assert call(page=-64) == INVALID
    assert call(ws=0) == WORKSPACE
    assert call(d=96) == UNSUPPORTED
    assert call(B=0, ptr=0, table=0, ws=0) == 0


def test_fp8_validation(binding):
    lib = binding.lib()
    assert lib.attn_fp8_padded_len(1000) == 1008 and lib.attn_fp8_padded_len(4096) == 4096
    assert lib.attn_fp8_padded_len(0) == 0
    assert lib.attn_fp8_workspace_size(2, 4, 300) == 256  # 2*4*3 floats, rounded up to 256
    assert lib.attn_fp8_workspace_size(4, 16, 4096) == 4 * 16 * 32 * 4

    def quant(B=1, Hq=2, Hkv=2, N=16, d=128, ptr=FAKE, ws=FAKE, ws_bytes=1 << 20):
        return lib.attn_fp8_quantize(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, B, Hq, Hkv, N,
                                     d, ws, ws_bytes, None)
    assert quant(B=-1) == INVALID
    assert quant(Hq=3) == INVALID
    assert quant(d=64) == UNSUPPORTED
    assert quant(ptr=0) == INVALID
    assert quant(ptr=FAKE + 8) == INVALID
    assert quant(ws=0) == WORKSPACE
    assert quant(ws_bytes=16) == WORKSPACE
    assert quant(ws=FAKE + 16) == INVALID
    assert quant(N=0, ptr=0, ws=0) == 0

    def fwd(B=1, Hq=2, Hkv=2, N=16, d=128, ptr=FAKE, causal=0, scale=0.1, o_dtype=0):
        return lib.attn_fwd_fp8(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, B, Hq, Hkv, N, d, causal,
                                -1, scale, None, o_dtype)
    assert fwd(B=-1) == INVALID
    assert fwd(Hq=3) == INVALID
    assert fwd(d=64) == UNSUPPORTED
    assert fwd(ptr=0) == INVALID
    assert fwd(ptr=FAKE + 4) == INVALID
    assert fwd(causal=2) == INVALID
    assert fwd(scale=float("nan")) == INVALID
    assert fwd(o_dtype=7) == INVALID
    assert fwd(B=0, ptr=0) == 0


def test_binding_rejects_host_and_mistyped_tensors(binding):
    """The Python wrappers refuse host tensors and wrong dtypes before any call."""
    import torch
    q = torch.zeros(1, 16, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.attn_fwd(q, q, q)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.attn_fp8_quantize(q, q, q)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.attn_fwd_fp8({"q8": q.to(torch.uint8), "k8": q.to(torch.uint8),
                              "v8t": q.to(torch.uint8), "q_exp": None, "k_exp": None,
                              "v_exp": None})
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.attn_bwd(q, q, q, q, torch.zeros(1, 2, 16), q)
