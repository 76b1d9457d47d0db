"""CPU tests of the debug build: libb300attn_debug.so is the same library
compiled with -DB300ATTN_DEBUG.  It exports the same C ABI as the release
build, and its host-side validation is the same."""

import ctypes
import os

import pytest

from exact_transformer_attention_flashattention_b300 import build

from .test_abi_cpu import header_functions


def test_debug_command_adds_the_flag_and_only_it():
    rel = build.nvcc_command("out.so")
    dbg = build.nvcc_command("out.so", debug=True)
    assert "-DB300ATTN_DEBUG" in dbg and "-DB300ATTN_DEBUG" not in rel
    assert [a for a in dbg if a != "-DB300ATTN_DEBUG"] == rel


@pytest.fixture(scope="module")
def debug_lib():
    path = build.build(debug=True)
    assert path == build.LIB_DEBUG and os.path.exists(path)
    return ctypes.CDLL(path)


def test_debug_library_exports_every_declared_symbol(debug_lib):
    for name in header_functions():
        assert hasattr(debug_lib, name), f"{name} missing from the debug library"


def test_debug_library_validates_on_the_host(debug_lib):
    from exact_transformer_attention_flashattention_b300 import binding
    for name, (res, args) in binding.SIGNATURES.items():
        fn = getattr(debug_lib, name)
        fn.restype, fn.argtypes = res, args
    fake = 0x10000
    # negative batch, then an unsupported head dimension: rejected before any GPU work
    assert debug_lib.attn_fwd(fake, fake, fake, fake, fake, -1, 2, 2, 16, 64, 0, -1, 0.125,
                              None, 0) == binding.ERR_INVALID
    assert debug_lib.attn_fwd(fake, fake, fake, fake, fake, 1, 2, 2, 16, 96, 0, -1, 0.125,
                              None, 0) == binding.ERR_UNSUPPORTED
