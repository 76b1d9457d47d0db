"""The boundary is a plain C ABI: a C program (gcc, no CUDA headers, no C++)
includes include/b300attn.h, links libb300attn.so and calls it.  Only calls
that need no GPU are made: the version, sizing helpers, and argument errors
that the library rejects on the host before touching the device."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include "b300attn.h"

int main(void) {
  int fails = 0;
  if (attn_version() < 100) { puts("version"); ++fails; }
  /* sizing helpers */
  if (attn_decode_chunk(1048576, 2048) != 512) { puts("chunk"); ++fails; }
  if (attn_fp8_padded_len(1000) != 1008) { puts("fp8 pad"); ++fails; }
  if (attn_bwd_workspace_size(2, 4, 300) != 9728) { puts("bwd ws"); ++fails; }
  /* host-side argument errors: nothing reaches the device */
  void* p = (void*)0x10000;
  if (attn_fwd(p, p, p, p, (float*)p, -1, 2, 2, 16, 64, 0, -1, 0.125f, 0, B300ATTN_BF16)
      != B300ATTN_ERR_INVALID) { puts("negative B"); ++fails; }
  if (attn_fwd(p, p, p, p, (float*)p, 1, 2, 2, 16, 80, 0, -1, 0.125f, 0, B300ATTN_BF16)
      != B300ATTN_ERR_UNSUPPORTED) { puts("d=80"); ++fails; }
  if (attn_last_error()[0] == '\0') { puts("no message"); ++fails; }
  if (lse_tree_combine((const float*)p, (const float*)p, (const float*)p, p, (float*)p, 4, 0,
                       128, 0, B300ATTN_F32) == B300ATTN_OK) { puts("zero splits"); ++fails; }
  /* nothing to compute: OK with NULL pointers */
  if (attn_fwd(0, 0, 0, 0, 0, 0, 2, 2, 16, 64, 0, -1, 0.125f, 0, B300ATTN_BF16) != B300ATTN_OK) {
    puts("empty batch"); ++fails;
  }
  printf("%d failures\n", fails);
  return fails;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    from exact_transformer_attention_flashattention_b300 import build
    build.build()
    return os.path.join(ROOT, "exact_transformer_attention_flashattention_b300")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_plain_c_program_links_and_calls_the_library(lib_dir, tmp_path):
    src = tmp_path / "use_abi.c"
    exe = tmp_path / "use_abi"
    src.write_text(C_PROGRAM)
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
           "-L", lib_dir, "-lb300attn", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failures" in r.stdout
