"""The boundary is a C ABI: include/gqa.h must compile as C99 (warnings as
errors), and a C program must link against the built libgqa.so and call it.
Only calls that need no GPU run here (status strings, workspace sizes)."""
import os
import shutil
import subprocess

import pytest

from shared_kv_cache_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include "gqa.h"

int main(void) {
  gqa_dims_t d = {0};
  d.batch = 2;
  d.seq_len = 1;
  d.num_heads = 8;
  d.kv_num_heads = 2;
  d.head_size = 64;
  d.max_seq_len = 128;
  d.dtype = GQA_DTYPE_FP16;
  /* every entry point of the header is declared and linkable */
  gqa_status_t (*fwd)(const gqa_dims_t*, const void*, const void*, const void*, const void*, const void*,
                      void*, void*, const int32_t*, int32_t, const void*, const void*, float, int32_t,
                      const void*, void*, void*, size_t, void*) = gqa_forward;
  gqa_status_t (*fwd_host)(const gqa_dims_t*, const void*, const void*, const void*, const void*, const void*,
                           void*, void*, const int32_t*, int32_t, const void*, const void*, float, int32_t,
                           const void*, void*, void*, size_t, void*) = gqa_forward_host;
  gqa_status_t (*noalloc)(const gqa_dims_t*, const void*, const void*, const void*, const void*, const void*,
                          void*, void*, const int32_t*, int32_t, const void*, const void*, float, int32_t,
                          const void*, void*, void*) = gqa_decode_noalloc;
  gqa_status_t (*check)(void*) = gqa_check_device_status;
  if (!fwd || !fwd_host || !noalloc || !check) return 1;
  /* generic path (head size 64): rotated queries B x S x H x D x 2 bytes */
  printf("%s %zu %zu\n", gqa_status_string(GQA_ERR_KV_OVERFLOW), gqa_workspace_size(&d, 64, 0),
         gqa_workspace_size_host(&d, 64, 0));
  return 0;
}
"""


def test_header_is_c99_and_links(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = build.build()
    src = tmp_path / "use.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "use"
    libdir = os.path.dirname(lib)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(lib), "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60).stdout.split()
    assert out[0] == "GQA_ERR_KV_OVERFLOW"
    assert int(out[1]) == 2 * 1 * 8 * 64 * 2
    # plus query, key, value, seqlens_k and output copies, each rounded to 256
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert int(out[2]) == r(int(out[1])) + 2 * r(2 * 8 * 64 * 2) + 2 * r(2 * 2 * 64 * 2) + r(2 * 4)
