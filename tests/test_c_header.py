"""The public header is plain C: a C99 program includes include/mla_decode.h,
links against libmla_decode.so and calls the entry points that need no GPU
(sizes, status strings, the host-buffer cut, argument rejection).  This is the
boundary a non-Python caller sees; nothing here touches a GPU."""
import os
import shutil
import subprocess

import pytest

from mla_decode_attention_03_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mla_decode.h"

int main(void) {
  int32_t seqlens[6] = {4096, 4096, 0, 64, 65, 4096};
  int32_t bounds[MLA_HOST_MAX_CHUNKS + 1];
  int n = mla_host_chunks(seqlens, 6, 3, bounds);
  printf("chunks %d:", n);
  for (int k = 0; k <= n; ++k) printf(" %d", bounds[k]);
  printf("\n");
  printf("workspace %zu\n", mla_workspace_bytes(128, 1, 128, 76));
  printf("metadata %zu\n", mla_metadata_ints(76));
  printf("scratch %zu\n", mla_host_scratch_bytes(128, 1, 128, 64, 76));
  printf("status %s\n", mla_status_string(MLA_ERR_ALIGNMENT));
  printf("destroy_null %d\n", (int)mla_host_pipeline_destroy(NULL));
  printf("decode_null %d\n", (int)mla_decode_with_kvcache(NULL, 1, 1, 128, 576, NULL, 1, 64, 1, 576, NULL, 1,
                                                          NULL, 512, NULL, 1, NULL, 0.04f, 0, NULL, NULL, NULL,
                                                          0, NULL, NULL));
  printf("static_bytes %zu\n", (size_t)MLA_STATIC_WORKSPACE_BYTES);
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    return build.build()


def test_header_compiles_as_c99_and_links(tmp_path, lib_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_header"
    lib_dir = os.path.dirname(str(lib_path))
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", lib_dir, "-l:libmla_decode.so", f"-Wl,-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    # costs 65, 65, 1, 2, 3, 65 (pages + 1): total 201; shares 1, 2, 1 (in
    # halves of a middle run) give targets 51 and 151; the second bound is
    # pulled back to 5 so that the last run keeps a sequence
    assert out["chunks"] == "3: 0 1 5 6"
    o = (128 + 76) * 128 * 512 * 4  # fp32 partial outputs
    lse = (128 + 76) * 128 * 4
    assert int(out["workspace"]) == o + (lse + 255) // 256 * 256
    assert int(out["metadata"]) == 76 * 8
    assert int(out["scratch"]) > int(out["workspace"])
    assert out["status"].startswith("MLA_ERR_ALIGNMENT")
    assert out["destroy_null"] == "0"
    assert out["decode_null"] == "-1"
    assert int(out["static_bytes"]) == 64 << 20
