"""The boundary is plain C: a C99 client that includes include/nvfp4moe.h
compiles with warnings as errors, links against libnvfp4moe.so and gets the
same host-side answers as the Python binding (sizes, layout, argument
errors) without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "nvfp4moe.h"

int main(void) {
  nvfp4_moe_layout L;
  int rc;
  static float logits[16];
  printf("version %d\n", nvfp4_version());
  printf("ws %zu\n", nvfp4_moe_workspace_size(8192, 4096, 2048, 48, 6));
  rc = nvfp4_moe_workspace_layout(8192, 4096, 2048, 48, 6, &L);
  printf("layout %d %lld %zu %zu\n", rc, (long long)L.capacity, L.a1, L.total);
  /* top_k above E: refused on the host, with a reason (the logits pointer is
     never dereferenced on the host) */
  rc = nvfp4_moe_forward(NULL, logits, 4, 256, 128, 2, 3, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                         10.0f, 10.0f, NULL, 0, NULL, NULL);
  printf("bad_topk %d %s | %s\n", rc, nvfp4_status_string(rc), nvfp4_last_error());
  /* K not a multiple of 64 */
  rc = nvfp4_quantize(NULL, 128, 100, 100, 0, 1, NULL, NULL, NULL, 0, NULL, NULL, 128, NULL);
  printf("bad_k %d\n", rc);
  /* T = 0 is a valid no-op that touches nothing */
  rc = nvfp4_moe_forward(NULL, NULL, 0, 256, 128, 4, 2, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                         10.0f, 10.0f, NULL, 0, NULL, NULL);
  printf("empty %d\n", rc);
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    from nvfp4_mixture_experts_expert_gb300 import _build
    _build.build()
    return os.path.dirname(_build.LIB)


def test_c99_client_compiles_links_and_runs_without_a_gpu(tmp_path, lib_dir):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(CLIENT)
    exe = tmp_path / "client"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", lib_dir, "-lnvfp4moe", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    res = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60)
    out = dict(line.split(" ", 1) for line in res.stdout.strip().splitlines())

    from nvfp4_mixture_experts_expert_gb300 import binding as B
    assert int(out["version"]) == B.nvfp4_version()
    assert int(out["ws"]) == B.nvfp4_moe_workspace_size(8192, 4096, 2048, 48, 6)
    rc, cap, a1, total = out["layout"].split()
    lay = B.nvfp4_moe_workspace_layout(8192, 4096, 2048, 48, 6)
    assert int(rc) == 0 and int(a1) == lay["a1"] and int(total) == lay["total"]
    assert int(cap) % 128 == 0 and int(cap) >= 8192 * 6
    code, rest = out["bad_topk"].split(" ", 1)
    assert int(code) == 1 and "top_k" in rest  # NVFP4_ERR_INVALID_ARG with its reason
    assert int(out["bad_k"]) == 1
    assert int(out["empty"]) == 0
