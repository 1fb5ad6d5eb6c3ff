"""The boundary as a plain C program sees it: include/sage.h compiled as C99
with gcc, linked against libsage.so, and the host-only entry points called
(workspace size and layout, argument checks, status strings).  Nothing here
touches a GPU: every call below returns before any CUDA work."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "sage.h"

int main(void) {
  sage_shape s = {4, 32, 8, 4096, 65536, 128};
  sage_ws_layout L;
  sage_status st = sage_workspace_layout(&s, SAGE_Q8_PV8, 128, 128, &L);
  if (st != SAGE_OK) { printf("layout %d\n", (int)st); return 1; }
  printf("bytes %zu\n", sage_workspace_bytes(&s, SAGE_Q8_PV8, 128, 128));
  printf("total %zu\n", L.total);
  printf("pads %d %d %d %d\n", L.N_pad, L.M_pad, L.Tm, L.Tn);
  /* checks that return before any device work */
  sage_shape bad = {1, 3, 2, 256, 256, 64};
  printf("hq_hkv %zu\n", sage_workspace_bytes(&bad, SAGE_Q8_PV8, 128, 64));
  printf("null_ws %d\n", (int)sage_attn_fwd(&s, 0, 0.125f, SAGE_Q8_PV8, SAGE_SMOOTH_K, 128, 128, NULL, 0, NULL, NULL));
  printf("flags %d\n", (int)sage_quantize_qkv(&s, SAGE_Q8_PV8, 64, 128, 128, NULL, NULL, NULL, NULL, 0, NULL));
  printf("str %s\n", sage_status_str(SAGE_ERR_WORKSPACE));
  {
    sage_shape sb = {1, 2, 2, 256, 256, 64};
    printf("bwd_null %d\n", (int)sage_attn_bwd(&sb, 0, 0.125f, SAGE_SAGEBWD_I8, SAGE_SMOOTH_K, 128, 64, NULL, 0,
                                                  NULL, NULL, NULL, NULL, NULL, NULL));
  }
  {
    const int cq[4] = {0, 100, 100, 400}, ck[4] = {0, 150, 160, 700};
    printf("varlen %zu\n", sage_varlen_workspace_bytes(3, cq, ck, 8, 2, 128, SAGE_Q8_PV8, 128, 64));
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    import __graft_entry__
    __graft_entry__.build_library()
    lib_dir = os.path.join(ROOT, "bit_quantized_attention_gb300")
    d = tmp_path_factory.mktemp("capi")
    src = d / "use_sage.c"
    src.write_text(PROGRAM)
    exe = d / "use_sage"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    "-o", str(exe), str(src), "-L", lib_dir, "-lsage", "-Wl,-rpath," + lib_dir], check=True)
    return str(exe)


def test_header_compiles_as_c99_and_links(program):
    out = subprocess.run([program], capture_output=True, text=True, check=True).stdout
    vals = dict(line.split(" ", 1) for line in out.strip().splitlines())
    import bit_quantized_attention_gb300 as sage
    s = sage.Shape(4, 32, 8, 4096, 65536, 128)
    assert int(vals["bytes"]) == sage.sage_workspace_bytes(s, 0, 128, 128) == int(vals["total"])
    assert vals["pads"] == "4096 65536 32 512"
    assert int(vals["hq_hkv"]) == 0
    assert int(vals["null_ws"]) == 1 and int(vals["flags"]) == 1
    assert vals["str"] == "workspace too small"
    assert int(vals["bwd_null"]) == 1
    assert int(vals["varlen"]) > sage.sage_workspace_bytes(sage.Shape(3, 8, 2, 300, 540, 128), 0, 128, 64)
