"""The boundary as a C caller sees it (no GPU needed).

include/dsa_indexer.h must compile as C99 and as C++17 with every warning an
error, and a C program linked against the library must be able to call the
entry points that need no device: the ABI version, the status strings, the
shape-only workspace size, and host-side argument validation (a NULL shape,
a bad head count) returning the documented status codes.
"""
import os
import re
import shutil
import subprocess

import pytest

from infra_dsa_indexer_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include "dsa_indexer.h"
#include <stdio.h>
#include <string.h>

int main(void) {
  idx_shape sh;
  memset(&sh, 0, sizeof(sh));
  sh.B = 1; sh.S = 4; sh.N = 1024; sh.H = 64; sh.D = 128;
  sh.fmt = IDX_FMT_BF16; sh.w_fmt = IDX_W_F32; sh.out_row_stride = 1024;
  const long long ws = (long long)indexer_logits_topk_workspace_bytes(&sh);
  const long long ws_null = (long long)indexer_logits_topk_workspace_bytes(NULL);
  /* Argument checks run on the host before the device is touched: any
     16-byte aligned addresses pass the pointer checks here. */
  static float buf[64] __attribute__((aligned(16)));
  static int win[8] __attribute__((aligned(16)));
  sh.H = 32;  /* only H = 64 is supported */
  const int bad_h = indexer_logits(buf, NULL, buf, NULL, NULL, buf, win, win, 0.1f, 1, buf,
                                   &sh, (idx_stream_t)0);
  const int null_shape = indexer_logits(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0.1f,
                                        1, NULL, NULL, (idx_stream_t)0);
  printf("version %d\n", indexer_version());
  printf("ok %s\n", indexer_status_string(IDX_OK));
  printf("ws %lld %lld\n", ws, ws_null);
  printf("codes %d %d\n", bad_h, null_shape);
  return 0;
}
"""


def status_codes():
    """The idx_status values as the header defines them."""
    text = open(os.path.join(INCLUDE, "dsa_indexer.h")).read()
    return {k: int(v) for k, v in re.findall(r"\b(IDX_(?:OK|ERR_\w+))\s*=\s*(\d+)", text)}


def compiler(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not found")
    return path


@pytest.mark.parametrize("lang", ["c99", "c++17"])
def test_header_compiles_cleanly(tmp_path, lang):
    cc = compiler("gcc" if lang == "c99" else "g++")
    src = tmp_path / ("h.c" if lang == "c99" else "h.cpp")
    src.write_text('#include "dsa_indexer.h"\nint main(void) { return indexer_version() > 0 ? 0 : 1; }\n')
    subprocess.run([cc, f"-std={lang}", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                    "-I", INCLUDE, str(src)], check=True, capture_output=True, text=True)


def test_c_program_calls_the_library(tmp_path):
    cc = compiler("gcc")
    lib = build.build()
    src = tmp_path / "caller.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
                    "-L", libdir, "-l:" + os.path.basename(lib), "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    fields = dict(line.split(" ", 1) for line in out if line)
    L = binding.load()
    assert int(fields["version"]) == L.indexer_version()
    assert fields["ok"] == binding.indexer_status_string(binding.IDX_OK)
    ws, ws_null = (int(x) for x in fields["ws"].split())
    shape = binding.make_shape(1, 4, 1024, 64, 128, 0, 0, out_row_stride=1024)
    assert ws == binding.indexer_logits_topk_workspace_bytes(shape) and ws > 0
    assert ws_null == -1
    codes = status_codes()
    bad_h, null_shape = (int(x) for x in fields["codes"].split())
    assert bad_h == codes["IDX_ERR_SHAPE"]
    assert null_shape == codes["IDX_ERR_NULL"]
