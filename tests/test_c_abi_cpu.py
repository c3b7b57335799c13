"""The boundary from plain C, without Python or a GPU: include/fgemm.h compiles as ISO C99 with
-pedantic and warnings as errors, and a C program linked against the built library calls the
host-side entries (status strings, the grouped tile order, the launch plan for a described
device, the unfused workspace size, argument validation)."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from conftest import read_golden  # noqa: E402

PKG = os.path.join(ROOT, "gemm_epilogue_gb300")
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fgemm.h"

int main(void) {
  fgemm_plan_info info;
  fgemm_opts opts;
  int64_t m, n, p;
  memset(&opts, 0, sizeof opts);
  if (strcmp(fgemm_status_string(FGEMM_ERR_TIMEOUT), "FGEMM_ERR_TIMEOUT") != 0) return 10;
  for (p = 0; p < 6; ++p) {
    if (fgemm_tile_of(p, 3, 2, 2, &m, &n) != FGEMM_OK) return 11;
    printf("tile %lld %lld %lld\n", (long long)p, (long long)m, (long long)n);
  }
  /* 4096^3 bf16 bias + ReLU on a described device of 152 SMs and 76 resident CTA pairs; the
     addresses are only checked for alignment, never dereferenced */
  if (fgemm_plan_on((const void*)0x10000000, (const void*)0x20000000, (const void*)0x30000000,
                    NULL, (const void*)0x50000000, 4096, 4096, 4096, FGEMM_BF16, FGEMM_EPI_RELU,
                    &opts, 152, 76, &info) != FGEMM_OK)
    return 12;
  printf("plan %d %d %d %d %d\n", info.path, info.grid, info.cluster, info.tiles, info.work_items);
  printf("unfused %lu\n", (unsigned long)fgemm_unfused_workspace_bytes(4096, 4096, FGEMM_BF16, 0));
  /* validation happens before any device is looked for */
  if (fgemm_bias_relu(NULL, NULL, NULL, NULL, -1, 1, 1, FGEMM_BF16, NULL) != FGEMM_ERR_INVALID_VALUE)
    return 13;
  if (fgemm_bias_relu(NULL, NULL, NULL, NULL, 0, 8, 8, FGEMM_BF16, NULL) != FGEMM_OK) return 14;
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    from gemm_epilogue_gb300 import build
    return build.build()


def _cc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    return cc


def test_header_is_iso_c99(tmp_path):
    src = tmp_path / "only_header.c"
    src.write_text('#include "fgemm.h"\nint main(void) { return 0; }\n')
    r = subprocess.run([_cc(), "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", INCLUDE,
                        "-c", str(src), "-o", str(tmp_path / "only_header.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_calls_the_host_entries(tmp_path, lib_path):
    src = tmp_path / "host_calls.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "host_calls"
    r = subprocess.run([_cc(), "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
                        lib_path, "-Wl,-rpath," + os.path.dirname(lib_path)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    lines = run.stdout.split("\n")
    # the grouped order of the page's table ("I3 ...", "Tiles and grouped ownership")
    g = read_golden("grouped_order_3x2_g2.txt")
    tiles = [ln.split()[1:] for ln in lines if ln.startswith("tile ")]
    assert [(int(p), int(m), int(n)) for p, m, n in tiles] == \
        [(p, *(int(v) for v in g[str(p)].split(","))) for p in range(6)]
    # 16 x 16 tiles of 256 x 256 on 76 pairs (152 CTAs); the 28 tiles of the last round in two
    # 128-column pieces: 228 + 56 work items
    assert "plan 1 152 2 256 284" in lines
    assert f"unfused {4096 * 4096 * 2}" in lines
