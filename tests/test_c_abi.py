"""The C ABI from C: include/sa.h compiles as C99 with warnings as errors, and
a C program linked against libsa_gb300.so calls the host-side entry points
(parameter set-up, sizes, argument checks, status names). No GPU needed."""

import os
import shutil
import subprocess

import pytest

from helpers import lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "sa.h"

int main(void) {
  sa_params p;
  sa_params_init(&p, 1, 38247, 56, 128, 951, 1.0f);
  if (sa_num_blocks(&p) != 598) return 1;
  if (sa_route_rows(&p) != 56 * 598) return 2;
  if (sa_route_max_nnz(&p) != (int64_t)56 * 598 * 598) return 3;
  if (sa_route_workspace_bytes(&p) == 0 || sa_attn_workspace_bytes(&p) == 0) return 4;
  p.q_block = 128;
  if (sa_route_workspace_bytes(&p) == 0) return 5;
  p.q_block = 96;
  if (sa_route_workspace_bytes(&p) != 0) return 6;        /* rejected */
  p.q_block = 0;
  /* a NULL q is rejected before anything is launched */
  if (sa_route(&p, NULL, NULL, NULL, NULL, 0, NULL, 0, NULL, NULL) != SA_ERR_INVALID_ARG) return 7;
  if (sa_dev_status_decode(SA_DEV_TIMEOUT | SA_DEV_CAPACITY) != SA_ERR_TIMEOUT) return 8;
  if (strcmp(sa_status_string(SA_ERR_CAPACITY), "SA_ERR_CAPACITY") != 0) return 9;
  printf("ok %u\n", (unsigned)sizeof(sa_params));
  return 0;
}
"""


@pytest.fixture(scope="module")
def built():
    lib()                                   # builds libsa_gb300.so if needed
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    return os.path.join(ROOT, "block_sparse_attention_sa_gb300")


def test_header_is_c99_and_host_calls_work_from_c(built, tmp_path):
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", built, "-lsa_gb300", f"-Wl,-rpath,{built}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")
