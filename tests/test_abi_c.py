"""The boundary from plain C: a C11 program that includes only include/lp.h and
links liblp.so (no Python, no torch) compiles with gcc and runs.  Without a
GB300 its valid calls fail with LP_ERR_UNSUPPORTED_DEVICE; argument errors are
reported before any device check; the host-only helpers answer."""

import os
import shutil
import subprocess

import pytest
import torch

from invariant_token_logprobs_gb300 import _build_lib, lp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "lp.h"

int main(void) {
  int64_t b = 0, e = 0;
  if (lp_vocab_shard_range(151936, 1, 4, &b, &e) != LP_OK || b != 37984 || e != 75968) return 1;
  if (strcmp(lp_status_string(LP_ERR_TIMEOUT), "LP_ERR_TIMEOUT") != 0) return 2;
  if (strcmp(lp_backend_id(), "lp.sm103a.bitwise.v1") != 0) return 3;
  /* a fake, aligned device address: these calls never dereference it */
  const void* A = (const void*)(uintptr_t)(1u << 20);
  float* F = (float*)(uintptr_t)(1u << 20);
  const int64_t* Y = (const int64_t*)(uintptr_t)(1u << 20);
  size_t ws = lp_linear_logprob_workspace_size(64, 256, 8192);
  if (ws == 0) return 4;
  /* argument errors come first */
  if (lp_linear_logprob(A, 256, A, 256, Y, 64, 256, 8192, NULL, F, (void*)A, ws, NULL) !=
      LP_ERR_INVALID_ARGUMENT) return 5;
  if (lp_linear_logprob(A, 256, A, 256, Y, 64, 256, 8192, F, F, (void*)A, ws - 1, NULL) !=
      LP_ERR_WORKSPACE_TOO_SMALL) return 6;
  if (lp_logprob_from_logits((const float*)A, 100, Y, 4, 100, F, F, NULL) !=
      (EXPECT_DEVICE)) return 7;
  if (lp_linear_logprob(A, 256, A, 256, Y, 64, 256, 8192, F, F, (void*)A, ws, NULL) !=
      (EXPECT_DEVICE)) return 8;
  const float* parts[2] = {F, F};
  if (lp_merge_grad_h_partials(parts, 3, 8, 256, F, NULL) != LP_ERR_INVALID_ARGUMENT) return 9;
  printf("ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_against_the_header(tmp_path):
    lib = lp.load()._name
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    if torch.cuda.is_available():
        pytest.skip("the device checks expect a machine without a GPU")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic",
                    "-DEXPECT_DEVICE=LP_ERR_UNSUPPORTED_DEVICE",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib),
                    "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.returncode
    assert out.stdout.strip() == "ok"
