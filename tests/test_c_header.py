"""The boundary as a plain C caller sees it: include/grpo_rowpass.h compiles as C99 (no
C++ in it), and a C program linked against the library calls it (host-side paths only:
status strings, argument validation and the workspace-size query; nothing is launched)."""
import os
import shutil
import subprocess

import pytest

from rl_fine_tuning_pass_gb300.build import INCLUDE, LIB_PATH, PKG, build

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "grpo_rowpass.h"

int main(void) {
  grpo_rows x;
  uint64_t ws = 0;
  memset(&x, 0, sizeof(x));
  x.dtype = GRPO_BF16;
  x.B = 2; x.L = 3; x.V = 0;                       /* V = 0 is rejected on the host */
  if (grpo_loss_fwd(&x, NULL, NULL, NULL, NULL, NULL, 1.0f, 0.0f, 0.2f, 0.2f, NULL, NULL, NULL, NULL, NULL,
                    NULL, NULL, NULL) != GRPO_ERR_INVALID_ARG) return 1;
  if (strncmp(grpo_status_string(GRPO_OK), "GRPO_OK", 7) != 0) return 2;
  if (grpo_fused_linear_workspace_size(1024, 151936, 1024, &ws) != GRPO_OK || ws < 151936ull * 1024 * 2) return 3;
  x.V = 8; x.B = 0;                                 /* no rows: valid, nothing launched */
  if (entropy_from_logits(&x, 1.0f, NULL, NULL, NULL) != GRPO_OK) return 4;
  printf("ok\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    return build()


def test_header_is_c99_and_a_c_program_links_and_runs(tmp_path, lib_path):
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "caller"
    res = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", INCLUDE, str(src), "-o", str(exe),
                          "-L", PKG, "-lgrpo_rowpass", f"-Wl,-rpath,{PKG}"], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stdout, run.stderr)
