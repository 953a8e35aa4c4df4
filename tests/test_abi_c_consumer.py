"""The C ABI from a plain C99 program (no GPU): include/mla.h compiles as C
with warnings as errors, the program links against the built library and
calls its host-side entry points (validation, workspace sizing, options)."""
import os
import shutil
import subprocess

import pytest

from latent_causal_attention_gb300 import _lib
from latent_causal_attention_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "mla.h"

int main(void) {
  if (strcmp(mla_status_string(MLA_OK), "ok") != 0) return 1;
  if (mla_set_option(MLA_OPT_ATTN_PATH, 9) != MLA_ERR_SHAPE) return 2;
  if (mla_latent_attention(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 1, 64, 64, 0.125f, 1,
                           MLA_BF16, MLA_F32, NULL, 0, NULL) != MLA_ERR_NULL)
    return 3;
  if (mla_kv_latent_project(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 8, 64, 64, 0,
                            MLA_BF16, MLA_BF16, NULL) != MLA_ERR_NULL)
    return 4;
  {
    /* decode-shaped call: q' and o_lat in the workspace */
    size_t ws = mla_latent_attention_workspace_size(64, 1, 4096, 128, 128, 512, MLA_BF16, 1);
    if (ws < (size_t)2 * 64 * 128 * 512 * 2) return 5;
    printf("ok %zu\n", ws);
  }
  return 0;
}
"""


def test_header_compiles_and_links_as_c99(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    build()
    src = tmp_path / "use_mla.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "use_mla"
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lmla_gb300", f"-Wl,-rpath,{libdir}"], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0, (res.returncode, res.stdout, res.stderr)
    assert res.stdout.startswith("ok ")
