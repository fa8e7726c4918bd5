"""The boundary from plain C: include/td.h compiles as C99 with warnings as
errors, and a C program linked against libtd.so sizes a workspace, names
status codes and gets argument errors back -- all host-side, no GPU."""
import os
import shutil
import subprocess

import pytest

from sparse_attention_td_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "td.h"

int main(void)
{
    td_shape s = {2, 8, 2, 128, 1000, 0.0f};   /* batch, q heads, kv heads, d, N, scale */
    size_t a = td_workspace_size(&s, 0), b = td_workspace_size(&s, 64);
    if (a == 0 || b <= a) return 1;
    td_shape bad = s;
    bad.head_dim = 64;
    if (td_workspace_size(&bad, 0) != 0) return 2;
    if (strcmp(td_status_string(TD_ERR_NO_SELECTION), "TD_ERR_NO_SELECTION") != 0) return 3;
    /* host-side validation: nothing is launched, no device memory touched */
    if (td_full_attn_select(&s, NULL, NULL, NULL, NULL, 0, NULL, NULL, NULL, NULL, NULL, 0, NULL)
        != TD_ERR_INVALID_ARG) return 4;
    if (td_index_overlap(&s, NULL, NULL, 4, NULL, NULL) != TD_ERR_INVALID_ARG) return 5;
    int32_t modes[2] = {TD_MODE_FULL, TD_MODE_SPARSE};
    if (td_set_tuning("no_such_knob", 1) != TD_ERR_INVALID_ARG) return 6;
    (void)modes;
    printf("ok %zu %zu\n", a, b);
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    return libbuild.build()


def test_header_is_c99_and_the_abi_links_from_c(tmp_path, lib_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib_path)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", libdir, "-ltd", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert run.stdout.startswith("ok ")
