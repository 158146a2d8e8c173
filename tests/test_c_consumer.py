"""The C ABI from plain C: ``include/sparse_attn.h`` compiles as strict C99 and
a C program linked against ``libsparse_attn.so`` calls the host-side entry
points (no GPU, no Python in between). The pattern table it prints must equal
the oracle's own draw bit for bit."""

import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import bigbird_random_table

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "sparse_attn.h"

int main(void) {
    enum { H = 2, N = 1024, B = 64, G = 2, W = 3, R = 3 };
    int32_t table[H * (N / B) * R];
    sa_status st = build_bigbird_pattern(77u, H, N, B, G, W, R, table);
    if (st != SA_OK) return 10;
    /* invalid arguments come back as SA_ERR_INVALID_ARG, not a crash */
    if (build_bigbird_pattern(77u, H, 1000, B, G, W, R, table) != SA_ERR_INVALID_ARG) return 11;
    if (strcmp(sa_status_string(SA_ERR_TIMEOUT), "SA_ERR_TIMEOUT") != 0) return 12;
    if (sa_set_option(999, 1) != SA_ERR_INVALID_ARG) return 13;
    for (int i = 0; i < H * (N / B) * R; ++i) printf("%d\n", (int)table[i]);
    return 0;
}
"""


@pytest.fixture(scope="module")
def libpath():
    from block_sparse_long_bigbird_gb300 import _build, _lib

    if not os.path.exists(_lib.LIB_PATH):
        _build.build()
    return _lib.LIB_PATH


def test_header_is_strict_c99_and_the_library_links_from_c(tmp_path, libpath):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consumer.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(libpath)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), libdir + "/libsparse_attn.so", "-Wl,-rpath," + libdir]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stderr)
    got = np.array([int(x) for x in run.stdout.split()], dtype=np.int32).reshape(2, 1024 // 64, 3)
    want = bigbird_random_table(77, 2, 1024, 64, 2, 3, 3)
    assert np.array_equal(got, want)
