"""The C ABI from plain C (no GPU): include/tg_gemm.h compiles as strict C99
with every warning an error, and a C program linked against the library
gets the planner's choice for the 8192^3 problem, status strings, the scale
buffer size, and argument errors returned before any CUDA call."""

from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "tg_gemm.h"

int main(void) {
    tg_plan_info info;
    tg_options opts;
    const void *a = (const void *)(size_t)4096, *b = (const void *)(size_t)8192;
    float *d = (float *)(size_t)16384;
    tg_status st;

    memset(&opts, 0, sizeof(opts));
    st = tg_plan(8192, 8192, 8192, a, 8192, b, 8192, d, 8192, TG_BF16, &opts, 152, &info);
    printf("plan %d %d %d %d %d %lld %d\n", (int)st, info.block_m, info.block_n, info.cta_pair,
           info.grid, (long long)info.tiles, info.stages);
    /* lda < K: rejected before anything touches CUDA. */
    st = tg_gemm(64, 64, 64, 1.0f, a, 32, b, 64, d, 64, TG_BF16, TG_EPILOGUE_RELU, NULL);
    printf("lda %d %s\n", (int)st, tg_status_string(st));
    /* Unknown epilogue and operand type. */
    st = tg_gemm(64, 64, 64, 1.0f, a, 64, b, 64, d, 64, TG_BF16, (tg_epilogue)7, NULL);
    printf("epi %d\n", (int)st);
    st = tg_gemm(64, 64, 64, 1.0f, a, 64, b, 64, d, 64, (tg_dtype)42, TG_EPILOGUE_NONE, NULL);
    printf("dtype %d\n", (int)st);
    /* An empty output launches nothing. */
    st = tg_gemm(0, 64, 64, 1.0f, NULL, 64, b, 64, NULL, 1, TG_BF16, TG_EPILOGUE_NONE, NULL);
    printf("empty %d %s\n", (int)st, tg_status_string(st));
    printf("scales %lld\n", (long long)tg_mx_scale_bytes(300, 1000));
    printf("version %d\n", (int)tg_version());
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib():
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    return tg.LIBRARY_PATH


def test_header_is_strict_c99(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "h.c"
    src.write_text('#include "tg_gemm.h"\nint main(void) { return (int)TG_OK; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o",
                        str(tmp_path / "h.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_against_the_library(tmp_path, lib):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "prog.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "prog"
    libdir = os.path.dirname(lib)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", libdir,
                        "-ltg_gemm", "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr
    out = dict((ln.split(" ", 1)[0], ln.split(" ", 1)[1]) for ln in r.stdout.splitlines())
    assert out["plan"] == "0 256 256 1 152 1024 7"
    assert out["lda"].startswith("1 ") and "INVALID" in out["lda"]
    assert out["epi"] == "1" and out["dtype"] == "1"
    assert out["empty"].startswith("0 ")
    assert out["scales"] == str(3 * 8 * 512)      # 3 row blocks x ceil(1000/128) atom columns
    assert int(out["version"]) > 0
