"""The boundary is a C ABI: include/dcp.h must compile as plain C (C11, no
C++), and a C program linked against the library must be able to call it.
The program below only exercises calls that validate and return on the host
(sizes, alignment, aliasing, status strings), so it needs no GPU."""
import os
import subprocess

import pytest

from decode_context_attention_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "dcp.h"

#define A ((void*)0x10000000)
#define L ((float*)0x20000000)
#define C ((void*)0x30000000)
#define W ((float*)0x40000000)

int main(void) {
    int bad = 0;
    bad |= dcp_lse_pack_dim(DCP_F32) != 1;
    bad |= dcp_lse_pack_dim(DCP_BF16) != 2;
    bad |= dcp_lse_pack_dim(DCP_FP8_E4M3) != 4;
    bad |= dcp_lse_pack_dim(99) != -1;
    bad |= strlen(dcp_status_string(DCP_ERR_ALIAS)) == 0;
    /* H = 6 is not a multiple of N = 4: refused before any launch */
    dcp_status_t s = dcp_pack_send(DCP_BF16, 4, 2, 6, 8, 1, A, 96, 48, 8, L, 12, 6, 1,
                                   C, 80, 20, 10, 10, W, 8, 2, 1, 1, NULL);
    bad |= s != DCP_ERR_HEADS_NOT_DIVISIBLE;
    bad |= strstr(dcp_last_error_message(), "multiple") == NULL;
    /* an unknown flag on the combine */
    s = dcp_lse_combine(DCP_F32, 2, 2, 4, 8, 1, A, 128, 64, 32, 8, L, 16, 8, 4, 1,
                        C, 64, 32, 8, W, 8, 4, 1, DCP_LSE_BASE_E, 1, 8u, NULL);
    bad |= s != DCP_ERR_INVALID_ARG;
    /* empty problems succeed and launch nothing */
    s = dcp_unpack_combine(DCP_F16, 2, 0, 4, 8, 1, A, 160, 80, 40, 10, C, 64, 32, 8, W, 8, 4, 1,
                           DCP_LSE_BASE_2, 1, 0u, NULL);
    bad |= s != DCP_OK;
    bad |= dcp_decode_attention_workspace_size(4, 3, 8, 128, 4001, 1000) != (size_t)4 * 3 * 8 * 2 * 129 * 4;
    printf(bad ? "FAIL\n" : "OK\n");
    return bad;
}
"""


def test_header_compiles_as_c_and_the_library_links_and_validates(tmp_path):
    lib = build.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-L", libdir, "-ldcp_gb300", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr
