"""The C ABI from plain C (CPU).

include/attn.h must compile as strict C99 (no C++ or CUDA types in it), a C
program must link against the library, and the entry points that need no
device must behave as documented when called from C: the ABI version, the
status strings, the block-mask size query, the options, and argument errors
returned before any device work.
"""
import os
import shutil
import subprocess

import pytest

import attention_attn_fwd_04_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "attn.h"

int main(void) {
    attn_mod_desc m;
    double v = -1.0;
    attn_status a, b, c;
    memset(&m, 0, sizeof m);
    m.version = ATTN_MOD_DESC_VERSION;
    m.mask_flags = ATTN_MASK_CAUSAL;
    printf("abi %d\n", attn_abi_version());
    printf("bytes %lu\n", (unsigned long)attn_block_mask_bytes(2, 32, 8192, 8192, &m));
    printf("status %s\n", attn_status_string(ATTN_ERR_INVALID_ARG));
    a = attn_set_option(ATTN_OPT_RESCALE_THRESHOLD, 4.0);
    b = attn_get_option(ATTN_OPT_RESCALE_THRESHOLD, &v);
    c = attn_set_option(ATTN_OPT_RESCALE_THRESHOLD, 8.0);
    printf("option %d %d %d %g\n", (int)a, (int)b, (int)c, v);
    /* null tensors: rejected before any device work */
    printf("null %d\n", (int)attn_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 128, 128, 128,
                                      0.125f, NULL, NULL));
    return 0;
}
"""


def test_header_compiles_as_c99_and_host_entry_points_answer(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(attn.library_path())
    if not os.path.exists(attn.library_path()):
        pytest.skip("library not built")
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-L", lib_dir,
                    "-lattn_gb300", "-Wl,-rpath," + lib_dir, "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True,
                         timeout=120).stdout.splitlines()
    got = dict(line.split(" ", 1) for line in out)
    assert int(got["abi"]) == attn.lib().attn_abi_version()
    m = attn.ModDesc()
    m.version = attn.MOD_DESC_VERSION
    m.mask_flags = attn.MASK_CAUSAL
    import ctypes
    assert int(got["bytes"]) == attn.lib().attn_block_mask_bytes(2, 32, 8192, 8192,
                                                                 ctypes.byref(m))
    assert got["status"] == "ATTN_ERR_INVALID_ARG"
    assert got["option"].split() == ["0", "0", "0", "4"]
    assert int(got["null"]) == 1  # ATTN_ERR_INVALID_ARG
