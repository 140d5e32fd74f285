"""The boundary from plain C: include/sage.h compiles as C11, a C program
links against the built library and gets sizes, refusals and their reasons
without touching a GPU."""
import os
import shutil
import subprocess
import tempfile

import pytest

from quantized_attention_smooth_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "sage.h"

int main(void) {
  size_t ws = sage_workspace_bytes(2, 24, 24, 4096, 4096, 128);
  size_t wh = sage_workspace_bytes_host(2, 24, 24, 4096, 4096, 128, 0);
  /* D = 129 is refused before anything touches a device */
  sage_status s = sage_attn_fwd((const void*)0x10000, (const void*)0x10000,
                                (const void*)0x10000, (float*)0x10000, 1, 2, 2, 128, 128,
                                129, SAGE_HND, 0, 0.0f, SAGE_F16, (void*)0x10000,
                                (size_t)1 << 30, (sage_stream_t)0);
  printf("ws %zu\nhost %zu\nstatus %d\nreason %s\n", ws, wh, (int)s, sage_last_error());
  return (ws > 0 && wh > 0 && s == SAGE_ERR_UNSUPPORTED) ? 0 : 1;
}
"""


def test_header_compiles_as_c_and_links():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = _build.build()
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "use_sage.c")
        exe = os.path.join(tmp, "use_sage")
        with open(src, "w") as f:
            f.write(C_SOURCE)
        subprocess.check_call([gcc, "-std=c11", "-Wall", "-Werror", "-pedantic",
                               "-I", os.path.join(ROOT, "include"), src, "-o", exe,
                               lib, "-Wl,-rpath," + os.path.dirname(lib)])
        run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    fields = dict(line.split(" ", 1) for line in run.stdout.strip().splitlines())
    assert int(fields["ws"]) > 0 and int(fields["host"]) > 0
    assert "D" in fields["reason"] and "128" in fields["reason"]
