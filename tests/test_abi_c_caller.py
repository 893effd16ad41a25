"""The boundary is a C ABI: include/cdg.h compiles as C99, and a plain C
program links libcdg.so and plans dgrad and wgrad shapes through it (host-only
planning, so no device is needed)."""
import os
import shutil
import subprocess

import pytest

import implicit_gemm_dgrad_gb300 as cdg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include "cdg.h"
#include <stdio.h>
int main(void)
{
    cdg_handle_t d = 0;
    cdg_wgrad_t w = 0;
    cdg_plan_info_t di;
    cdg_wgrad_info_t wi;
    int rc = cdg_plan_host(2, 16, 16, 32, 32, 3, 3, 2, 1, 1, CDG_BF16, CDG_EPI_RELU_BWD, 148, &d);
    if (rc != CDG_OK || cdg_plan_get_info(d, &di) != CDG_OK) return 10 + rc;
    rc = cdg_wgrad_plan_host(2, 16, 16, 32, 32, 3, 3, 2, 1, 1, CDG_BF16, 0, 0, 148, &w);
    if (rc != CDG_OK || cdg_wgrad_get_info(w, &wi) != CDG_OK) return 20 + rc;
    printf("%d %d %d %d %zu %lld\n", di.num_phases, di.P, wi.P, wi.pos_box[0] * wi.pos_box[1] * wi.pos_box[2],
           cdg_packed_weight_bytes(d), cdg_relu_mask_bytes(10, 136));
    rc = cdg_dgrad(d, 0, 0, 0, 0, 0);  /* NULL tensors: an argument error, no launch */
    cdg_destroy(d);
    cdg_wgrad_destroy(w);
    cdg_destroy(0);                    /* NULL-safe */
    return rc == CDG_ERR_INVALID_ARG ? 0 : 30;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_plain_c_program_uses_the_library(tmp_path):
    lib = cdg.load_library()
    libdir = os.path.dirname(lib._name)
    src = tmp_path / "caller.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "caller"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-lcdg", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    phases, P, wP, box, wbytes, mbytes = out.stdout.split()
    assert (int(phases), int(P), int(wP), int(box)) == (4, 8, 8, 64)
    assert int(wbytes) == 2 * 32 * 9 * 32 and int(mbytes) == 10 * 32
