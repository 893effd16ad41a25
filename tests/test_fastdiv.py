"""The kernels divide item indices by tile counts with a precomputed
multiplier and shift (CdgDiv, the round-up method of Granlund and
Montgomery).  This compiles the host constructor from the kernels' parameter
header and checks n / d = (mulhi(n, mul) + n) >> shr against integer
division for every divisor up to 4096 and for large ones, at the edges and
at random n below 2^31."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "implicit_gemm_dgrad_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include <random>
#include "cdg_params.h"
static uint32_t q(uint32_t n, CdgDiv d)
{
    const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(n) * d.mul) >> 32);
    return (hi + n) >> d.shr;
}
int main()
{
    std::mt19937 rng(12345);
    long bad = 0, checked = 0;
    auto check = [&](uint32_t d) {
        const CdgDiv v = cdg_make_div(d);
        const uint32_t edges[] = {0u, 1u, d - 1u, d, d + 1u, 2u * d - 1u, 0x7FFFFFFFu, 0x7FFFFFFEu, 0x40000000u};
        for (uint32_t n : edges) {
            if (n > 0x7FFFFFFFu) continue;
            ++checked;
            if (q(n, v) != n / d) ++bad;
        }
        for (int i = 0; i < 64; ++i) {
            const uint32_t n = rng() & 0x7FFFFFFFu;
            ++checked;
            if (q(n, v) != n / d) ++bad;
        }
    };
    for (uint32_t d = 1; d <= 4096; ++d) check(d);
    for (int i = 0; i < 4096; ++i) check(1u + (rng() & 0x3FFFFFFFu));
    for (uint32_t k = 0; k < 31; ++k) { check(1u << k); check((1u << k) + 1u); }
    std::printf("%ld %ld\n", checked, bad);
    return bad != 0;
}
"""


def test_fast_division_matches_integer_division(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "div.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "div"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run([cxx, "-O2", "-std=c++17", f"-I{CSRC}", f"-I{cuda_inc}", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    checked, bad = map(int, out.stdout.split())
    assert out.returncode == 0 and bad == 0 and checked > 500_000
