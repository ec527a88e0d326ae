"""Host-side arithmetic of the library, checked on the CPU (no GPU needed):
the invariant-divisor division the tensor-core epilogue uses to map tile rows
to output positions, compiled from the library's own header with nvcc as a
host program and compared with integer division."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "transposed_convolution_convt3d_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include "convt3d_internal.h"
using namespace convt3d;
int main() {
    uint64_t bad = 0, checked = 0, x = 88172645463325252ull;
    auto rnd = [&]() { x ^= x << 13; x ^= x >> 7; x ^= x << 17; return x; };
    for (uint32_t d = 1; d < 4096; ++d) {
        const FastDiv f = make_fastdiv(d);
        for (uint32_t n = 0; n < 5000; ++n, ++checked) bad += fastdiv(n, f) != n / d;
        for (int i = 0; i < 200; ++i, ++checked) { const uint32_t n = (uint32_t)rnd(); bad += fastdiv(n, f) != n / d; }
        bad += fastdiv(0xFFFFFFFFu, f) != 0xFFFFFFFFu / d; ++checked;
    }
    for (int k = 0; k < 20000; ++k) {
        const uint32_t d = 1 + (uint32_t)(rnd() % 0x7FFFFFFFu);
        const FastDiv f = make_fastdiv(d);
        for (int i = 0; i < 16; ++i, ++checked) { const uint32_t n = (uint32_t)rnd(); bad += fastdiv(n, f) != n / d; }
    }
    std::printf("%llu %llu\n", (unsigned long long)bad, (unsigned long long)checked);
    return bad != 0;
}
"""


def test_fastdiv_matches_integer_division(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "fastdiv_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "fastdiv_check"
    subprocess.run([nvcc, "-std=c++17", "-O2", "-I", INCLUDE, "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    bad, checked = (int(v) for v in out.stdout.split())
    assert out.returncode == 0 and bad == 0
    assert checked > 20_000_000


def test_bench_reports_the_compute_dtype_of_each_precision():
    import bench
    assert bench.compute_dtype("3xtf32") == "f32" and bench.compute_dtype("3xbf16") == "f32"
    assert bench.compute_dtype("ffma") == "f32"
    assert bench.compute_dtype("tf32") == "tf32" and bench.compute_dtype("bf16") == "bf16"
