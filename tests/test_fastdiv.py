"""The multiply-shift division the kernels use for tile and row indices
(Granlund and Montgomery, "Division by Invariant Integers using
Multiplication", PLDI 1994, Figure 4.1), checked on the CPU against plain
integer division.

The header's host form (the same formula with the multiply-high done in
64-bit arithmetic; the device form uses __umulhi, which computes the same
high word) is compiled with g++ into a small program that prints, for each
divisor, the quotients of edge and random dividends; every one must equal
n // d.  Divisors cover 1, small values, powers of two and their
neighbours, and the 32-bit extremes.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "int8_quantized_q8ta_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include "fastdiv.h"
int main() {
  unsigned d, n;
  while (std::scanf("%u %u", &d, &n) == 2) {
    const q8::FastDiv f = q8::make_fastdiv(d);
    std::printf("%u\n", q8::fast_div_host(n, f));
  }
  return 0;
}
"""

DIVISORS = [1, 2, 3, 5, 6, 7, 9, 10, 11, 12, 13, 46, 64, 100, 152, 255, 256, 257, 511, 512,
            640, 1000, 4095, 4096, 4097, 65535, 65536, 65537, 1 << 20, (1 << 24) + 1,
            (1 << 31) - 1, 1 << 31, (1 << 31) + 1, (1 << 32) - 2, (1 << 32) - 1]


@pytest.fixture(scope="module")
def prog(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    d = tmp_path_factory.mktemp("fastdiv")
    src = d / "fd.cpp"
    src.write_text(PROGRAM)
    exe = d / "fd"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)])
    return str(exe)


def test_quotients_equal_integer_division(prog):
    rng = np.random.default_rng(7)
    cases = []
    for d in DIVISORS:
        ns = {0, 1, d - 1, d, d + 1, 2 * d - 1, 2 * d, (1 << 32) - 1, (1 << 32) - 2, (1 << 31),
              (1 << 31) - 1}
        ns |= {int(v) for v in rng.integers(0, 1 << 32, 200, dtype=np.uint64)}
        k = ((1 << 32) - 1) // d
        ns |= {k * d, k * d - 1 if k * d > 0 else 0, (k // 2) * d + d - 1}
        cases += [(d, n) for n in sorted(ns) if 0 <= n < (1 << 32)]
    inp = "\n".join(f"{d} {n}" for d, n in cases) + "\n"
    out = subprocess.run([prog], input=inp, capture_output=True, text=True, check=True).stdout
    got = [int(v) for v in out.split()]
    assert len(got) == len(cases)
    bad = [(d, n, q) for (d, n), q in zip(cases, got) if q != n // d]
    assert not bad, bad[:5]
