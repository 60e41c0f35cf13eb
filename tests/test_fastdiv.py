"""Host check of csrc/fastdiv.h: division by an invariant divisor as multiply-high and shifts must
equal the built-in unsigned division for every dividend the kernel can pass (all 32-bit values).

The header is plain C++; the test builds a small driver with the system C++ compiler and compares
against `/` for edge dividends (0, 1, d-1, d, d+1, multiples and 2^32-1) and random ones, over small,
power-of-two, odd, prime and large divisors."""

import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_verification_82_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include <cstdint>
#include <random>
#include "fastdiv.h"
using namespace specv;
static int check(uint32_t n, const FastDiv& f) {
  if (fdiv(n, f) != n / f.d) { std::printf("FAIL n=%u d=%u got %u\n", n, f.d, fdiv(n, f)); return 1; }
  return 0;
}
int main() {
  std::mt19937_64 rng(12345);
  const uint32_t ds[] = {1u, 2u, 3u, 5u, 7u, 8u, 10u, 11u, 16u, 19u, 32u, 60u, 61u, 66u, 88u, 128u, 176u, 208u,
                         256u, 1000u, 1009u, 4097u, 65535u, 65536u, 65537u, 1000003u, 16777216u, 2147483647u,
                         2147483648u, 4294967295u};
  int bad = 0;
  for (uint32_t d : ds) {
    const FastDiv f = make_fastdiv(d);
    const uint32_t edge[] = {0u, 1u, d - 1u, d, d + 1u, 2u * d, 2u * d - 1u, 4294967295u, 4294967294u,
                             2147483647u, 2147483648u, 4294967295u / d * d, 4294967295u / d * d - 1u};
    for (uint32_t n : edge) bad += check(n, f);
    for (int i = 0; i < 200000; ++i) bad += check((uint32_t)rng(), f);
    for (uint32_t n = 0; n < 5000; ++n) bad += check(n, f);
  }
  for (int i = 0; i < 2000; ++i) {  // random divisors
    const uint32_t d = (uint32_t)(rng() % 4294967295ull) + 1u;
    const FastDiv f = make_fastdiv(d);
    for (int j = 0; j < 200; ++j) bad += check((uint32_t)rng(), f);
  }
  std::printf("bad %d\n", bad);
  return bad != 0;
}
"""


def test_fastdiv_matches_builtin_division():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.cpp")
        exe = os.path.join(d, "t")
        with open(src, "w") as f:
            f.write(DRIVER)
        subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, src, "-o", exe], check=True)
        r = subprocess.run([exe], capture_output=True, text=True)
        assert r.returncode == 0, r.stdout
        assert "bad 0" in r.stdout
