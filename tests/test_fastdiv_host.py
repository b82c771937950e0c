"""Host pin of the gathers' division by invariant divisors (fg_abi.h,
fast_div): floor(x / d) = floor(x * mul / 2^sh) for every dividend below
2^31, against plain integer division: every divisor up to 5000 with edge and
random dividends, divisors around each power of two up to 2^31, divisors
above 2^31 (quotient 0) and a million random pairs.  Compiled with the host
C++ compiler against the library's own header."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "group_execution_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <cstdint>
#include <cstdio>
#include <random>
#include "fg_abi.h"
using namespace fg;
static uint32_t div_inv(uint32_t x, FastDiv f) { return (uint32_t)(((uint64_t)x * f.mul) >> f.sh); }
int main() {
  std::mt19937_64 rng(7);
  unsigned long long bad = 0, n = 0;
  const uint32_t xmax = 0x7fffffffu;
  auto check = [&](int64_t d, uint32_t x) {
    const FastDiv f = fast_div(d);
    const uint32_t want = (uint32_t)((uint64_t)x / (uint64_t)d);
    ++n;
    if (div_inv(x, f) != want) ++bad;
    if (f.mul != 0 && f.sh > 63) ++bad;
  };
  for (int64_t d = 1; d <= 5000; ++d) {
    for (int k = 0; k < 20; ++k) check(d, (uint32_t)(rng() % (xmax + 1ull)));
    const uint64_t m = (xmax / d) * d;
    check(d, 0); check(d, xmax); check(d, (uint32_t)m);
    if (m) check(d, (uint32_t)(m - 1));
    if (d <= xmax) { check(d, (uint32_t)d); check(d, (uint32_t)(d - 1)); }
  }
  for (int s = 2; s <= 31; ++s)
    for (int64_t dd = -2; dd <= 2; ++dd) {
      const int64_t d = (int64_t(1) << s) + dd;
      for (int k = 0; k < 500; ++k) check(d, (uint32_t)(rng() % (xmax + 1ull)));
      check(d, xmax);
    }
  for (int k = 0; k < 1000000; ++k) check(1 + (int64_t)(rng() % (uint64_t(1) << 31)), (uint32_t)(rng() % (xmax + 1ull)));
  for (int64_t d : {(int64_t(1) << 31) + 1, int64_t(1) << 32, int64_t(1) << 40}) { check(d, xmax); check(d, 12345); }
  printf("%llu %llu\n", n, bad);
  return bad != 0;
}
"""


def test_fast_div_matches_integer_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda.h")):
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    src = tmp_path / "fastdiv.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "fastdiv"
    subprocess.run([cxx, "-O2", "-std=c++17", f"-I{CSRC}", f"-I{CUDA_INC}", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    n, bad = (int(v) for v in out.stdout.split())
    assert n > 1_000_000 and bad == 0, out.stdout
