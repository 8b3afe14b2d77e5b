"""The page-size division of the paged kernels (csrc/page_div.h), host side.

The kernels divide key indices by the page size with a multiply-high and a
shift (magic numbers made once per call on the host). The same header's host
path is compiled here and checked against plain integer division: every
divisor from 2 to 4096, every multiple of 64 up to 2^20 and a few large
ones, on numerators at the edges of every quotient (k*d - 1, k*d, k*d + 1),
a sweep of small values and the largest index, 2^31 - 1.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "infra_dsa_indexer_gb300", "csrc")

PROGRAM = r"""
#include "page_div.h"
#include <cstdio>
#include <vector>
int main() {
  std::vector<uint32_t> ds;
  for (uint32_t d = 2; d <= 4096; ++d) ds.push_back(d);
  for (uint32_t d = 4160; d <= (1u << 20); d += 64) ds.push_back(d);
  for (uint32_t d : {1000003u, 1u << 24, (1u << 24) + 64, 1u << 30, (1u << 31) - 1, 1u << 31})
    ds.push_back(d);
  long long checks = 0, bad = 0;
  const uint32_t nmax = 0x7fffffffu;
  for (uint32_t d : ds) {
    const dsa::PageDiv pd = dsa::page_div_make(d);
    auto check = [&](uint64_t n) {
      if (n > nmax) return;
      ++checks;
      if (dsa::page_div(static_cast<uint32_t>(n), pd.magic, pd.shift) != n / d) ++bad;
    };
    for (uint32_t n = 0; n < 4096; ++n) check(n);
    check(nmax);
    check(nmax - 1);
    // quotient edges across the whole range, 64 quotients per divisor
    const uint64_t qmax = nmax / d;
    for (uint64_t i = 0; i <= 64; ++i) {
      const uint64_t k = qmax * i / 64;
      check(k * d);
      if (k * d > 0) check(k * d - 1);
      check(k * d + 1);
      check(k * d + d - 1);
    }
  }
  std::printf("%lld %lld\n", checks, bad);
  return 0;
}
"""


def test_page_div_matches_integer_division(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not found")
    src = tmp_path / "page_div_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "page_div_check"
    subprocess.run([cxx, "-std=c++17", "-O2", "-Wall", "-Werror", "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    checks, bad = (int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                                  text=True).stdout.split())
    assert checks > 10_000_000
    assert bad == 0
