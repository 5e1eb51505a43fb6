"""Division by plan-time divisors (multiply-high + shift, Granlund and
Montgomery 1994): the host build of the same header function is compiled
with g++ and compared against integer division over every divisor up to
4096, the largest ones the planner can produce, and numerators at the
edges of each quotient step and of the 32-bit range."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = r"""
#include <cstdio>
#include <cstdint>
#include "plan.h"
using namespace mhla;
int main() {
  uint64_t bad = 0, checked = 0;
  uint32_t st = 12345u;
  auto rnd = [&]() { st = st * 1664525u + 1013904223u; return st; };
  auto check = [&](uint32_t n, const FastDiv& f) {
    ++checked;
    if (fdiv(n, f) != n / f.d) { if (bad < 5) std::printf("n=%u d=%u got %u\n", n, f.d, fdiv(n, f)); ++bad; }
  };
  const uint32_t big[] = {65535u, 65536u, 65537u, 1u << 20, (1u << 24) + 7u, 2147483647u, 1000003u};
  for (uint32_t d = 1; d <= 4096 + 7; ++d) {
    const FastDiv f = make_fastdiv(d <= 4096 ? d : big[d - 4097]);
    const uint32_t dd = f.d;
    const uint32_t edges[] = {0u, 1u, dd - 1, dd, dd + 1, 2 * dd - 1, 2 * dd, 0x7fffffffu, 0x80000000u, 0xffffffffu,
                              0xffffffffu - dd, (0xffffffffu / dd) * dd, (0xffffffffu / dd) * dd - 1};
    for (uint32_t n : edges) check(n, f);
    for (int k = 0; k < 400; ++k) {
      const uint32_t q = (uint32_t)(rnd() % (0xffffffffull / dd + 1));
      check(q * dd, f);
      if (q * dd > 0) check(q * dd - 1, f);
      check(rnd(), f);
      check(rnd() >> (rnd() % 32), f);
    }
  }
  std::printf("checked %llu bad %llu\n", (unsigned long long)checked, (unsigned long long)bad);
  return bad ? 1 : 0;
}
"""


def test_fastdiv_matches_integer_division(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "fastdiv.cpp"
    src.write_text(SRC)
    exe = tmp_path / "fastdiv"
    subprocess.run([gxx, "-O2", "-std=c++17", f"-I{ROOT}/include", f"-I{ROOT}/token_level_head_phi_gb300/csrc",
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    assert " bad 0" in out.stdout
