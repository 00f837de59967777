"""The extend kernel maps work items to (row-tile pair, kv head, request) by
dividing by launch constants with a multiply-high and a shift (FastDiv in
csrc/internal.h).  This builds the header's host path with the system C++
compiler and checks it against exact division: every divisor up to 300 and
some large ones, dense small numerators, random ones and values next to 2^31."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

PROG = r"""
#include "internal.h"
#include <cstdio>
#include <cstdint>
int main() {
  uint64_t s = 88172645463325252ull, bad = 0, checked = 0;
  auto rnd = [&]() { s ^= s << 13; s ^= s >> 7; s ^= s << 17; return (uint32_t)(s & 0x7FFFFFFFu); };
  const uint32_t big[] = {1000u, 4096u, 65535u, 100003u, (1u << 20) + 7u, (1u << 30) - 1u, 2147483647u};
  for (int k = 0; k < 300 + 7; ++k) {
    const uint32_t d = k < 300 ? (uint32_t)(k + 1) : big[k - 300];
    const pkv::FastDiv f = pkv::make_fastdiv(d);
    auto check = [&](uint32_t n) {
      ++checked;
      if (f.div(n) != n / d || f.mod(n) != n % d) ++bad;
    };
    for (uint32_t n = 0; n < 5000; ++n) check(n);
    for (int i = 0; i < 5000; ++i) check(rnd());
    for (uint32_t n = 2147483647u - 64u; n <= 2147483647u - 1u; ++n) check(n);
    check(2147483647u);
  }
  std::printf("%llu %llu\n", (unsigned long long)checked, (unsigned long long)bad);
  return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.isdir(CUDA_INC),
                    reason="needs g++ and the CUDA headers")
def test_fastdiv_matches_exact_division():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.cpp")
        exe = os.path.join(d, "t")
        with open(src, "w") as f:
            f.write(PROG)
        subprocess.run(["g++", "-O2", "-std=c++17", "-I", os.path.join(ROOT, "paged_kv_cache_285_gb300", "csrc"),
                        "-I", CUDA_INC, src, "-o", exe], check=True, capture_output=True)
        out = subprocess.run([exe], capture_output=True, text=True)
        checked, bad = map(int, out.stdout.split())
        assert checked > 3_000_000 and bad == 0, out.stdout
