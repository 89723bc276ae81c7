"""The kernels' invariant-divisor division (csrc/fastdiv.h) agrees with
integer division: compiled for the host with g++ and checked over dense
ranges, near the numerator bound and around multiples of many divisors
(CPU only)."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <cstdio>
#include "fastdiv.h"
int main() {
  const uint32_t divs[] = {1u, 2u, 3u, 5u, 6u, 7u, 8u, 9u, 12u, 16u, 24u, 31u, 36u, 64u, 80u, 96u,
                           127u, 128u, 255u, 1000u, 1024u, 2047u, 2048u, 4096u, 65535u, 65537u,
                           1000003u, (1u << 30) + 7u, (1u << 31) - 1u};
  long bad = 0;
  for (uint32_t d : divs) {
    hc::FastDivmod f(d);
    for (uint32_t n = 0; n < 2000000u; ++n) bad += f.div(n) != n / d;
    for (uint32_t k = 0; k < 2000000u; ++k) {
      const uint32_t n = 0x7fffffffu - k;
      bad += f.div(n) != n / d;
    }
    for (uint64_t n = d - 1; n < 0x80000000ull; n += d) {   // around multiples of d
      bad += f.div((uint32_t)n) != (uint32_t)(n / d);
      if (n + 1 < 0x80000000ull) bad += f.div((uint32_t)n + 1) != (uint32_t)((n + 1) / d);
      if (d < 512) n += d * 4093ull;                         // sampled for small divisors
    }
  }
  std::printf("%ld\n", bad);
  return bad != 0;
}
"""


def test_fastdiv_matches_integer_division():
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    with tempfile.TemporaryDirectory() as td:
        src = os.path.join(td, "t.cc")
        exe = os.path.join(td, "t")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run([gxx, "-O2", "-std=c++17", "-I",
                        os.path.join(ROOT, "kv_cache_quantization_hc_gb300", "csrc"), src, "-o", exe],
                       check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0 and r.stdout.strip() == "0", r.stdout + r.stderr
