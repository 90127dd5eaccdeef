"""Host check of the division-by-invariant-integer constants the fused decode
kernel uses to split global top-k positions by shard count and block size
(Granlund and Montgomery, "Division by invariant integers using
multiplication", 1994).  Compiles a small C++ program against the library's
internal header and compares (umulhi(n, m) + n) >> s with n / d for every
divisor up to 4096, edge values and random n < 2^31."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_mla_decode_dcp_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include <random>
#include "smla_internal.h"
int main() {
  std::mt19937_64 g(1);
  long bad = 0, checked = 0;
  for (uint32_t d = 1; d <= 4096; ++d) {
    const smla::FastDiv f = smla::make_fastdiv(d);
    auto q = [&](uint32_t n) {
      return uint32_t(((uint64_t(n) * f.mul >> 32) + n) >> f.shift);
    };
    const uint32_t top = 0x7fffffffu;
    const uint32_t edge[] = {0u, 1u, d - 1, d, d + 1, 2 * d - 1, 2 * d, top,
                             top - top % d, top - top % d - 1};
    for (uint32_t n : edge) {
      if (n > top) continue;
      ++checked;
      bad += q(n) != n / d;
    }
    for (int i = 0; i < 500; ++i) {
      const uint32_t n = uint32_t(g() & top);
      ++checked;
      bad += q(n) != n / d;
    }
  }
  std::printf("%ld %ld\n", checked, bad);
  return bad != 0;
}
"""


def _cuda_include():
    for root in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if root and os.path.exists(os.path.join(root, "include", "cuda_runtime.h")):
            return os.path.join(root, "include")
    return None


def test_fastdiv_constants_divide_exactly():
    gxx = shutil.which("g++")
    inc = _cuda_include()
    if gxx is None or inc is None:
        pytest.skip("needs g++ and the CUDA headers")
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "fastdiv.cpp")
        exe = os.path.join(tmp, "fastdiv")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run([gxx, "-O2", "-std=c++17", "-I", inc, "-I", CSRC, src, "-o", exe],
                       check=True, capture_output=True)
        out = subprocess.run([exe], capture_output=True, text=True)
    checked, bad = map(int, out.stdout.split())
    assert checked > 2_000_000 and bad == 0, out.stdout
