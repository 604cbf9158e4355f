"""The multiply-and-shift division of the task decoder (fa_schedule.h,
FastDiv) against plain integer division, compiled for the host from the same
header the kernel includes.  Covers every divisor up to 4096, powers of two
and their neighbours up to 2^31 - 1, and dividends at 0, around each multiple
boundary and at 2^31 - 1."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "exact_attention_forward_08_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <cstdint>
#include <vector>
#include "fa_schedule.h"
static int check(int d, long long n) {
  const fa::FastDiv f = fa::make_fastdiv(d);
  const int q = fa::fdiv(static_cast<int>(n), f);
  if (q != static_cast<int>(n / d)) { std::printf("FAIL d=%d n=%lld got %d\n", d, n, q); return 1; }
  return 0;
}
int main() {
  std::vector<int> ds;
  for (int d = 1; d <= 4096; ++d) ds.push_back(d);
  for (int e = 12; e <= 30; ++e) { ds.push_back((1 << e) - 1); ds.push_back(1 << e); ds.push_back((1 << e) + 1); }
  ds.push_back(2147483647); ds.push_back(2147483646); ds.push_back(1431655765); ds.push_back(715827883);
  const long long top = 2147483647LL;
  uint64_t x = 0x9E3779B97F4A7C15ull;
  long long checked = 0;
  for (int d : ds) {
    int bad = 0;
    for (long long n = 0; n < 3000 && n <= top; ++n) bad |= check(d, n);
    for (long long k = 1; k <= 64; ++k) {  // around multiples of d near the bottom and the top
      for (long long n : {k * d - 1, k * d, k * d + 1, (top / d - k) * d - 1, (top / d - k) * d, (top / d - k) * d + 1})
        if (n >= 0 && n <= top) bad |= check(d, n);
    }
    for (long long n = top - 3000; n <= top; ++n) bad |= check(d, n);
    for (int r = 0; r < 2000; ++r) {
      x ^= x << 13; x ^= x >> 7; x ^= x << 17;
      bad |= check(d, static_cast<long long>(x % 2147483648ull));
    }
    if (bad) return 1;
    checked += 1;
  }
  std::printf("ok %lld divisors\n", checked);
  return 0;
}
"""


def test_fastdiv_matches_integer_division(tmp_path):
    src = str(tmp_path / "h.cpp")
    exe = str(tmp_path / "h")
    open(src, "w").write(HARNESS)
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-I", CSRC, "-o", exe, src])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout[-2000:]
    assert out.stdout.startswith("ok")
