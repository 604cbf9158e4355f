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


DECODE_HARNESS = r"""
#include <cstdio>
#include <vector>
#include "fa_schedule.h"
// The task decodings the kernels instantiate (plain division for the
// non-causal long-task kernels, multiply and shift elsewhere) must agree on
// every task of the balanced static orders.
static bool same(const fa::Task& a, const fa::Task& b) {
  return a.b == b.b && a.g == b.g && a.mb == b.mb && a.kvh == b.kvh && a.pos0[0] == b.pos0[0] &&
         a.pos0[1] == b.pos0[1] && a.n[0] == b.n[0] && a.n[1] == b.n[1] && a.nmax == b.nmax &&
         a.ksplit == b.ksplit && a.kend == b.kend && a.kshift == b.kshift && a.sq == b.sq;
}
int main() {
  struct Case { int B, Hq, Hkv, Sq, Sk, causal; };
  const Case cases[] = {
    {4, 16, 16, 8192, 8192, 0}, {4, 16, 16, 8192, 8192, 1}, {32, 16, 16, 1024, 1024, 1}, {1, 16, 16, 32768, 32768, 1},
    {4, 32, 8, 8192, 8192, 1}, {4, 32, 1, 8192, 8192, 1}, {2, 16, 16, 16384, 16384, 1}, {1, 4, 4, 1000, 1000, 0},
    {1, 3, 3, 384, 640, 0}, {2, 5, 5, 700, 1500, 0}, {1, 4, 2, 1000, 1500, 1}, {3, 6, 2, 777, 1300, 1},
    {2, 12, 4, 2048, 2048, 1}, {5, 7, 7, 300, 900, 1}, {1, 2, 2, 4608, 4608, 1}, {2, 4, 4, 2048, 2048, 1}};
  const int grids[] = {152, 148, 132, 97, 13, 11, 7, 5, 3, 2};
  long long checked = 0;
  for (const Case& c : cases) {
    for (int G : grids) {
      fa::Problem p = fa::make_problem(c.B, c.Hq, c.Hkv, c.Sq, c.Sk, 128, 128, c.causal, 64ll << 20, 0);
      const fa::Problem plain = p;
      fa::set_balance(p, G);
      // every (unit, tile, key block) visited exactly once, with the plain order's blocks
      const int units = p.B * p.groups, tiles = 2 * p.mblocks;
      std::vector<int> seen(static_cast<size_t>(units) * tiles * p.kv_blocks, 0), want(seen.size(), 0);
      auto mark = [&](std::vector<int>& v, const fa::Task& k, int s, int first, int n) {
        const int tile = k.pos0[s] / p.pos_per_tile;
        for (int j = first; j < first + n; ++j)
          ++v[(static_cast<size_t>(k.b * p.groups + k.g) * tiles + tile) * p.kv_blocks + j];
      };
      for (int t = 0; t < static_cast<int>(plain.num_tasks); ++t) {
        const fa::Task k = fa::decode_task_k<-1, false, true, true>(plain, t);
        for (int s = 0; s < 2; ++s) mark(want, k, s, 0, k.n[s]);
      }
      for (int t = 0; t < static_cast<int>(p.num_tasks); ++t) {
        const fa::Task k = fa::decode_task_k<-1, false, true, true>(p, t);
        if (k.ksplit) {
          mark(seen, k, 0, 0, k.n[0]);
          mark(seen, k, 1, k.ksplit, k.n[1]);
        } else {
          for (int s = 0; s < 2; ++s) mark(seen, k, s, 0, k.n[s]);
        }
      }
      if (seen != want) {
        std::printf("FAIL coverage B%d H%d/%d S%d/%d c%d G%d\n", c.B, c.Hq, c.Hkv, c.Sq, c.Sk, c.causal, G);
        return 1;
      }
      for (size_t i = 0; i < want.size(); ++i)
        if (want[i] > 1) { std::printf("FAIL plain order visits a cell twice\n"); return 1; }
      for (int t = 0; t < static_cast<int>(p.num_tasks); ++t) {
        fa::Task ref = fa::decode_task_k<-1, false, true, true>(p, t);
        fa::Task a = c.causal ? fa::decode_task_k<1, true, false, true>(p, t)
                              : fa::decode_task_k<-1, false, true, false>(p, t);
        fa::Task d = c.causal ? fa::decode_task_k<1, true, false, true>(p, t)
                              : fa::decode_task_k<0, true, true, false>(p, t);
        if (!same(ref, a) || !same(ref, d)) {
          std::printf("FAIL case B%d H%d/%d S%d/%d c%d G%d t%d\n", c.B, c.Hq, c.Hkv, c.Sq, c.Sk, c.causal, G, t);
          return 1;
        }
        ++checked;
      }
    }
  }
  std::printf("ok %lld tasks\n", checked);
  return 0;
}
"""


def test_kernel_decodings_agree_on_balanced_orders(tmp_path):
    src = str(tmp_path / "d.cpp")
    exe = str(tmp_path / "d")
    open(src, "w").write(DECODE_HARNESS)
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-I", CSRC, "-o", exe, src])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout[-2000:]
    assert out.stdout.startswith("ok")
