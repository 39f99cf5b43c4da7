"""Host check of position rolling's rank digits (the table-entry arithmetic the
decode kernel and the table builder share): compiled from the library's own
header into a small host program.  For every digit width and many cache
sizes, each rank 0..C splits into per-level entries that index inside the
tables, fall in their level's block, and add back up to the rank."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kv_cache_eviction_03_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "h2o_internal.cuh"
using namespace h2o;
int main() {
  std::vector<int> sizes;
  for (int c = 1; c <= 300; ++c) sizes.push_back(c);
  for (int e = 4; e <= 16; ++e)
    for (int d = -2; d <= 2; ++d) sizes.push_back((1 << e) + d);
  sizes.push_back(410); sizes.push_back(1640); sizes.push_back(2048); sizes.push_back(65536);
  long long checked = 0;
  for (int C : sizes) {
    if (C < 1 || C > 65536) continue;
    for (int low = kRopeMinBits; low <= kRopeMaxBits; ++low)
      for (int hi = kRopeMinBits; hi <= kRopeMaxBits; ++hi) {
        const int levels = rope_levels_for(C, low, hi), entries = rope_entries_for(C, low, hi);
        if (levels < 1 || levels > 5) { printf("FAIL levels C=%d low=%d hi=%d: %d\n", C, low, hi, levels); return 1; }
        // the largest rank needs every level and no more
        const long long span = 1LL << (low + hi * (levels - 1));
        if (C >= span || (levels > 1 && C < (1LL << (low + hi * (levels - 2))))) {
          printf("FAIL span C=%d low=%d hi=%d levels=%d\n", C, low, hi, levels); return 1;
        }
        for (int r = 0; r <= C; ++r) {
          long long back = 0;
          for (int l = 0; l < levels; ++l) {
            const int e = rope_entry(r, l, low, hi);
            const int base = l == 0 ? 0 : (1 << low) + (1 << hi) * (l - 1);
            const int width = l == 0 ? (levels == 1 ? C + 1 : (1 << low)) : (1 << hi);
            if (e < 0 || e >= entries || e < base || e >= base + width) {
              printf("FAIL entry C=%d low=%d hi=%d r=%d l=%d e=%d entries=%d\n", C, low, hi, r, l, e, entries);
              return 1;
            }
            const long long w = l == 0 ? 1 : (1LL << (low + hi * (l - 1)));
            back += (long long)(e - base) * w;
          }
          if (back != r) { printf("FAIL sum C=%d low=%d hi=%d r=%d back=%lld\n", C, low, hi, r, back); return 1; }
          ++checked;
        }
      }
  }
  printf("OK %lld\n", checked);
  return 0;
}
"""


def test_rank_digits_reconstruct_every_rank():
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "digits.cu"), os.path.join(d, "digits")
        with open(src, "w") as f:
            f.write(PROGRAM)
        r = subprocess.run([nvcc, "-std=c++17", "-O2", "-I", CSRC, "-I", INCLUDE, src, "-o", exe],
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-3000:]
        out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout[-2000:]
