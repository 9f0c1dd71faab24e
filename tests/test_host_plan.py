"""Host-side work planning of the decode kernel, compiled with the host C++
compiler and checked on the CPU over many random sizes.

RunSplit (csrc/internal.h) cuts the T work items of a decode launch
(128-token tiles) into one contiguous run per CTA.  The split-KV workspace is
sized from its promise that a unit of n consecutive items touches at most
ceil(n / min_run) + 1 runs, i.e. leaves at most that many partial results
(the split-KV partition of the decode pages).  These checks pin that promise
and the runs' coverage, independently of any GPU.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_gqa_07_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

HARNESS = r"""
#include <cstdio>
#include <random>
#include <set>

#include "internal.h"

using qattn::RunSplit;

static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fails++ < 10) std::printf(__VA_ARGS__); } } while (0)

int main() {
  std::mt19937_64 rng(20261202);
  long units_checked = 0;
  for (int it = 0; it < 4000; ++it) {
    const int P = 1 + static_cast<int>(rng() % 320);
    const int min_run = 1 + static_cast<int>(rng() % 10);
    const int T = 1 + static_cast<int>(rng() % (it % 2 ? 6000 : 600));
    const RunSplit s{T, P, min_run};
    CHECK(s.begin(0) == 0, "begin(0) T=%d P=%d m=%d\n", T, P, min_run);
    CHECK(s.begin(P) == T, "begin(P) T=%d P=%d m=%d\n", T, P, min_run);
    for (int k = 0; k < P; ++k) {
      const int b0 = s.begin(k), b1 = s.begin(k + 1);
      CHECK(b0 <= b1, "order k=%d T=%d P=%d m=%d\n", k, T, P, min_run);
      if (s.balanced())
        CHECK(b1 - b0 >= min_run, "short run k=%d T=%d P=%d m=%d\n", k, T, P, min_run);
      else
        CHECK(b1 - b0 == min_run || b1 == T, "run k=%d T=%d P=%d m=%d\n", k, T, P, min_run);
      for (int u = b0; u < b1; ++u)
        CHECK(s.cta_of(u) == k, "cta_of(%d)=%d not %d T=%d P=%d m=%d\n", u, s.cta_of(u), k,
              T, P, min_run);
    }
    // Units: consecutive random lengths over [0, T), as sequences' chunk
    // ranges are laid out in the work list.
    for (int u0 = 0; u0 < T;) {
      const int n = 1 + static_cast<int>(rng() % (1 + (rng() % 4 == 0 ? T : 64)));
      const int u1 = u0 + n < T ? u0 + n : T;
      std::set<int> runs;
      for (int u = u0; u < u1; ++u) runs.insert(s.cta_of(u));
      const int len = u1 - u0;
      const int bound = (len + min_run - 1) / min_run + 1;
      CHECK(static_cast<int>(runs.size()) <= bound, "unit [%d,%d) touches %d runs > %d T=%d "
            "P=%d m=%d\n", u0, u1, static_cast<int>(runs.size()), bound, T, P, min_run);
      ++units_checked;
      u0 = u1;
    }
  }
  // The workspace's part bound covers the runs a unit of L tokens can meet
  // (128-token tiles, runs of at least kTcMinTilesPerCta tiles).
  for (int L = 1; L <= 70000; ++L) {
    const int tiles = (L + qattn::kTcTileTokens - 1) / qattn::kTcTileTokens;
    const int parts = (tiles + qattn::kTcMinTilesPerCta - 1) / qattn::kTcMinTilesPerCta + 1;
    CHECK(parts <= qattn::decode_max_parts(L), "L=%d: %d parts > workspace bound\n", L, parts);
  }
  std::printf("%s %ld\n", fails ? "FAIL" : "ok", units_checked);
  return fails ? 1 : 0;
}
"""


def test_run_split_covers_and_bounds_parts(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None or not os.path.isdir(CUDA_INC):
        pytest.skip("no host C++ compiler or CUDA headers")
    src = tmp_path / "plan.cc"
    src.write_text(HARNESS)
    exe = tmp_path / "plan"
    subprocess.run([cxx, "-std=c++17", "-O2", "-Wall", "-I", CSRC, "-I", CUDA_INC, str(src),
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
    status, n = r.stdout.split()
    assert status == "ok" and int(n) > 10000
