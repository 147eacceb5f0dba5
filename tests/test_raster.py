"""Host-side check of the GEMM raster (gemm_common.cuh, TileSched): for a
range of tile grids and group heights the walk visits every tile exactly
once, stays inside the grid, and each raster group starts on the tile column
its predecessor ended on (odd groups walk the columns backwards, so the
columns of B read last are read again first, while still in L2).

The scheduler is a __host__ __device__ function, so a small host program
compiled with nvcc calls the library's own code; no GPU is needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_scaled_quantized_mx_gb300", "csrc")
BUILD = os.path.join(ROOT, "block_scaled_quantized_mx_gb300", "_build")

HARNESS = r"""
#include <cstdio>
#include <vector>
#include "gemm_common.cuh"

int main() {
  long checked = 0;
  int bad = 0;
  const int ns[] = {1, 2, 3, 7, 32, 33};
  const int gs[] = {1, 2, 3, 8, 16, 32, 64};
  for (int num_m = 1; num_m <= 40; ++num_m)
    for (int num_n : ns)
      for (int group : gs) {
        mxk::TileSched s;
        s.num_m = num_m;
        s.num_n = num_n;
        s.total = num_m * num_n;
        s.group = group;
        std::vector<int> seen(s.total, 0);
        int prev_nb = -1;
        for (int t = 0; t < s.total; ++t) {
          int mb = -1, nb = -1;
          s.tile(t, mb, nb);
          ++checked;
          if (mb < 0 || mb >= num_m || nb < 0 || nb >= num_n) {
            if (bad++ < 5) std::printf("out of grid: %d %d %d t=%d -> %d %d\n",
                                       num_m, num_n, group, t, mb, nb);
            continue;
          }
          ++seen[mb * num_n + nb];
          // a new group (its first tile) starts on the column the last one ended on
          if (t > 0 && t % (group * num_n) == 0 && nb != prev_nb) {
            if (bad++ < 5) std::printf("group start: %d %d %d t=%d nb=%d prev=%d\n",
                                       num_m, num_n, group, t, nb, prev_nb);
          }
          prev_nb = nb;
        }
        for (int i = 0; i < s.total; ++i)
          if (seen[i] != 1 && bad++ < 5)
            std::printf("tile %d of %d x %d (group %d) seen %d times\n", i, num_m, num_n,
                        group, seen[i]);
      }
  std::printf("checked %ld bad %d\n", checked, bad);
  return bad != 0;
}
"""


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


def test_raster_walk_is_a_permutation_with_backward_odd_groups():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(BUILD, "raster_check.cu")
    exe = os.path.join(BUILD, "raster_check")
    with open(src, "w") as f:
        f.write(HARNESS)
    subprocess.check_call([nvcc, "-std=c++17", "-O1", "-gencode",
                           "arch=compute_103a,code=sm_103a", "-I", CSRC,
                           "-I", os.path.join(ROOT, "include"), src, "-o", exe])
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    assert "bad 0" in out.stdout
