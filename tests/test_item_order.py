"""The persistent kernels' work-item order (banded_item and cost_band_count in
csrc/cpattn_internal.h), compiled for the host and checked without a GPU:
every item index maps to exactly one (group, rank, sub) item, the band counts
of the named workloads are the ones the kernels were measured with, and the
snake deal of the persistent CTAs over the banded list gives every CTA about
the same number of tiles (the tiles an item visits under the causal rule)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "context_causal_attention_zigzag_gb300", "csrc")
CUDA_INCLUDE = "/usr/local/cuda/include"

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <vector>
#include "cpattn_internal.h"
using namespace cpattn;

int main(int argc, char** argv) {
  if (argc >= 2 && !strcmp(argv[1], "bijection")) {
    const int groups[] = {1, 3, 8, 32}, ranks[] = {1, 2, 5, 10, 33, 128, 1024};
    const int inners[] = {1, 4}, grids[] = {1, 7, 152}, caps[] = {0, 4};
    int shapes = 0;
    for (int ng : groups) for (int nr : ranks) for (int inner : inners) for (int grid : grids)
      for (int cap : caps) {
        const int n = ng * nr * inner;
        std::vector<int> seen(n, 0);
        for (int i = 0; i < n; ++i) {
          int g, r, s;
          banded_item(i, ng, nr, inner, grid, cap, g, r, s);
          if (g < 0 || g >= ng || r < 0 || r >= nr || s < 0 || s >= inner) return 2;
          if (seen[(g * nr + r) * inner + s]++) return 3;
        }
        ++shapes;
      }
    printf("%d\n", shapes);
    return 0;
  }
  if (argc == 6 && !strcmp(argv[1], "bands")) {
    printf("%d\n", cost_band_count(atoi(argv[2]), atoi(argv[3]), atoi(argv[4]), atoi(argv[5])));
    return 0;
  }
  if (argc == 7 && !strcmp(argv[1], "ranks")) {  // the rank of every item index, in order
    const int ng = atoi(argv[2]), nr = atoi(argv[3]), inner = atoi(argv[4]);
    const int grid = atoi(argv[5]), cap = atoi(argv[6]);
    for (int i = 0; i < ng * nr * inner; ++i) {
      int g, r, s;
      banded_item(i, ng, nr, inner, grid, cap, g, r, s);
      printf("%d\n", r);
    }
    return 0;
  }
  return 1;
}
"""


@pytest.fixture(scope="module")
def order_tool(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INCLUDE, "cuda_runtime.h")):
        pytest.skip("needs g++ and the CUDA headers")
    d = tmp_path_factory.mktemp("item_order")
    src, exe = d / "order.cpp", d / "order"
    src.write_text(PROGRAM)
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    "-I", CUDA_INCLUDE, str(src), "-o", str(exe)], check=True)
    return lambda *args: subprocess.run([str(exe)] + [str(a) for a in args], check=True,
                                        capture_output=True, text=True).stdout


def test_banded_item_is_a_bijection(order_tool):
    assert int(order_tool("bijection")) == 4 * 7 * 2 * 3 * 2


GRID = 152


@pytest.mark.parametrize("name,per_group,nrank,cap,bands", [
    # S=131072, H=32, Hkv=8: forward (query pairs x 4 heads), dK/dV (K/V tiles), dQ
    ("S=131072 forward", 512 * 4, 512, 0, 2),
    ("S=131072 dK/dV", 1024, 1024, 4, 4),
    ("S=131072 dQ", 1024 * 4, 1024, 0, 2),
    # S=32768 forward, S=8192 forward (H = Hkv = 32), S=16384 dK/dV (capped heads)
    ("S=32768 forward", 128 * 4, 128, 0, 8),
    ("S=8192 forward", 32, 32, 0, 32),
    ("S=16384 dK/dV", 128, 128, 4, 2),
])
def test_band_counts_of_named_workloads(order_tool, name, per_group, nrank, cap, bands):
    assert int(order_tool("bands", per_group, nrank, GRID, cap)) == bands, name


def snake_max_over_mean(costs, grid=GRID):
    load = [0] * grid
    for i, c in enumerate(costs):
        k, j = divmod(i, grid)
        load[(grid - 1 - j) if k & 1 else j] += c
    return max(load) / (sum(costs) / grid)


@pytest.mark.parametrize("name,ng,nr,inner,cap,cost,bound", [
    # costs: K/V tiles a query pair visits, query tiles that see a K/V tile,
    # K/V tiles a query tile visits (causal, natural order; rank 0 the largest)
    ("S=131072 forward", 8, 512, 4, 0, lambda r, n: 2 * (n - 1 - r) + 2, 1.006),
    ("S=131072 dK/dV", 32, 1024, 1, 4, lambda r, n: n - r, 1.006),
    ("S=131072 dQ", 8, 1024, 4, 0, lambda r, n: n - r, 1.006),
    ("S=8192 forward", 32, 32, 1, 0, lambda r, n: 2 * (n - 1 - r) + 2, 1.02),
])
def test_snake_deal_balances_the_banded_list(order_tool, name, ng, nr, inner, cap, cost, bound):
    ranks = [int(x) for x in order_tool("ranks", ng, nr, inner, GRID, cap).split()]
    assert len(ranks) == ng * nr * inner
    ratio = snake_max_over_mean([cost(r, nr) for r in ranks])
    assert ratio <= bound, (name, ratio)
