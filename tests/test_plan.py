"""Launch planning of the persistent MoE kernels (csrc/plan.h), checked on the
host with injected SM counts and occupancies: the header is plain C++, so it
is compiled here with g++ into a small program that prints the decisions."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_diffusion_moe_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "plan.h"
using namespace clover::plan;
int main() {
  // tokens, experts, sms -> fused?
  const int cases[][3] = {{32, 256, 152}, {33, 256, 152}, {1, 256, 152}, {32, 256, 32}, {32, 256, 31},
                          {8, 16, 152}, {8, 16, 7}, {8, 16, 8}, {1, 256, 20}, {256, 256, 152}, {32, 300, 32}};
  for (auto& c : cases) printf("fused %d %d %d %d\n", c[0], c[1], c[2], moe_fused(c[0], c[1], c[2]) ? 1 : 0);
  // sms, resident per SM -> grid
  const int grids[][2] = {{152, 1}, {152, 2}, {152, 0}, {0, 1}, {20, 1}, {1, 1}};
  for (auto& g : grids) printf("grid %d %d %d\n", g[0], g[1], persistent_grid(g[0], g[1]));
  return 0;
}
"""


@pytest.fixture(scope="module")
def decisions(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("plan")
    src = d / "plan_check.cpp"
    src.write_text(PROGRAM)
    exe = d / "plan_check"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    fused, grid = {}, {}
    for line in out.splitlines():
        f = line.split()
        if f[0] == "fused":
            fused[tuple(map(int, f[1:4]))] = int(f[4])
        else:
            grid[tuple(map(int, f[1:3]))] = int(f[3])
    return fused, grid


def test_fused_layer_kernel_takes_one_block_at_full_sm_count(decisions):
    fused, _ = decisions
    assert fused[(32, 256, 152)] == 1      # the Clover block of 32 on a GB300
    assert fused[(1, 256, 152)] == 1
    assert fused[(8, 16, 152)] == 1        # the tiny configuration
    assert fused[(33, 256, 152)] == 0      # more than 32 tokens: standalone kernels
    assert fused[(256, 256, 152)] == 0


def test_fused_layer_kernel_needs_enough_ctas(decisions):
    """With fewer SMs (a partitioned GPU) the fused kernel needs one CTA per
    token for the top-k and at most 8 router rows per CTA; otherwise the
    standalone path takes the call."""
    fused, _ = decisions
    assert fused[(32, 256, 32)] == 1       # 8 router rows per CTA, 32 CTAs for 32 tokens
    assert fused[(32, 256, 31)] == 0       # 9 rows per CTA and one CTA short
    assert fused[(8, 16, 7)] == 0          # 7 CTAs cannot select 8 tokens
    assert fused[(8, 16, 8)] == 1
    assert fused[(1, 256, 20)] == 0        # 13 router rows per CTA
    assert fused[(32, 300, 32)] == 0


def test_persistent_grid_requires_residency(decisions):
    _, grid = decisions
    assert grid[(152, 1)] == 152           # one CTA per SM
    assert grid[(152, 2)] == 152           # the kernels are written for one CTA per SM
    assert grid[(20, 1)] == 20             # fewer SMs: a smaller grid, every CTA resident
    assert grid[(1, 1)] == 1
    assert grid[(152, 0)] == 0             # does not fit on an SM: rejected, not launched
    assert grid[(0, 1)] == 0
