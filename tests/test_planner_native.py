"""The weight pass's stage walker and activation windows on the CPU.

tests/native/gvm_plan_check.cu includes the kernel header and drives its
__host__ __device__ functions (the stage walker and the window function the
kernel itself runs) over 400 random launches: ragged widths, 1-8 activation
rows, 1-8 ops of 1-3 segments, the 8- and 16-warp layouts and small grids.
It checks stage coverage and order, window coverage, disjointness, budget
and plane stride, and that the device's rerun of the window function with
the host's computed size stages the same windows.  It also runs the
staging loops' index helpers (the column walk's forward-only window cursor
and the small-window item split) for every thread of a 256- and a
512-thread CTA and checks that each staged (window, float4 column, row) is
visited exactly once.  Compiled with nvcc; no GPU.
"""
import os
import subprocess

from layer_drafting_draft_b300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "layer_drafting_draft_b300", "csrc")


def test_walker_and_windows(tmp_path):
    exe = str(tmp_path / "gvm_plan_check")
    cmd = [build.nvcc(), *build.ARCH, "-std=c++17", "--expt-relaxed-constexpr", "-O2", "-I", CSRC,
           "-o", exe, os.path.join(HERE, "native", "gvm_plan_check.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr[-3000:]
    assert "0 failed checks" in r.stdout


def test_tensor_core_pass_layout_and_units(tmp_path):
    """tests/native/tc_plan_check.cu drives tc_layout and tc_unit (the
    planner's and the kernel's own functions) over 3000 random launches:
    row chunks, stages, shared memory for one or two CTAs per SM, tensor-
    memory columns, cluster size, and that the grid's CTAs partition every
    tile's k-blocks in rank order.  Compiled with nvcc; no GPU."""
    exe = str(tmp_path / "tc_plan_check")
    cmd = [build.nvcc(), *build.ARCH, "-std=c++17", "--expt-relaxed-constexpr", "-O2", "-I", CSRC,
           "-o", exe, os.path.join(HERE, "native", "tc_plan_check.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr[-3000:]
    assert " 0 failed checks" in r.stdout
