"""Host-side check of the tcgen05 GEMM's static tile schedule (no GPU).

The kernel walks a flat tile index and decodes it into (split, batch, pair of 128-row tiles,
n-tile).  `tests/host/tile_schedule_check.cu` compiles that decode as host code and checks, over
plain, split-K, grouped and row-batched causal shapes, that each tile a launch must compute is
visited exactly once by both CTAs of a pair and nothing else is; for causal attention scores (mode
1) that is the tiles on or below the diagonal.  `tests/host/attn_schedule_check.cu` does the same for the
work-item order of the attention kernels without materialised scores.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _nvcc():
    from rank_bottleneck_block_gb300 import build

    try:
        return build.nvcc()
    except RuntimeError:
        return None


def test_tile_schedule_visits_each_tile_once(tmp_path):
    nvcc = _nvcc()
    if nvcc is None or shutil.which(nvcc) is None and not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "tile_schedule_check")
    src = os.path.join(HERE, "host", "tile_schedule_check.cu")
    cc = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                         "--expt-relaxed-constexpr", "-O2", "-o", exe, src], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr[-2000:]
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.startswith("ok"), run.stdout[-2000:]


def test_attention_item_order_visits_each_item_once(tmp_path):
    nvcc = _nvcc()
    if nvcc is None or shutil.which(nvcc) is None and not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "attn_schedule_check")
    src = os.path.join(HERE, "host", "attn_schedule_check.cu")
    cc = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                         "--expt-relaxed-constexpr", "-O2", "-o", exe, src], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr[-2000:]
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.startswith("ok"), run.stdout[-2000:]
