"""The stream kernel's launch shapes for every accepted head count (CPU).

Compiles tests/launch_shapes_check.cu, a host-only program over the
library's own headers that evaluates the same constexpr functions the
launches use, and runs it: it launches nothing on a GPU."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


@pytest.mark.skipif(not (os.path.exists(NVCC) or shutil.which("nvcc")), reason="nvcc not available")
def test_stream_kernel_shapes_for_every_head_count(tmp_path):
    exe = str(tmp_path / "launch_shapes_check")
    cmd = [NVCC if os.path.exists(NVCC) else "nvcc", "-std=c++17", "--expt-relaxed-constexpr",
           "-gencode", "arch=compute_103a,code=sm_103a",
           "-I", os.path.join(ROOT, "diffusion_transformer_joint_txt_b300", "csrc"), "-I", os.path.join(ROOT, "include"),
           "-o", exe, os.path.join(HERE, "launch_shapes_check.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
    for name in ("Bf16Rows", "AmaxRows", "E4m3Rows"):
        assert "%s: 0 bad of 192 head counts" % name in r.stdout, r.stdout
