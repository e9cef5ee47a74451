"""The u8 fast kernel's shared-memory layout, checked on the host for every
template width and height the fast path can take (tests/host_layout_check.cu,
compiled with nvcc as a host program; no GPU is used)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_fast_kernel_smem_layout(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "layout_check"
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "--expt-relaxed-constexpr",
                        "-gencode", "arch=compute_103a,code=sm_103a",
                        "-I", os.path.join(ROOT, "include"),
                        os.path.join(HERE, "host_layout_check.cu"), "-o", str(exe)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout[-3000:]
    assert "0 failures" in out.stdout
