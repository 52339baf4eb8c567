"""Builds and runs tests/gpu_probe/tcgen05_conventions.cu: the tcgen05 operand conventions the
attention kernels use (S = Q K^T from K-major swizzled shared memory, O = P V with P in tensor
memory and V MN-major; bf16 and e4m3; head dims 64 and 128) must reproduce the CPU's results
exactly on small-integer data."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gpu_probe",
                   "tcgen05_conventions.cu")


def test_tcgen05_operand_conventions_exact(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "tcgen05_conventions")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-o", exe, SRC], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    print(res.stdout)
    assert res.returncode == 0 and "PROBE PASS" in res.stdout
    assert res.stdout.count("max_err=0 bad=0") == 8  # S and O of four cases
