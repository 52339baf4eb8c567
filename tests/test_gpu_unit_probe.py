"""Builds and runs the sm_103a unit probe: exact tcgen05 operand conventions (bf16/e4m3, d 64/128,
SMEM and TMEM A operands) and the per-SM MUFU / FFMA / MMA rates the kernel design relies on."""
import os
import re
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "exact_attention_13_gb300", "csrc", "unit_probe.cu")


def test_unit_probe(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "unit_probe")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-o", exe, SRC], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300).stdout
    print(out)
    assert "PROBE PASS" in out
    m = re.search(r"\[rate\] ex2\.f32\s+([\d.]+) instr/clk/SM", out)
    assert m and float(m.group(1)) >= 15.5
    m = re.search(r"mma SS bf16 M128 N128 K16\s+([\d.]+) cycles/mma", out)
    assert m and float(m.group(1)) < 70
    # the attention order issued one product per asm block, as the kernels issue it, keeps the
    # tensor core at its full rate
    m = re.search(r"chains: attention order \+ commit\s+([\d.]+) cycles/mma\s+err=0", out)
    assert m and float(m.group(1)) < 70
