"""Failure detection without a GPU fault: a test build of the library whose producer stops after
the Q tiles makes the kernel's first K/V wait run out.  The kernel must give up within its wait
limit, record FA_ERR_DEVICE_TIMEOUT in the status word, free its tensor memory and exit, and the
CUDA context must stay usable: the regular library still computes correct attention afterwards.
"""
import ctypes
import math
import os
import shutil
import subprocess
import time

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "exact_attention_13_gb300", "csrc", "fa_api.cu")


def test_wait_timeout_sets_status_and_context_survives(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_13_gb300 as ea
    from oracle import oracle
    from tests.parity import compare
    from workloads import random_inputs

    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    lib_path = str(tmp_path / "libexattn_stall.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-DEXATTN_INJECT_STALL=1",
                    "-DEXATTN_WAIT_LIMIT_NS=50000000ull", "-o", lib_path, SRC], check=True)
    stall = ctypes.CDLL(lib_path)
    res, args = ea.SIGNATURES["fa_fwd_ex"]
    stall.fa_fwd_ex.restype, stall.fa_fwd_ex.argtypes = res, args

    dev = torch.device("cuda:0")
    B, H, N, d = 1, 2, 300, 128
    q = torch.randn(B, H, N, d, device=dev).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    opts = ea.FwdOpts(1.0, 1.0, 1.0, status.data_ptr())
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    rc = stall.fa_fwd_ex(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         B, H, N, d, 1.0 / math.sqrt(d), 0, ea.FA_DTYPE_BF16, ctypes.byref(opts),
                         stream)
    assert rc == ea.FA_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == ea.FA_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0, elapsed

    # the context is still healthy: the regular library computes correct attention
    inp = random_inputs(1, 2, 300, 128, "bf16", seed=404)
    qq, kk, vv = (getattr(inp, n).to(dev) for n in "qkv")
    out, l2 = ea.fwd(qq, kk, vv, causal=True)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_fwd_inputs(inp, 1 / math.sqrt(128), True)
    compare(out, l2, o_ref, l_ref, "bf16", "after timeout")
    assert ea.device_status(clear=True) == 0
