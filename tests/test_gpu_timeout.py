"""Failure detection without a GPU fault: a test build of the library whose producers stop after
the CTA's fixed tiles (forward: the Q tiles; backward: K_j, V_j and Q_i, dO_i) makes each kernel's
first streamed wait run out.  The kernels must give up within their wait limit (50 ms in the test
build), record FA_ERR_DEVICE_TIMEOUT in the status word, free their tensor memory and exit, and
the CUDA context must stay usable: the regular library still computes correct results afterwards.
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


@pytest.fixture(scope="module")
def stall(tmp_path_factory):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    lib_path = str(tmp_path_factory.mktemp("stall") / "libexattn_stall.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-DEXATTN_INJECT_STALL=1",
                    "-DEXATTN_WAIT_LIMIT_NS=50000000ull", "-o", lib_path, SRC], check=True)
    return ctypes.CDLL(lib_path)


def test_wait_timeout_sets_status_and_context_survives(stall):
    import torch

    import exact_attention_13_gb300 as ea
    from oracle import oracle
    from tests.parity import compare
    from workloads import random_inputs

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


def test_bwd_wait_timeout_sets_status_and_context_survives(stall):
    import torch

    import exact_attention_13_gb300 as ea
    from oracle import oracle
    from workloads import random_bwd_inputs

    res, args = ea.SIGNATURES["fa_bwd"]
    stall.fa_bwd.restype, stall.fa_bwd.argtypes = res, args
    dev = torch.device("cuda:0")
    B, H, N, d = 1, 2, 300, 128
    inp = random_bwd_inputs(B, H, N, d, seed=405)
    q, k, v, do = (getattr(inp, n).to(dev) for n in ("q", "k", "v", "do"))
    o, lse = ea.fwd(q, k, v, causal=True)
    grads = [torch.full_like(q, 3.0) for _ in range(3)]
    ws = torch.empty(ea.bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = stall.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      do.data_ptr(), *(g.data_ptr() for g in grads), B, H, N, d,
                      1.0 / math.sqrt(d), 1, ws.data_ptr(), ws.numel(), status.data_ptr(), stream)
    assert rc == ea.FA_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == ea.FA_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0, elapsed
    # an aborted kernel writes no gradient
    for g in grads:
        assert bool((g == 3.0).all())

    # the context is still healthy: the regular library computes correct gradients
    dq, dk, dv = ea.bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    ref = oracle.get().attention_bwd(*(inp.raw(n) for n in ("q", "k", "v", "do")),
                                     1.0 / math.sqrt(d), True, "bf16")
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        want = ref[name]
        err = np.abs(got.double().cpu().numpy() - want).max()
        assert err <= 3e-2 * np.abs(want).max() + 1e-3, (name, err)
    assert ea.device_status(clear=True) == 0
