"""GPU parity of the key-split path (fa_fwd_split + merge) against the fp64 oracle."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle
from tests.parity import compare
from workloads import random_inputs, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def ea():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_13_gb300 as mod

    mod.lib()
    mod.device_status(clear=True)
    yield mod
    assert mod.device_status(clear=True) == 0


def run(ea, inp, causal, splits, workspace=None):
    q, k, v = (getattr(inp, n).to(DEV) for n in "qkv")
    o, lse = ea.fwd(q, k, v, causal=causal, num_splits=splits, workspace=workspace,
                    descale=(inp.descale_q, inp.descale_k, inp.descale_v))
    torch.cuda.synchronize()
    return o, lse


CASES = [
    # (B, H, N, d, dtype, causal, splits)
    (1, 2, 300, 128, "bf16", False, 2),
    (1, 2, 300, 128, "bf16", True, 2),
    (1, 1, 1000, 64, "bf16", True, 3),
    (2, 1, 777, 128, "bf16", False, 5),
    (1, 1, 200, 128, "bf16", True, 5),      # more splits than key blocks: empty partials
    (1, 1, 1, 64, "bf16", False, 2),
    (1, 2, 640, 128, "e4m3", False, 3),
    (1, 2, 513, 128, "e4m3", True, 2),
    (1, 1, 2048, 64, "bf16", False, 16),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,splits", CASES,
                         ids=[f"B{b}H{h}N{n}d{d}-{t}-{'causal' if c else 'full'}-s{s}"
                              for b, h, n, d, t, c, s in CASES])
def test_split_parity(ea, B, H, N, d, dtype, causal, splits):
    inp = random_inputs(B, H, N, d, dtype, seed=5000 + N + d + splits + int(causal))
    o, lse = run(ea, inp, causal, splits)
    o_ref, l_ref = oracle.attention_fwd_inputs(inp, 1.0 / math.sqrt(d), causal)
    compare(o, lse, o_ref, l_ref, dtype, f"split {splits}")


def test_split_matches_unsplit_and_ignores_workspace_contents(ea):
    """A workspace full of NaN on entry changes nothing; split and unsplit agree within the
    parity tolerance (each split rounds its P to bf16 relative to its own running max, so the
    two differ by a few bf16 ulps, not bit for bit)."""
    inp = random_inputs(1, 3, 1500, 128, "bf16", seed=5101)
    o1, l1 = run(ea, inp, True, 1)
    nbytes = ea.split_workspace_bytes(1, 3, 1500, 128, 4)
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device=DEV)
    o4, l4 = run(ea, inp, True, 4, workspace=ws)
    o_ref, l_ref = oracle.attention_fwd_inputs(inp, 1 / math.sqrt(128), True)
    compare(o4, l4, o_ref, l_ref, "bf16", "split 4, NaN workspace")
    assert float((o4.float() - o1.float()).abs().max()) < 1e-2
    assert float((l4 - l1).abs().max()) < 1e-4


def test_split_full_size_sampled(ea):
    """A long single-sequence shape where splitting matters (64 CTAs without it)."""
    B, H, N, d = 1, 2, 16384, 128
    inp = random_inputs(B, H, N, d, "bf16", seed=5202)
    o, lse = run(ea, inp, False, 4)
    rows = sample_rows(N, 5202)
    o_ref, l_ref = oracle.attention_fwd_inputs(inp, 1 / math.sqrt(d), False, rows=rows)
    compare(o[:, :, rows], lse[:, :, rows], o_ref, l_ref, "bf16", "split 4 sampled")
    oc, lc = run(ea, inp, True, 3)
    o_ref, l_ref = oracle.attention_fwd_inputs(inp, 1 / math.sqrt(d), True, rows=rows)
    compare(oc[:, :, rows], lc[:, :, rows], o_ref, l_ref, "bf16", "split 3 causal sampled")
