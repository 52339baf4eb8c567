"""GPU parity of the attention backward (fa_bwd) against the fp64 oracle's gradients.

The forward kernel supplies O and LSE (as a training step would); the oracle recomputes
everything from Q, K, V and dO itself.  Tolerance (derived from the arithmetic): P and dS enter
the tensor-core products rounded to bf16 (relative 2^-9 each), O enters D rounded to bf16, and
the gradients are rounded to bf16 on output, so each element may be off by a few 2^-9 of the
magnitude of its summands; the gate is |g - g_ref| <= 1e-2 max|g_ref| + half a bf16 ulp of
|g_ref| + a floor, per gradient tensor and head.  The floor covers gradients that vanish exactly
(a row with one visible key has dS = 0): D_i is formed from the bf16-rounded O, so dP_ij - D_i
carries up to 2^-8 sum_t |dO_it O_it| of rounding, which dQ multiplies by scale max|K| and dK by
scale max|Q|.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle
from tests.parity import bf16_half_ulp
from workloads import random_bwd_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
REL = 1e-2


@pytest.fixture(scope="module")
def ea():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_13_gb300 as mod

    mod.lib()
    mod.device_status(clear=True)
    yield mod
    assert mod.device_status(clear=True) == 0


def run_bwd(ea, inp, causal):
    q, k, v, do = (getattr(inp, n).to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = ea.fwd(q, k, v, causal=causal)
    dq, dk, dv = ea.bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    return dq, dk, dv


def floors(inp, ref, d):
    """Per-head absolute floor of each gradient (see the module docstring)."""
    do = inp.do.double().numpy()
    dmag = np.abs(do * ref["o"]).sum(axis=3).max(axis=2)[:, :, None, None]
    qmax = np.abs(inp.q.double().numpy()).max(axis=(2, 3), keepdims=True)
    kmax = np.abs(inp.k.double().numpy()).max(axis=(2, 3), keepdims=True)
    s = 1.0 / math.sqrt(d)
    return {"dq": 2.0 ** -8 * s * kmax * dmag, "dk": 2.0 ** -8 * s * qmax * dmag, "dv": 0.0}


def check(name, got, want, where, floor=0.0):
    g = got.double().cpu().numpy()
    assert np.isfinite(g).all(), f"{where}: non-finite {name}"
    err = np.abs(g - want)
    scale = np.abs(want).max(axis=(2, 3), keepdims=True)
    bound = REL * scale + bf16_half_ulp(want) + floor
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err - bound, -1)), err.shape)
        raise AssertionError(f"{where}: {name} off at {idx}: got {g[idx]}, want {want[idx]} "
                             f"({int(bad.sum())} elements; max rel {float((err / np.maximum(scale, 1e-30)).max()):.3g})")
    return float((err / np.maximum(scale, 1e-30)).max())


SHAPES = [
    # (B, H, N, d, causal)
    (1, 1, 1, 64, False),
    (1, 1, 1, 128, True),
    (1, 2, 128, 128, False),
    (1, 2, 128, 128, True),
    (1, 1, 200, 64, True),
    (2, 1, 257, 128, False),
    (1, 2, 300, 128, True),
    (1, 1, 513, 64, False),
    (1, 2, 640, 128, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", SHAPES,
                         ids=[f"B{b}H{h}N{n}d{d}-{'causal' if c else 'full'}"
                              for b, h, n, d, c in SHAPES])
def test_bwd_parity(ea, B, H, N, d, causal):
    inp = random_bwd_inputs(B, H, N, d, seed=13 * N + d + int(causal))
    dq, dk, dv = run_bwd(ea, inp, causal)
    ref = oracle.get().attention_bwd(*(inp.raw(n) for n in ("q", "k", "v", "do")),
                                     1.0 / math.sqrt(d), causal, "bf16")
    where = f"{(B, H, N, d, causal)}"
    fl = floors(inp, ref, d)
    rel = {name: check(name, got, ref[name], where, fl[name])
           for name, got in (("dq", dq), ("dk", dk), ("dv", dv))}
    print(where, rel)


def test_bwd_larger_head(ea):
    """A longer sequence (several key and query blocks per CTA loop) on two heads."""
    B, H, N, d = 1, 2, 2048, 128
    for causal in (False, True):
        inp = random_bwd_inputs(B, H, N, d, seed=777 + int(causal))
        dq, dk, dv = run_bwd(ea, inp, causal)
        ref = oracle.get().attention_bwd(*(inp.raw(n) for n in ("q", "k", "v", "do")),
                                         1.0 / math.sqrt(d), causal, "bf16")
        fl = floors(inp, ref, d)
        rel = {name: check(name, got, ref[name], f"N{N} causal={causal}", fl[name])
               for name, got in (("dq", dq), ("dk", dk), ("dv", dv))}
        print("N2048", causal, rel)


def test_bwd_zero_dout_gives_zero_gradients(ea):
    inp = random_bwd_inputs(1, 1, 300, 64, seed=99)
    inp.do.zero_()
    for causal in (False, True):
        dq, dk, dv = run_bwd(ea, inp, causal)
        for t in (dq, dk, dv):
            assert torch.count_nonzero(t) == 0


def test_bwd_no_writes_past_the_outputs(ea):
    B, H, N, d = 1, 2, 300, 128
    inp = random_bwd_inputs(B, H, N, d, seed=98)
    q, k, v, do = (getattr(inp, n).to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = ea.fwd(q, k, v, causal=True)
    n_el = B * H * N * d
    bufs = [torch.full((n_el + 4096,), 7.0, dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    outs = [b[:n_el].view(B, H, N, d) for b in bufs]
    ea.bwd(q, k, v, o, lse, do, causal=True, dq=outs[0], dk=outs[1], dv=outs[2])
    torch.cuda.synchronize()
    for b in bufs:
        assert (b[n_el:] == 7.0).all()
