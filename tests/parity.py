"""Comparison of the CUDA path's outputs with the oracle's, element by element.

Tolerances (the targets of the method's accuracy statement): bf16 operands max|O - O_ref| <= 1e-2
and |LSE - LSE_ref| <= 1e-3; fp8-e4m3 operands 5e-2 and 5e-3.  O_ref is the exact fp64 result,
while the kernel must round O to bf16, whose half-ulp alone is up to 2^-7 = 0.0078 for
|O| in [2, 4) and 0.0156 for |O| in [4, 8).  Each element therefore gets the tolerance plus half
a bf16 ulp of |O_ref|.  The returned statistics also give the raw error against the unwidened
tolerance: how many elements exceed it and the largest |O_ref| among them (where the kernel's
bf16 output cannot get closer than the rounding of O_ref itself).
"""
from __future__ import annotations

import numpy as np
import torch

TOL = {"bf16": (1e-2, 1e-3), "e4m3": (5e-2, 5e-3)}


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype: str, where: str = ""):
    """Raise AssertionError unless every element is within tolerance; return the error stats."""
    tol_o, tol_l = TOL[dtype]
    o = o_gpu.double().cpu().numpy() if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu)
    lse = lse_gpu.double().cpu().numpy() if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert lse.shape == lse_ref.shape, (lse.shape, lse_ref.shape)
    assert np.isfinite(o).all(), f"{where}: non-finite O"
    assert np.isfinite(lse).all(), f"{where}: non-finite LSE"
    err_o = np.abs(o - o_ref)
    err_l = np.abs(lse - lse_ref)
    ref_bf16 = torch.from_numpy(o_ref).to(torch.bfloat16).double().numpy()
    over = err_o > tol_o
    stats = {
        "max_err_o": float(err_o.max()),
        "max_err_o_vs_bf16_ref": float(np.abs(o - ref_bf16).max()),
        "max_err_lse": float(err_l.max()),
        "mean_err_o": float(err_o.mean()),
        "n_over_unwidened": int(over.sum()),
        "max_abs_ref_over_unwidened": float(np.abs(o_ref[over]).max()) if over.any() else 0.0,
    }
    bad = err_o > tol_o + bf16_half_ulp(o_ref)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err_o, 0)), err_o.shape)
        raise AssertionError(f"{where}: O out of tolerance at {idx}: got {o[idx]}, want "
                             f"{o_ref[idx]} ({int(bad.sum())} bad elements) {stats}")
    if (err_l > tol_l).any():
        idx = np.unravel_index(np.argmax(err_l), err_l.shape)
        raise AssertionError(f"{where}: LSE out of tolerance at {idx}: got {lse[idx]}, want "
                             f"{lse_ref[idx]} {stats}")
    return stats
