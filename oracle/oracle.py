"""Python face of the fp64 attention oracle -- TEST INFRASTRUCTURE, NOT THE PRODUCT PATH.

Only ``tests/``, the smoke check and the CPU-baseline leg of ``bench.py`` use this module.  It
builds ``attention_oracle.c`` with gcc (no CUDA) into ``oracle/_build/`` and calls it through
ctypes.  The CUDA library never imports, links or calls anything here, and nothing here imports
the CUDA library.

See ``attention_oracle.c`` for what is computed and which passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attention_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")

DTYPE_CODES = {"bf16": 0, "e4m3": 1, "f64": 2}

_lock = threading.Lock()
_default = None


def build(out_path: str | None = None, mutation: int = 0) -> str:
    """Compile the oracle (optionally with a planted mistake) and return the .so path."""
    if out_path is None:
        out_path = os.path.join(BUILD_DIR, "liboracle.so")
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-std=c11",
           f"-DORACLE_MUTATION={int(mutation)}", SRC, "-o", out_path + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out_path + ".tmp", out_path)
    return out_path


def _needs_build(path: str) -> bool:
    return (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(SRC)


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        f = lib.oracle_attention_fwd
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                      ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                      ctypes.c_double, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                      ctypes.c_double, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_int]
        g = lib.oracle_attention_fwd_blockscaled
        g.restype = ctypes.c_int
        g.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                      ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                      ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        bw = lib.oracle_attention_bwd
        bw.restype = ctypes.c_int
        bw.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_int64] * 4 + [
            ctypes.c_double, ctypes.c_int] + [ctypes.c_void_p] * 6 + [ctypes.c_int]
        lib.oracle_decode_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_decode_e4m3_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_mutation_id.restype = ctypes.c_int
        self._lib = lib
        self.mutation = lib.oracle_mutation_id()

    def decode(self, raw: np.ndarray, dtype: str) -> np.ndarray:
        """Exact fp64 values of bf16 (uint16) or e4m3 (uint8) bit patterns."""
        raw = np.ascontiguousarray(raw)
        out = np.empty(raw.shape, dtype=np.float64)
        if dtype == "bf16":
            assert raw.dtype == np.uint16
            self._lib.oracle_decode_bf16_array(raw.ctypes.data, out.ctypes.data, raw.size)
        elif dtype == "e4m3":
            assert raw.dtype == np.uint8
            self._lib.oracle_decode_e4m3_array(raw.ctypes.data, out.ctypes.data, raw.size)
        else:
            raise ValueError(dtype)
        return out

    @staticmethod
    def _operands(q, k, v, dtype):
        q = np.ascontiguousarray(q)
        k = np.ascontiguousarray(k)
        v = np.ascontiguousarray(v)
        if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
            raise ValueError("q, k, v must share one [B,H,N,d] shape")
        want = {"f64": np.float64, "bf16": np.uint16, "e4m3": np.uint8}[dtype]
        for t in (q, k, v):
            if t.dtype != want:
                raise TypeError(f"{dtype} operands must be {np.dtype(want).name}, got {t.dtype}")
        return q, k, v

    @staticmethod
    def _rows(rows, N):
        if rows is None:
            return N, None, None
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        return rows_arr.size, rows_arr, rows_arr.ctypes.data

    def attention_fwd_blockscaled(self, q, k, v, scale: float, causal: bool, dtype: str,
                                  dq_blk, dk_blk, dv_blk, blk_rows: int = 128, rows=None,
                                  threads: int | None = None):
        """Like ``attention_fwd`` with per-block descales: ``dq_blk`` etc. are [B,H,nblk]
        arrays, nblk = ceil(N / blk_rows); row i of head (b, h) is scaled by
        ``d*_blk[b, h, i // blk_rows]``."""
        q, k, v = self._operands(q, k, v, dtype)
        B, H, N, d = q.shape
        nblk = -(-N // blk_rows)
        scales = []
        for s in (dq_blk, dk_blk, dv_blk):
            s = np.ascontiguousarray(np.asarray(s, dtype=np.float64))
            if s.shape != (B, H, nblk):
                raise ValueError(f"block descales must be [B,H,{nblk}], got {s.shape}")
            scales.append(s)
        R, rows_arr, rows_ptr = self._rows(rows, N)
        o = np.empty((B, H, R, d), dtype=np.float64)
        lse = np.empty((B, H, R), dtype=np.float64)
        rc = self._lib.oracle_attention_fwd_blockscaled(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, DTYPE_CODES[dtype], B, H, N, d,
            float(scale), int(bool(causal)), scales[0].ctypes.data, scales[1].ctypes.data,
            scales[2].ctypes.data, int(blk_rows), rows_ptr, R, o.ctypes.data, lse.ctypes.data,
            int(threads or os.cpu_count() or 1))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_fwd_blockscaled failed with code {rc}")
        return o, lse

    def attention_bwd(self, q, k, v, dout, scale: float, causal: bool = False,
                      dtype: str = "f64", threads: int | None = None):
        """Gradients of L = sum(O * dout): returns dict of fp64 arrays dq, dk, dv [B,H,N,d] and
        the recomputed o [B,H,N,d], lse [B,H,N], delta [B,H,N] (D_i = dO_i . O_i)."""
        if dtype not in ("f64", "bf16"):
            raise ValueError("the backward takes bf16 or f64 operands")
        q, k, v = self._operands(q, k, v, dtype)
        dout = np.ascontiguousarray(dout)
        if dout.shape != q.shape or dout.dtype != q.dtype:
            raise ValueError("dout must match q in shape and dtype")
        B, H, N, d = q.shape
        out = {n: np.empty((B, H, N, d)) for n in ("dq", "dk", "dv", "o")}
        out["lse"] = np.empty((B, H, N))
        out["delta"] = np.empty((B, H, N))
        rc = self._lib.oracle_attention_bwd(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, DTYPE_CODES[dtype],
            B, H, N, d, float(scale), int(bool(causal)), out["dq"].ctypes.data,
            out["dk"].ctypes.data, out["dv"].ctypes.data, out["o"].ctypes.data,
            out["lse"].ctypes.data, out["delta"].ctypes.data,
            int(threads or os.cpu_count() or 1))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_bwd failed with code {rc}")
        return out

    def attention_fwd(self, q, k, v, scale: float, causal: bool = False, dtype: str = "f64",
                      descale=(1.0, 1.0, 1.0), rows=None, threads: int | None = None):
        """O [B,H,R,d] and LSE [B,H,R] in fp64 for the requested rows (all rows if None).

        ``q``, ``k``, ``v`` are numpy arrays of shape [B,H,N,d]: float64 values for dtype
        "f64", uint16 bf16 bit patterns for "bf16", uint8 e4m3 bit patterns for "e4m3".
        """
        q, k, v = self._operands(q, k, v, dtype)
        B, H, N, d = q.shape
        R, rows_arr, rows_ptr = self._rows(rows, N)
        o = np.empty((B, H, R, d), dtype=np.float64)
        lse = np.empty((B, H, R), dtype=np.float64)
        if threads is None:
            threads = os.cpu_count() or 1
        rc = self._lib.oracle_attention_fwd(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, DTYPE_CODES[dtype], B, H, N, d,
            float(scale), int(bool(causal)), float(descale[0]), float(descale[1]),
            float(descale[2]), rows_ptr, R, o.ctypes.data, lse.ctypes.data, int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_fwd failed with code {rc}")
        return o, lse


def get() -> Oracle:
    """The default (unmutated) oracle, built on first use."""
    global _default
    with _lock:
        if _default is None:
            path = os.path.join(BUILD_DIR, "liboracle.so")
            if _needs_build(path):
                build(path)
            _default = Oracle(path)
        return _default


def attention_fwd(*args, **kwargs):
    return get().attention_fwd(*args, **kwargs)


def attention_fwd_inputs(inp, scale: float, causal: bool, rows=None, threads=None):
    """Run the oracle on a ``workloads.Inputs`` bundle (the same bytes the GPU path gets)."""
    dt = inp.dtype
    return get().attention_fwd(inp.raw("q"), inp.raw("k"), inp.raw("v"), scale, causal, dt,
                               (inp.descale_q, inp.descale_k, inp.descale_v), rows, threads)
