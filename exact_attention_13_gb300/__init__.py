"""exact_attention_13_gb300 -- fused exact-attention forward on GB300 (sm_103a).

A thin ctypes binding over ``libexattn.so`` (C ABI in ``include/exact_attention.h``).  This
module only checks and marshals arguments; every step of the attention forward runs in the
library's CUDA kernel.  PyTorch supplies device memory and the current stream.  There is no
fallback: if the library is missing or fails to load, importing ``lib()`` raises.

    import exact_attention_13_gb300 as ea
    o, lse = ea.fwd(q, k, v, causal=True)           # q, k, v: [B, H, N, d] bf16 on cuda
    o, lse = ea.fwd(q8, k8, v8, descale=(dq, dk, dv))  # float8_e4m3fn operands
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_CUDA = 4
FA_ERR_DEVICE_TIMEOUT = 5
FA_QUANT_POW2_DESCALE = 1
FA_DTYPE_BF16 = 0
FA_DTYPE_FP8_E4M3 = 1
FA_DTYPE_FP8_E4M3_PV16 = 2

LIB_PATH = _build.LIB_PATH

# every entry point of include/exact_attention.h: (restype, argtypes)
_c = ctypes
SIGNATURES = {
    "fa_fwd": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                          _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_float, _c.c_int, _c.c_int,
                          _c.c_void_p]),
    "fa_fwd_ex": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                             _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_float, _c.c_int,
                             _c.c_int, _c.c_void_p, _c.c_void_p]),
    "fa_fwd_split": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                _c.c_void_p, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_float,
                                _c.c_int, _c.c_int, _c.c_int, _c.c_void_p, _c.c_size_t,
                                _c.c_void_p, _c.c_void_p]),
    "fa_fwd_split_workspace_bytes": (_c.c_size_t, [_c.c_int, _c.c_int, _c.c_int, _c.c_int,
                                                   _c.c_int]),
    "fa_fwd_split_noalloc": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                        _c.c_void_p, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                                        _c.c_float, _c.c_int, _c.c_int, _c.c_int, _c.c_void_p,
                                        _c.c_void_p]),
    "fa_fwd_fp8_blockscaled": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                          _c.c_void_p, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                                          _c.c_float, _c.c_int, _c.c_int, _c.c_void_p, _c.c_void_p,
                                          _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_size_t,
                                          _c.c_void_p, _c.c_void_p]),
    "fa_quantize_e4m3": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int,
                                    _c.c_int, _c.c_int, _c.c_void_p, _c.c_int, _c.c_void_p]),
    "fa_bwd": (_c.c_int, [_c.c_void_p] * 5 + [_c.c_void_p] * 4 + [_c.c_int] * 4 + [
        _c.c_float, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p, _c.c_void_p]),
    "fa_bwd_workspace_bytes": (_c.c_size_t, [_c.c_int, _c.c_int, _c.c_int]),
    "fa_device_status": (_c.c_int, [_c.c_int, _c.POINTER(_c.c_int)]),
    "fa_status_string": (_c.c_char_p, [_c.c_int]),
    "fa_version": (_c.c_int, []),
    "fa_debug_exp2": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_longlong, _c.c_int,
                                 _c.c_void_p]),
}


class FwdOpts(ctypes.Structure):
    """Mirror of ``fa_fwd_opts``."""

    _fields_ = [("descale_q", ctypes.c_float), ("descale_k", ctypes.c_float),
                ("descale_v", ctypes.c_float), ("dev_status", ctypes.c_void_p)]


class AttentionError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = _status_name(code)
        super().__init__(f"{what}: {msg} (status {code})" if what else f"{msg} (status {code})")


_lock = threading.Lock()
_lib = None


def lib(path: str | None = None) -> ctypes.CDLL:
    """The loaded library (built first if the sources are newer).  Raises if it cannot load."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if path is None and not _build.up_to_date():
                _build.build()
            if not os.path.exists(p):
                raise ImportError(f"libexattn.so not found at {p}; run the build first")
            handle = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def _status_name(code: int) -> str:
    try:
        return lib().fa_status_string(code).decode()
    except Exception:  # noqa: BLE001 -- message formatting only
        return "status"


def _check(code: int, what: str):
    if code != FA_OK:
        raise AttentionError(code, what)


def fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, causal, dtype, stream) -> int:
    """Direct C-ABI call with raw device pointers; returns the status code."""
    return lib().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, int(causal),
                        dtype, stream)


def fa_fwd_ex(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, causal, dtype,
              descale=(1.0, 1.0, 1.0), status_ptr=None, stream=None) -> int:
    opts = FwdOpts(float(descale[0]), float(descale[1]), float(descale[2]), status_ptr)
    return lib().fa_fwd_ex(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, int(causal),
                           dtype, ctypes.byref(opts), stream)


def fa_fwd_split(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, causal, dtype,
                 num_splits, workspace_ptr, workspace_bytes, descale=(1.0, 1.0, 1.0),
                 status_ptr=None, stream=None) -> int:
    opts = FwdOpts(float(descale[0]), float(descale[1]), float(descale[2]), status_ptr)
    return lib().fa_fwd_split(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale,
                              int(causal), dtype, int(num_splits), workspace_ptr,
                              int(workspace_bytes), ctypes.byref(opts), stream)


def fa_fwd_split_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, causal, dtype,
                         num_splits, descale=(1.0, 1.0, 1.0), status_ptr=None,
                         stream=None) -> int:
    """Key-split forward whose partials use the library's fixed device scratch (no allocation
    anywhere); see fa_fwd_split_noalloc in include/exact_attention.h for the limits."""
    opts = FwdOpts(float(descale[0]), float(descale[1]), float(descale[2]), status_ptr)
    return lib().fa_fwd_split_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale,
                                      int(causal), dtype, int(num_splits), ctypes.byref(opts),
                                      stream)


def fa_fwd_fp8_blockscaled(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, causal,
                           dq_blk_ptr, dk_blk_ptr, dv_blk_ptr, num_splits=1, workspace_ptr=None,
                           workspace_bytes=0, status_ptr=None, stream=None,
                           dtype=FA_DTYPE_FP8_E4M3) -> int:
    return lib().fa_fwd_fp8_blockscaled(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale,
                                        int(causal), int(dtype), dq_blk_ptr, dk_blk_ptr,
                                        dv_blk_ptr, int(num_splits), workspace_ptr,
                                        int(workspace_bytes), status_ptr, stream)


def fa_quantize_e4m3(x_ptr, codes_ptr, descales_ptr, B, H, N, d, signs_ptr=None, flags=0,
                     stream=None) -> int:
    return lib().fa_quantize_e4m3(x_ptr, codes_ptr, descales_ptr, B, H, N, d, signs_ptr,
                                  int(flags), stream)


def split_workspace_bytes(B: int, H: int, N: int, d: int, num_splits: int) -> int:
    return int(lib().fa_fwd_split_workspace_bytes(B, H, N, d, num_splits))


def device_status(clear: bool = True) -> int:
    out = ctypes.c_int(0)
    _check(lib().fa_device_status(int(clear), ctypes.byref(out)), "fa_device_status")
    return out.value


def version() -> int:
    return lib().fa_version()


def fwd(q, k, v, causal: bool = False, scale: float | None = None, descale=None, out=None,
        lse=None, status=None, num_splits: int = 1, workspace=None, pv16: bool = False):
    """Attention forward on torch CUDA tensors [B, H, N, d]; returns (o bf16, lse fp32).

    ``descale`` = (dq, dk, dv) for float8_e4m3fn operands; both of their products are fp8
    unless ``pv16`` asks for an f16 P V product (P rounded to f16: slower, more accurate); with
    ``causal`` the first 256 query rows of each head always take the f16 P V product.  ``out``/``lse`` may be given
    (contiguous, right shape and dtype) to avoid allocation.  ``status`` is an optional int32
    CUDA tensor of one element the kernel sets to FA_ERR_DEVICE_TIMEOUT if a wait runs out.
    ``num_splits`` > 1 splits each query tile's keys over that many CTAs and merges the partial
    results (fa_fwd_split); its scratch is ``workspace`` (a CUDA tensor of at least
    split_workspace_bytes(...) bytes) or, if None, a temporary allocated here by torch.
    """
    import torch

    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k, v must share one dtype")
    if q.dtype == torch.bfloat16:
        dtype = FA_DTYPE_BF16
    elif q.dtype == torch.float8_e4m3fn:
        dtype = FA_DTYPE_FP8_E4M3_PV16 if pv16 else FA_DTYPE_FP8_E4M3
    else:
        raise ValueError(f"unsupported operand dtype {q.dtype}")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    dq, dk, dv = descale if descale is not None else (1.0, 1.0, 1.0)
    st = status.data_ptr() if status is not None else None
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        if num_splits == 1:
            rc = fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), B, H, N, d, float(scale), causal, dtype, (dq, dk, dv),
                           st, stream)
            _check(rc, "fa_fwd_ex")
            return out, lse
        need = split_workspace_bytes(B, H, N, d, num_splits)
        if need == 0:
            raise ValueError(f"invalid split configuration (num_splits={num_splits}, d={d})")
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        nbytes = workspace.numel() * workspace.element_size()
        rc = fa_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr(), B, H, N, d, float(scale), causal, dtype, num_splits,
                          workspace.data_ptr(), nbytes, (dq, dk, dv), st, stream)
    _check(rc, "fa_fwd_split")
    return out, lse


def quantize_e4m3(x, signs=None, pow2: bool = False, codes=None, descales=None):
    """Block-quantise a bf16 CUDA tensor [B, H, N, d] to e4m3 (one fp32 descale per 128-row
    block of each head), first applying the incoherent transform diag(signs) Had / sqrt(d) to
    every row when ``signs`` (a CUDA fp32 tensor of d values +-1) is given; ``pow2`` rounds the
    descales up to powers of two (use it for V).  Returns (codes float8_e4m3fn [B, H, N, d],
    descales fp32 [B, H, ceil(N / 128)])."""
    import torch

    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 4 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 CUDA tensor [B, H, N, d]")
    B, H, N, d = x.shape
    nblk = -(-N // 128)
    if codes is None:
        codes = torch.empty((B, H, N, d), dtype=torch.float8_e4m3fn, device=x.device)
    if descales is None:
        descales = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    if codes.shape != x.shape or codes.dtype != torch.float8_e4m3fn or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous float8_e4m3fn tensor shaped like x")
    if descales.shape != (B, H, nblk) or descales.dtype != torch.float32:
        raise ValueError(f"descales must be fp32 [B, H, {nblk}]")
    sp = None
    if signs is not None:
        if signs.shape != (d,) or signs.dtype != torch.float32 or not signs.is_cuda:
            raise ValueError("signs must be a CUDA fp32 tensor of d values")
        sp = signs.data_ptr()
    stream = torch.cuda.current_stream(x.device).cuda_stream
    with torch.cuda.device(x.device):
        rc = fa_quantize_e4m3(x.data_ptr(), codes.data_ptr(), descales.data_ptr(), B, H, N, d,
                              sp, FA_QUANT_POW2_DESCALE if pow2 else 0, stream)
    _check(rc, "fa_quantize_e4m3")
    return codes, descales


def fwd_fp8_blockscaled(q, k, v, dq_blk, dk_blk, dv_blk, causal: bool = False,
                        scale: float | None = None, out=None, lse=None, status=None,
                        num_splits: int = 1, workspace=None, pv16: bool = False):
    """Attention forward on float8_e4m3fn CUDA tensors with per-block descales
    (fp32 [B, H, ceil(N / 128)] each, as ``quantize_e4m3`` returns); returns (o bf16, lse)."""
    import torch

    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.float8_e4m3fn or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous float8_e4m3fn CUDA tensors")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    nblk = -(-N // 128)
    for t in (dq_blk, dk_blk, dv_blk):
        if (t.shape != (B, H, nblk) or t.dtype != torch.float32 or not t.is_cuda
                or not t.is_contiguous()):
            raise ValueError(f"block descales must be contiguous fp32 CUDA [B, H, {nblk}]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    ws_ptr, ws_bytes = None, 0
    if num_splits > 1:
        need = split_workspace_bytes(B, H, N, d, num_splits)
        if need == 0:
            raise ValueError(f"invalid split configuration (num_splits={num_splits}, d={d})")
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = status.data_ptr() if status is not None else None
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        rc = fa_fwd_fp8_blockscaled(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), B, H, N, d, float(scale), causal,
                                    dq_blk.data_ptr(), dk_blk.data_ptr(), dv_blk.data_ptr(),
                                    num_splits, ws_ptr, ws_bytes, st, stream,
                                    FA_DTYPE_FP8_E4M3_PV16 if pv16 else FA_DTYPE_FP8_E4M3)
    _check(rc, "fa_fwd_fp8_blockscaled")
    return out, lse


def fa_bwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, do_ptr, dq_ptr, dk_ptr, dv_ptr, B, H, N, d,
           scale, causal, workspace_ptr, workspace_bytes, status_ptr=None, stream=None) -> int:
    return lib().fa_bwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, do_ptr, dq_ptr, dk_ptr, dv_ptr, B, H,
                        N, d, scale, int(causal), workspace_ptr, int(workspace_bytes), status_ptr,
                        stream)


def bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, N))


def bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, dq=None,
        dk=None, dv=None, workspace=None, status=None):
    """Attention backward on bf16 CUDA tensors [B, H, N, d]: o and lse are the forward's outputs
    for q, k, v; dout is dL/dO.  Returns (dq, dk, dv), bf16."""
    import torch

    for t in (q, k, v, o, dout):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k, v, o, dout must be contiguous bf16 CUDA tensors")
        if t.shape != q.shape:
            raise ValueError("q, k, v, o, dout must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    need = bwd_workspace_bytes(B, H, N)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = status.data_ptr() if status is not None else None
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                    float(scale), causal, workspace.data_ptr(),
                    workspace.numel() * workspace.element_size(), st, stream)
    _check(rc, "fa_bwd")
    return dq, dk, dv


def debug_exp2(x, mode: int):
    """The kernel's 2^x routines on a CUDA float32 tensor (mode 0 MUFU, 1 FMA polynomial)."""
    import torch

    x = x.contiguous()
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    _check(lib().fa_debug_exp2(x.data_ptr(), y.data_ptr(), x.numel(), mode, stream),
           "fa_debug_exp2")
    return y
