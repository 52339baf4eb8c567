"""FP8 block quantisation with optional incoherent processing -- TEST INFRASTRUCTURE.

A plain numpy statement of the quantiser the fp8 attention path consumes.  Only ``tests/`` and
the benchmark's CPU-baseline leg use it; the CUDA library shares nothing with it.

What it computes (pages cited by title and section):

* Incoherent processing ("FlashAttention · InkStack", section 3.3.2 "Incoherent Processing";
  "FlashAttention 完全拆解（三）", section "精度问题二：非相干处理"): the same orthogonal matrix
  M = D·H/sqrt(d) multiplies the queries and the keys of a head, X' = X·M, where D = diag(s) is
  a random +-1 diagonal and H the d x d Sylvester-Hadamard matrix.  M·Mᵀ = I, so Q'K'ᵀ = QKᵀ and
  attention is unchanged; outlier energy is spread over all d coordinates.  The values are not
  transformed.  Here the transform is a dense fp64 product (the pages' fast transform is the
  kernel's business); the result is then rounded once to fp32, the precision the kernel keeps.
* Block quantisation ("FlashAttention · InkStack", sections 3.3.1 "Block Quantization" and 3.3.3
  "Scaling"): every block of ``blk_rows`` consecutive rows of one head gets its own descale
  ``amax(|X_blk|) / 448`` (448 is e4m3's largest finite value) and codes ``e4m3(X · scale)``
  with ``scale = 448 / amax``.  The arithmetic is fp32: descale and scale are correctly rounded
  fp32 quotients, X · scale an fp32 product, followed by round-to-nearest-even onto the e4m3
  grid with results beyond 448 clamped to 448.  A block whose amax is 0 gets descale and scale 1.

Readings where the pages leave a step open: the block is the attention kernel's 128-row tile;
one sign vector s serves every head; the pages only say that codes are the values scaled into
e4m3's range by the amax / 448 factor, and this states that scaling as a multiplication by the
fp32 reciprocal 448 / amax (one quotient per block instead of one per element).  Optionally
(``pow2``) the descale is raised to the next power of two, a choice of this library for value
blocks (e4m3's relative precision does not depend on the scale); the scale is then its exact
reciprocal.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def sylvester_hadamard(d: int) -> np.ndarray:
    """The d x d Hadamard matrix of Sylvester's construction, H_{2n} = [[H, H], [H, -H]]."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def incoherent_transform(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """X·D·H/sqrt(d) over the last axis, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    signs = np.asarray(signs, dtype=np.float64)
    if signs.shape != (d,) or not np.all(np.abs(signs) == 1.0):
        raise ValueError("signs must be d values of +-1")
    return (x * signs) @ sylvester_hadamard(d) / np.sqrt(d)


def _e4m3_positive_grid() -> np.ndarray:
    """Values of the e4m3fn codes 0x00..0x7E (ascending), from the format's bit fields."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append(m / 8.0 * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals)


_GRID = _e4m3_positive_grid()


def round_to_e4m3(y: np.ndarray):
    """Round fp32 values to e4m3 (nearest, ties to even code, clamp at 448).

    Returns (codes uint8, values float64).  Between two neighbours of the grid the nearer wins;
    on a tie the one with the even code (even mantissa) wins.
    """
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    a = np.abs(y)
    hi = np.clip(np.searchsorted(_GRID, a, side="left"), 0, len(_GRID) - 1)
    lo = np.clip(hi - 1, 0, None)
    d_lo = a - _GRID[lo]
    d_hi = _GRID[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(a >= _GRID[-1], len(_GRID) - 1, np.where(pick_hi, hi, lo))
    code = code.astype(np.uint8) | np.where(np.signbit(y), 0x80, 0).astype(np.uint8)
    val = np.where(np.signbit(y), -_GRID[code & 0x7F], _GRID[code & 0x7F])
    return code, val


def block_quantize(x: np.ndarray, blk_rows: int = 128, signs=None, pow2: bool = False):
    """Quantise X [B, H, N, d] block-wise; returns (codes uint8 [B,H,N,d], descales fp32
    [B,H,nblk], scaled fp64 [B,H,N,d]).  ``pow2`` rounds each descale up to a power of two.

    ``scaled`` is the fp64 value of (transformed fp32 value) x (fp32 scale) before any
    rounding, for tests that have to tell rounding ties apart from errors.
    """
    x = np.asarray(x)
    if signs is not None:
        x32 = incoherent_transform(x, signs).astype(np.float32)
    else:
        x32 = x.astype(np.float32)
    B, H, N, d = x32.shape
    nblk = -(-N // blk_rows)
    codes = np.empty((B, H, N, d), dtype=np.uint8)
    scaled = np.empty((B, H, N, d), dtype=np.float64)
    descales = np.empty((B, H, nblk), dtype=np.float32)
    for j in range(nblk):
        blk = x32[:, :, j * blk_rows:(j + 1) * blk_rows]
        amax = np.abs(blk).max(axis=(2, 3))
        one = np.float32(1.0)
        ds = np.where(amax > 0, amax / np.float32(E4M3_MAX), one).astype(np.float32)
        sc = np.where(amax > 0, np.float32(E4M3_MAX) / np.where(amax > 0, amax, one),
                      one).astype(np.float32)
        if pow2:
            ds = np.exp2(np.ceil(np.log2(ds.astype(np.float64)))).astype(np.float32)
            sc = (np.float32(1.0) / ds).astype(np.float32)
        descales[:, :, j] = ds
        y = (blk * sc[:, :, None, None]).astype(np.float32)
        codes[:, :, j * blk_rows:(j + 1) * blk_rows] = round_to_e4m3(y)[0]
        scaled[:, :, j * blk_rows:(j + 1) * blk_rows] = (blk.astype(np.float64)
                                                         * sc[:, :, None, None].astype(np.float64))
    return codes, descales, scaled
