"""Pins for the reference fp8 block quantiser and incoherent transform (CPU only).

Each check rests on something other than the quantiser's own code: scipy's Hadamard matrix,
orthogonality, the invariance of QKᵀ the pages state, torch's float -> e4m3 conversion, the
format's half-step error bound, and block maxima found here with a plain loop.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import quantize as qz


@pytest.mark.parametrize("d", [1, 2, 8, 64, 128, 256])
def test_sylvester_matches_scipy_hadamard(d):
    np.testing.assert_array_equal(qz.sylvester_hadamard(d), scipy.linalg.hadamard(d))


def test_transform_is_orthogonal_and_keeps_scores():
    """M = diag(s) H / sqrt(d) is orthogonal, so Q'K'ᵀ = QKᵀ ("FlashAttention · InkStack",
    section 3.3.2 "Incoherent Processing")."""
    rng = np.random.default_rng(31)
    for d in (64, 128):
        s = rng.choice([-1.0, 1.0], size=d)
        m = qz.incoherent_transform(np.eye(d), s)
        np.testing.assert_allclose(m @ m.T, np.eye(d), atol=1e-13)
        q = rng.standard_normal((40, d))
        k = rng.standard_normal((33, d))
        qt, kt = qz.incoherent_transform(q, s), qz.incoherent_transform(k, s)
        np.testing.assert_allclose(qt @ kt.T, q @ k.T, atol=1e-11)
        assert not np.allclose(qt, q)


def test_transform_spreads_an_outlier_evenly():
    """A single coordinate of size A becomes d coordinates of size A / sqrt(d)."""
    for d in (64, 128):
        s = np.where(np.arange(d) % 3 == 0, -1.0, 1.0)
        for pos in (0, 5, d - 1):
            x = np.zeros(d)
            x[pos] = 40.0
            y = qz.incoherent_transform(x, s)
            np.testing.assert_allclose(np.abs(y), 40.0 / np.sqrt(d), rtol=1e-14)


def test_transform_of_a_basis_vector_is_a_signed_hadamard_row():
    """e_k · diag(s) H / sqrt(d) = s_k · (row k of scipy's Hadamard matrix) / sqrt(d): the sign
    flip comes before the Hadamard mix ("FlashAttention 完全拆解（三）", section on incoherent
    processing: a random +-1 diagonal times a Hadamard matrix)."""
    rng = np.random.default_rng(34)
    for d in (64, 128):
        s = rng.choice([-1.0, 1.0], size=d)
        h = scipy.linalg.hadamard(d)
        for k in (0, 3, d - 1):
            e = np.zeros(d)
            e[k] = 1.0
            np.testing.assert_allclose(qz.incoherent_transform(e, s), s[k] * h[k] / np.sqrt(d),
                                       rtol=0, atol=1e-15)


def test_transform_rejects_bad_signs():
    with pytest.raises(ValueError):
        qz.incoherent_transform(np.ones((2, 8)), np.full(8, 0.5))
    with pytest.raises(ValueError):
        qz.sylvester_hadamard(48)


def _torch_e4m3(y):
    return torch.from_numpy(np.asarray(y, dtype=np.float32)).to(torch.float8_e4m3fn)


def test_rounding_matches_torch_on_a_dense_sweep_and_on_ties():
    """Round-to-nearest-even onto the e4m3 grid agrees with torch's conversion for in-range
    values, including every midpoint between neighbours (ties go to the even code)."""
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    grid = grid.numpy()
    mids = (grid[:-1] + grid[1:]) / 2
    rng = np.random.default_rng(32)
    sweep = np.concatenate([grid, mids, rng.uniform(0, 448, 20000),
                            np.exp2(rng.uniform(-12, 8.8, 20000))])
    sweep = np.concatenate([sweep, -sweep]).astype(np.float32)
    sweep = sweep[np.abs(sweep) <= 448]
    codes, vals = qz.round_to_e4m3(sweep)
    want = _torch_e4m3(sweep)
    np.testing.assert_array_equal(codes, want.view(torch.uint8).numpy())
    np.testing.assert_array_equal(vals, want.to(torch.float64).numpy())


def test_rounding_saturates_at_448():
    codes, vals = qz.round_to_e4m3(np.array([460.0, 464.0, 1e6, -1e30], dtype=np.float32))
    np.testing.assert_array_equal(vals, [448.0, 448.0, 448.0, -448.0])
    np.testing.assert_array_equal(codes, [0x7E, 0x7E, 0x7E, 0xFE])


def _half_step(v):
    """Half the e4m3 spacing around |v| (2^-10 in the subnormal range)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 2.0 ** (e - 4)


@pytest.mark.parametrize("signs", [False, True])
def test_block_quantize_scales_and_error_bound(signs):
    """Per 128-row block of each head: descale = amax / 448 in fp32 (the block maxima found
    here row by row), the block's largest element maps to +-448, and every code is within
    half an e4m3 step (plus the fp32 rounding of the product) of x / descale
    ("FlashAttention · InkStack", sections 3.3.1, 3.3.3)."""
    rng = np.random.default_rng(33)
    B, H, N, d = 2, 3, 300, 64
    x = rng.standard_normal((B, H, N, d)).astype(np.float32)
    x[0, 1, 5, 7] = 60.0  # an outlier in one block of one head
    x[1, 2, 250:] = 0.0   # a ragged tail block that is all zero
    sg = np.where(rng.random(d) < 0.5, -1.0, 1.0) if signs else None
    codes, descales, scaled = qz.block_quantize(x, 128, sg)
    xt = qz.incoherent_transform(x, sg).astype(np.float32) if signs else x
    assert descales.shape == (B, H, 3)
    for b in range(B):
        for h in range(H):
            for j in range(3):
                rows = range(j * 128, min(N, (j + 1) * 128))
                amax = max(float(np.abs(xt[b, h, r]).max()) for r in rows)
                want = np.float32(amax) / np.float32(448) if amax > 0 else np.float32(1)
                assert descales[b, h, j] == want
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.all(np.abs(vals - scaled) <= _half_step(scaled) * (1 + 1e-12)
                  + np.abs(scaled) * 2.0 ** -23)
    quot = xt.astype(np.float64) / np.repeat(descales, 128, axis=2)[:, :, :N, None]
    np.testing.assert_allclose(scaled, quot, rtol=2.0 ** -22)
    assert np.abs(vals).max() == 448.0
    if not signs:
        assert vals[0, 1, 5, 7] == 448.0
        assert np.all(vals[1, 2, 250:] == 0) and descales[1, 2, 2] == 1.0
    # the reconstruction is close to the input: relative error of e4m3 (<= 2^-4) per element
    rec = vals * np.repeat(descales, 128, axis=2)[:, :, :N, None]
    err = np.abs(rec - xt)
    assert np.all(err <= np.abs(xt) * 2.0 ** -4 + np.repeat(descales, 128, axis=2)[:, :, :N, None]
                  * 2.0 ** -10)


def test_power_of_two_descales():
    """With ``pow2`` each descale is the smallest power of two at or above amax / 448, so the
    block's largest code lies in (224, 448] and x / descale is exact before the e4m3 rounding."""
    rng = np.random.default_rng(35)
    x = (rng.standard_normal((1, 2, 260, 64)) * rng.uniform(0.01, 50, (1, 2, 1, 1)))
    x = x.astype(np.float32)
    c1, d1, _ = qz.block_quantize(x, 128)
    c2, d2, scaled = qz.block_quantize(x, 128, pow2=True)
    m, e = np.frexp(d2.astype(np.float64))
    assert np.all(m == 0.5)
    assert np.all(d2 >= d1) and np.all(d2 < 2 * d1)
    vals = torch.from_numpy(c2).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for j in range(3):
        top = np.abs(vals[:, :, j * 128:(j + 1) * 128]).max(axis=(2, 3))
        assert np.all((top > 224) & (top <= 448))
    exact = x.astype(np.float64) / np.repeat(d2, 128, axis=2)[:, :, :260, None]
    np.testing.assert_array_equal(scaled, exact)
    np.testing.assert_array_equal(c2, qz.round_to_e4m3(exact.astype(np.float32))[0])
