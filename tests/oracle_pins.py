"""Pins for the fp64 oracle: checks against facts fixed by the pages and by mathematics.

Each pin takes an ``oracle.oracle.Oracle`` handle and raises AssertionError when it does not
hold.  ``test_oracle_pins.py`` runs them on the real oracle; ``test_oracle_mutations.py`` runs
them on builds with one planted mistake each and expects at least one pin to fail per build.

None of these re-types the oracle's loop: they use closed forms, invariants, library routines
(scipy's softmax / logsumexp, torch's dtype conversions) and a second evaluator that merges
column blocks with the online-softmax recurrence.
"""
from __future__ import annotations

import numpy as np
import scipy.special as sps
import torch

from oracle import online_softmax

PINS = []


def pin(fn):
    PINS.append(fn)
    return fn


def _rand(rng, shape):
    return rng.standard_normal(shape)


def _allowed(N, causal):
    m = np.ones((N, N), dtype=bool)
    return np.tril(m) if causal else m


@pin
def pin_library_softmax(orc):
    """Small cases equal scipy's softmax(.) @ V and logsumexp (a library routine)."""
    rng = np.random.default_rng(11)
    for causal in (False, True):
        for (B, H, N, d) in [(1, 1, 1, 1), (1, 2, 5, 3), (2, 1, 8, 4), (1, 1, 37, 16)]:
            q, k, v = _rand(rng, (3, B, H, N, d))
            scale = 0.7
            o, lse = orc.attention_fwd(q, k, v, scale, causal)
            for b in range(B):
                for h in range(H):
                    x = scale * (q[b, h] @ k[b, h].T)
                    x = np.where(_allowed(N, causal), x, -np.inf)
                    p = sps.softmax(x, axis=1)
                    np.testing.assert_allclose(o[b, h], p @ v[b, h], rtol=0, atol=1e-13)
                    np.testing.assert_allclose(lse[b, h], sps.logsumexp(x, axis=1), rtol=0,
                                               atol=1e-13)


@pin
def pin_online_merge_equals_two_pass(orc):
    """Block-merged online softmax (random column splits) equals the naive result."""
    rng = np.random.default_rng(12)
    B, H, N, d = 1, 2, 61, 8
    q, k, v = _rand(rng, (3, B, H, N, d))
    q *= 3.0  # wide logits so the running max moves a lot

    def splits(n):
        cuts = sorted(set(rng.integers(1, max(n, 2), size=min(n, 5)).tolist()))
        return [c for c in cuts if 0 < c < n]

    for causal in (False, True):
        o_ref, lse_ref = orc.attention_fwd(q, k, v, 0.5, causal)
        o_t, lse_t = online_softmax.attention_online(q, k, v, 0.5, causal, splits)
        np.testing.assert_allclose(o_ref, o_t, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse_ref, lse_t, rtol=0, atol=1e-12)
        # deferred-normalisation form with fixed 16-key blocks
        for b in range(B):
            for h in range(H):
                x = 0.5 * (q[b, h] @ k[b, h].T)
                for i in range(N):
                    n = i + 1 if causal else N
                    oo, ll = online_softmax.row_deferred(x[i, :n], v[b, h, :n], 16)
                    np.testing.assert_allclose(o_ref[b, h, i], oo, rtol=0, atol=1e-12)
                    assert abs(lse_ref[b, h, i] - ll) < 1e-12


@pin
def pin_probabilities_sum_to_one_and_convex_hull(orc):
    """sum_j exp(x_ij - LSE_i) = 1, and each O_i lies inside the box of its visible V rows."""
    rng = np.random.default_rng(13)
    B, H, N, d = 2, 2, 40, 8
    q, k, v = _rand(rng, (3, B, H, N, d))
    for causal in (False, True):
        o, lse = orc.attention_fwd(q, k, v, 0.9, causal)
        for b in range(B):
            for h in range(H):
                x = 0.9 * (q[b, h] @ k[b, h].T)
                x = np.where(_allowed(N, causal), x, -np.inf)
                s = np.exp(x - lse[b, h][:, None]).sum(axis=1)
                np.testing.assert_allclose(s, 1.0, rtol=0, atol=1e-13)
                for i in range(N):
                    vis = v[b, h, : (i + 1 if causal else N)]
                    assert np.all(o[b, h, i] <= vis.max(axis=0) + 1e-13)
                    assert np.all(o[b, h, i] >= vis.min(axis=0) - 1e-13)


@pin
def pin_identical_keys_give_mean_of_values(orc):
    """Identical K rows: P uniform, O_i = mean of visible V rows, LSE_i = s q_i.k + log|J_i|."""
    rng = np.random.default_rng(14)
    B, H, N, d = 1, 1, 33, 8
    q, _, v = _rand(rng, (3, B, H, N, d))
    k = np.broadcast_to(_rand(rng, (1, 1, 1, d)), (B, H, N, d)).copy()
    for causal in (False, True):
        o, lse = orc.attention_fwd(q, k, v, 0.3, causal)
        for i in range(N):
            n = i + 1 if causal else N
            np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n].mean(axis=0), rtol=0, atol=1e-13)
            want = 0.3 * float(q[0, 0, i] @ k[0, 0, 0]) + np.log(n)
            assert abs(lse[0, 0, i] - want) < 1e-13


@pin
def pin_dominant_logit_selects_its_value_row(orc):
    """One key far above the rest: O_i = v_J and LSE_i = x_iJ within N e^-50."""
    rng = np.random.default_rng(15)
    B, H, N, d = 1, 1, 24, 8
    q, k, v = _rand(rng, (3, B, H, N, d))
    i, J = 17, 5
    qi = q[0, 0, i]
    k[0, 0, J] = 80.0 * qi / np.linalg.norm(qi) ** 2  # x_iJ = 80 (scale 1)
    k[0, 0, np.arange(N) != J] *= 0.1
    o, lse = orc.attention_fwd(q, k, v, 1.0, False)
    x = q[0, 0, i] @ k[0, 0].T
    gap = x[J] - np.max(np.delete(x, J))
    assert gap > 50
    eps = np.finfo(np.float64).eps
    bound = N * np.exp(-50.0) * (1 + np.abs(v).max()) + 8 * eps * np.abs(v).max()
    np.testing.assert_allclose(o[0, 0, i], v[0, 0, J], rtol=0, atol=bound)
    # the LSE bound adds fp64 rounding of x_iJ = 80 itself
    assert abs(lse[0, 0, i] - x[J]) <= N * np.exp(-50.0) + 8 * eps * abs(x[J])


@pin
def pin_shift_invariance(orc):
    """K <- K + u shifts row i's logits by s q_i.u: O unchanged, LSE shifted by that constant.
    V <- V + c shifts every O_i by c (rows of P sum to one)."""
    rng = np.random.default_rng(16)
    B, H, N, d = 1, 2, 29, 8
    q, k, v = _rand(rng, (3, B, H, N, d))
    u = _rand(rng, (d,))
    c = _rand(rng, (d,))
    for causal in (False, True):
        o0, l0 = orc.attention_fwd(q, k, v, 0.6, causal)
        o1, l1 = orc.attention_fwd(q, k + u, v, 0.6, causal)
        o2, _ = orc.attention_fwd(q, k, v + c, 0.6, causal)
        np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l1 - l0, 0.6 * (q @ u), rtol=0, atol=1e-12)
        np.testing.assert_allclose(o2, o0 + c, rtol=0, atol=1e-12)


@pin
def pin_causal_first_rows(orc):
    """Causal row 0 is v_0 with LSE x_00; row 1 is the two-way logistic mix of v_0 and v_1."""
    rng = np.random.default_rng(17)
    B, H, N, d = 1, 1, 9, 4
    q, k, v = _rand(rng, (3, B, H, N, d))
    s = 0.8
    o, lse = orc.attention_fwd(q, k, v, s, True)
    x00 = s * q[0, 0, 0] @ k[0, 0, 0]
    np.testing.assert_array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - x00) < 1e-14
    x10, x11 = s * q[0, 0, 1] @ k[0, 0, 0], s * q[0, 0, 1] @ k[0, 0, 1]
    w0 = 1.0 / (1.0 + np.exp(x11 - x10))
    w1 = 1.0 / (1.0 + np.exp(x10 - x11))
    np.testing.assert_allclose(o[0, 0, 1], w0 * v[0, 0, 0] + w1 * v[0, 0, 1], rtol=0, atol=1e-14)
    assert abs(lse[0, 0, 1] - np.logaddexp(x10, x11)) < 1e-14


@pin
def pin_key_permutation_and_head_independence(orc):
    """Non-causal output is invariant to a joint permutation of (K, V) rows; heads and batch
    entries are independent problems."""
    rng = np.random.default_rng(18)
    B, H, N, d = 2, 3, 21, 8
    q, k, v = _rand(rng, (3, B, H, N, d))
    o, lse = orc.attention_fwd(q, k, v, 0.4, False)
    perm = rng.permutation(N)
    op, lp = orc.attention_fwd(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    np.testing.assert_allclose(op, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lp, lse, rtol=0, atol=1e-13)
    hp = [2, 0, 1]
    oh, lh = orc.attention_fwd(q[:, hp], k[:, hp], v[:, hp], 0.4, False)
    np.testing.assert_array_equal(oh, o[:, hp])
    np.testing.assert_array_equal(lh, lse[:, hp])


@pin
def pin_row_sampling_matches_full(orc):
    """Asking for a subset of rows returns exactly those rows of the full evaluation."""
    rng = np.random.default_rng(19)
    B, H, N, d = 1, 2, 70, 8
    q, k, v = _rand(rng, (3, B, H, N, d))
    rows = [0, 1, 5, 64, 69]
    for causal in (False, True):
        o, lse = orc.attention_fwd(q, k, v, 0.5, causal)
        os_, ls_ = orc.attention_fwd(q, k, v, 0.5, causal, rows=rows)
        np.testing.assert_array_equal(os_, o[:, :, rows])
        np.testing.assert_array_equal(ls_, lse[:, :, rows])


@pin
def pin_operand_decoding(orc):
    """bf16 and e4m3fn bit patterns decode to torch's values for every code; e4m3's largest
    finite value is 448 ("FlashAttention · InkStack", section 3.3.3 "Scaling")."""
    codes = np.arange(256, dtype=np.uint8)
    got = orc.decode(codes, "e4m3")
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert np.nanmax(got) == 448.0
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    gb = orc.decode(bits, "bf16")
    wb = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    wb = wb.numpy()
    fin = np.isfinite(wb)
    np.testing.assert_array_equal(gb[fin], wb[fin])


@pin
def pin_descaled_fp8_equals_f64_on_decoded_values(orc):
    """e4m3 operands with per-tensor descales give the f64 result on (code value x descale)."""
    rng = np.random.default_rng(20)
    B, H, N, d = 1, 2, 19, 16
    raw = rng.integers(0, 256, size=(3, B, H, N, d), dtype=np.uint8)
    raw[(raw & 0x7F) == 0x7F] = 0x38  # no NaN codes
    dq, dk, dv = 0.013, 0.021, 0.009
    vals = torch.from_numpy(raw.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for causal in (False, True):
        o8, l8 = orc.attention_fwd(raw[0], raw[1], raw[2], 0.25, causal, "e4m3", (dq, dk, dv))
        o64, l64 = orc.attention_fwd(vals[0] * dq, vals[1] * dk, vals[2] * dv, 0.25, causal)
        np.testing.assert_allclose(o8, o64, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l8, l64, rtol=1e-12, atol=1e-12)


def _e4m3_values(raw):
    return torch.from_numpy(raw.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _random_codes(rng, shape):
    raw = rng.integers(0, 256, size=shape, dtype=np.uint8)
    raw[(raw & 0x7F) == 0x7F] = 0x38  # no NaN codes
    return raw


@pin
def pin_block_descales_equal_f64_on_expanded_values(orc):
    """Per-block descales (one per 16-row block of each head, all different) give the f64
    result on code value x the descale of the row's block, the expansion done here with
    numpy's repeat ("FlashAttention · InkStack", section 3.3.1 "Block Quantization")."""
    rng = np.random.default_rng(21)
    B, H, N, d, blk = 2, 2, 37, 8, 16
    nblk = -(-N // blk)
    raw = _random_codes(rng, (3, B, H, N, d))
    vals = _e4m3_values(raw)
    sc = np.exp2(rng.uniform(-7, -3, size=(3, B, H, nblk)))
    full = [vals[t] * np.repeat(sc[t], blk, axis=2)[:, :, :N, None] for t in range(3)]
    for causal in (False, True):
        ob, lb = orc.attention_fwd_blockscaled(raw[0], raw[1], raw[2], 0.5, causal, "e4m3",
                                               sc[0], sc[1], sc[2], blk)
        o64, l64 = orc.attention_fwd(full[0], full[1], full[2], 0.5, causal)
        np.testing.assert_allclose(ob, o64, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lb, l64, rtol=1e-12, atol=1e-12)


@pin
def pin_uniform_block_descales_equal_per_tensor(orc):
    """Block descales that are all equal reduce to the per-tensor descaled result
    ("FlashAttention · InkStack", section 3.3.3 "Scaling")."""
    rng = np.random.default_rng(22)
    B, H, N, d = 1, 3, 40, 16
    raw = _random_codes(rng, (3, B, H, N, d))
    dq, dk, dv = 0.011, 0.017, 0.023
    for blk in (8, 128):
        nblk = -(-N // blk)
        s = [np.full((B, H, nblk), x) for x in (dq, dk, dv)]
        ob, lb = orc.attention_fwd_blockscaled(raw[0], raw[1], raw[2], 0.3, True, "e4m3",
                                               *s, blk)
        ot, lt = orc.attention_fwd(raw[0], raw[1], raw[2], 0.3, True, "e4m3", (dq, dk, dv))
        np.testing.assert_allclose(ob, ot, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lb, lt, rtol=1e-12, atol=1e-12)


def _torch_grads(q, k, v, dout, scale, causal):
    """Reference gradients from torch autograd in fp64 (a library routine)."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        n = s.shape[-1]
        s = s.masked_fill(~torch.ones(n, n, dtype=torch.bool).tril(), float("-inf"))
    o = torch.softmax(s, dim=-1) @ tv
    o.backward(torch.tensor(dout, dtype=torch.float64))
    return o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pin
def pin_backward_matches_torch_autograd(orc):
    """dQ, dK, dV of L = sum(O * dO) equal torch autograd's on small shapes ("FlashAttention ·
    InkStack", section 1.2.1: dV = P^T dO, dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q)."""
    rng = np.random.default_rng(40)
    for causal in (False, True):
        for (B, H, N, d) in [(1, 1, 1, 2), (1, 2, 7, 4), (2, 1, 33, 8)]:
            q, k, v, do = rng.standard_normal((4, B, H, N, d))
            g = orc.attention_bwd(q, k, v, do, 0.6, causal)
            o, dq, dk, dv = _torch_grads(q, k, v, do, 0.6, causal)
            for got, want in ((g["o"], o), (g["dq"], dq), (g["dk"], dk), (g["dv"], dv)):
                np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@pin
def pin_backward_finite_differences(orc):
    """Central differences of L = sum(O * dO) through the oracle's own forward agree with its
    gradients (no library involved)."""
    rng = np.random.default_rng(41)
    B, H, N, d = 1, 1, 6, 3
    q, k, v, do = rng.standard_normal((4, B, H, N, d))
    g = orc.attention_bwd(q, k, v, do, 0.9, True)

    def loss(q_, k_, v_):
        o, _ = orc.attention_fwd(q_, k_, v_, 0.9, True)
        return float((o * do).sum())

    h = 1e-6
    for name, arr in (("dq", q), ("dk", k), ("dv", v)):
        for idx in [(0, 0, 0, 0), (0, 0, 3, 1), (0, 0, N - 1, d - 1)]:
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args_p = [plus if a is arr else a for a in (q, k, v)]
            args_m = [minus if a is arr else a for a in (q, k, v)]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - g[name][idx]) < 1e-7, (name, idx, fd, g[name][idx])


@pin
def pin_backward_delta_identity(orc):
    """D_i = dO_i . O_i equals sum_j P_ij dP_ij with dP = dO V^T ("FlashAttention · InkStack",
    section 1.2.1), P taken from scipy's softmax."""
    rng = np.random.default_rng(42)
    B, H, N, d = 1, 2, 20, 5
    q, k, v, do = rng.standard_normal((4, B, H, N, d))
    g = orc.attention_bwd(q, k, v, do, 0.4, False)
    for h in range(H):
        p = sps.softmax(0.4 * q[0, h] @ k[0, h].T, axis=1)
        dp = do[0, h] @ v[0, h].T
        np.testing.assert_allclose(g["delta"][0, h], (p * dp).sum(axis=1), rtol=0, atol=1e-12)


@pin
def pin_backward_causal_last_key(orc):
    """Under the causal mask only the last query sees the last key: dV_{N-1} = P_{N-1,N-1} dO_{N-1}
    and dK_{N-1} = scale dS_{N-1,N-1} q_{N-1}."""
    rng = np.random.default_rng(43)
    B, H, N, d = 1, 1, 9, 4
    q, k, v, do = rng.standard_normal((4, B, H, N, d))
    g = orc.attention_bwd(q, k, v, do, 0.5, True)
    x = 0.5 * q[0, 0, -1] @ k[0, 0].T
    p = sps.softmax(x)
    dp = do[0, 0, -1] @ v[0, 0].T
    ds = p * (dp - (p * dp).sum())
    np.testing.assert_allclose(g["dv"][0, 0, -1], p[-1] * do[0, 0, -1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dk"][0, 0, -1], 0.5 * ds[-1] * q[0, 0, -1], rtol=0, atol=1e-12)


@pin
def pin_backward_key_shift_invariance(orc):
    """K <- K + u shifts every score of row i by the same amount, so P, dV and dQ are unchanged
    (the rows of dS sum to zero)."""
    rng = np.random.default_rng(44)
    B, H, N, d = 1, 1, 15, 6
    q, k, v, do = rng.standard_normal((4, B, H, N, d))
    u = rng.standard_normal(d)
    for causal in (False, True):
        g0 = orc.attention_bwd(q, k, v, do, 0.7, causal)
        g1 = orc.attention_bwd(q, k + u, v, do, 0.7, causal)
        np.testing.assert_allclose(g1["dq"], g0["dq"], rtol=0, atol=1e-11)
        np.testing.assert_allclose(g1["dv"], g0["dv"], rtol=0, atol=1e-11)
