"""Seeded synthetic inputs for the fused exact-attention forward.

This module is shared by the oracle's tests, the GPU parity tests, ``bench.py`` and the smoke
check.  It holds no attention arithmetic: only the workload table, random draws, rounding of the
draws to the operand dtype, the per-tensor fp8 input quantisation and the choice of sampled rows.

Input recipe (the same bytes go to the CUDA path and to the oracle):

* ``torch.Generator('cpu').manual_seed(seed)``; then ``randn`` fp32 for Q, then K, then V, each of
  shape ``[B, H, N, d]`` (head dim contiguous), in that order.
* bf16 operands: round-to-nearest-even of the fp32 draw (``Tensor.to(torch.bfloat16)``).  A
  ``q_mult`` (a power of two) is applied after the rounding, so it is exact.
* fp8-e4m3 operands: per-tensor descale ``amax(|X|) / 448`` (the format's largest finite value)
  and ``X_q = e4m3(RNE(X / descale))`` as in the per-tensor scaling of the FlashAttention
  explainer page (section 3.3.3 "Scaling").  The kernel and the oracle both receive ``X_q`` and the
  descale; the quantisation error itself is not part of the comparison.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    """One attention-forward problem: shapes, mask, operand dtype and seed."""

    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    dtype: str  # "bf16" or "e4m3"
    seed: int
    q_mult: float = 1.0
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4·B·H·N²·d, halved for the causal mask (the usual attention-forward convention)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def rows(self) -> int:
        return self.B * self.H * self.N

    def score_matrix_bytes(self, elem_bytes: int) -> int:
        """Bytes of one materialised N x N score (or probability) matrix per head: what the
        fused path never writes."""
        return self.N * self.N * elem_bytes

    def io_bytes(self, out_elem_bytes: int = 2) -> int:
        """HBM bytes the fused forward must move: Q, K, V read once, O and the fp32 LSE written
        once."""
        elem = 1 if self.dtype == "e4m3" else 2
        return self.rows * self.d * (3 * elem + out_elem_bytes) + 4 * self.rows

    def describe(self) -> str:
        mask = "causal" if self.causal else "non-causal"
        qm = f" Q*{self.q_mult:g}" if self.q_mult != 1.0 else ""
        return f"B{self.B} H{self.H} N{self.N} d{self.d} {self.dtype} {mask}{qm}"


# The five benchmark shapes of the method (plus the Q*8 stress variant of the causal one).
WORKLOADS = {
    "b1h1n256d64_bf16": Workload("b1h1n256d64_bf16", 1, 1, 256, 64, False, "bf16", 1000,
                                 note="small case the oracle finishes in well under a second"),
    "b4h16n2048d128_bf16_causal": Workload("b4h16n2048d128_bf16_causal", 4, 16, 2048, 128, True,
                                           "bf16", 1001),
    "b4h16n2048d128_bf16_causal_q8": Workload("b4h16n2048d128_bf16_causal_q8", 4, 16, 2048, 128,
                                              True, "bf16", 1001, q_mult=8.0,
                                              note="logits spread over about +-100"),
    "b2h32n8192d128_bf16": Workload("b2h32n8192d128_bf16", 2, 32, 8192, 128, False, "bf16", 1002,
                                    note="headline throughput shape"),
    "b1h16n32768d64_bf16_causal": Workload("b1h16n32768d64_bf16_causal", 1, 16, 32768, 64, True,
                                           "bf16", 1003, note="long sequence"),
    "b2h32n16384d128_e4m3": Workload("b2h32n16384d128_e4m3", 2, 32, 16384, 128, False, "e4m3",
                                     1004, note="fp8 operands, per-tensor descale"),
    # not one of the method's benchmark shapes: the fp8 shape under the causal mask (its first
    # query block of every head takes the f16 P V product)
    "b2h32n16384d128_e4m3_causal": Workload("b2h32n16384d128_e4m3_causal", 2, 32, 16384, 128,
                                            True, "e4m3", 1005,
                                            note="fp8 operands, per-tensor descale, causal"),
    # not one of the method's benchmark shapes: half the fp8 shape's batch, for counter captures
    # (2.7 GB on the device instead of 5.4)
    "b1h32n16384d128_e4m3": Workload("b1h32n16384d128_e4m3", 1, 32, 16384, 128, False, "e4m3",
                                     1006, note="fp8 operands, per-tensor descale, half batch"),
    # not one of the method's benchmark shapes: a single long sequence with too few query blocks
    # to fill the GPU, where splitting the keys over CTAs (split-KV) pays
    "b1h1n16384d128_bf16": Workload("b1h1n16384d128_bf16", 1, 1, 16384, 128, False, "bf16", 1100,
                                    note="64 CTAs without key splits"),
}

HEADLINE = "b2h32n8192d128_bf16"


@dataclass
class Inputs:
    """Operands on the host.  ``q``/``k``/``v`` are bf16 or float8_e4m3fn CPU tensors."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    descale_q: float = 1.0
    descale_k: float = 1.0
    descale_v: float = 1.0

    @property
    def dtype(self) -> str:
        return "e4m3" if self.q.dtype == torch.float8_e4m3fn else "bf16"

    def raw(self, name: str):
        """The operand's bytes as a numpy array (uint16 for bf16, uint8 for e4m3)."""
        t = getattr(self, name).contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view("uint16")
        return t.view(torch.uint8).numpy()


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor fp8 quantisation: returns (e4m3 tensor, fp32 descale)."""
    amax = float(x.abs().max())
    descale = amax / E4M3_MAX if amax > 0 else 1.0
    xq = (x / torch.tensor(descale, dtype=torch.float32)).to(torch.float8_e4m3fn)
    return xq, descale


def random_inputs(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0,
                  q_mult: float = 1.0) -> Inputs:
    """iid N(0,1) draws for Q, K, V in that order, rounded to the operand dtype."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if dtype == "bf16":
        qb = q.to(torch.bfloat16)
        if q_mult != 1.0:
            qb = qb * q_mult
        return Inputs(qb, k.to(torch.bfloat16), v.to(torch.bfloat16))
    if dtype == "e4m3":
        if q_mult != 1.0:
            q = q * q_mult
        qq, dq = quantize_e4m3(q)
        kq, dk = quantize_e4m3(k)
        vq, dv = quantize_e4m3(v)
        return Inputs(qq, kq, vq, dq, dk, dv)
    raise ValueError(f"unknown operand dtype {dtype!r}")


def outlier_inputs(B: int, H: int, N: int, d: int, seed: int = 0) -> Inputs:
    """Q, K, V with heavy-tailed entries N(0,1) + N(0,100)·Bernoulli(0.001), the outlier
    distribution of the pages' fp8 accuracy study ("FlashAttention 完全拆解（三）", section
    "数值误差验证"), drawn in fp32 (Q, then K, then V; per tensor: normal part, outlier part,
    Bernoulli mask) and rounded to bf16."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (B, H, N, d)
    out = []
    for _ in range(3):
        base = torch.randn(shape, generator=g, dtype=torch.float32)
        big = torch.randn(shape, generator=g, dtype=torch.float32) * 10.0
        mask = torch.rand(shape, generator=g, dtype=torch.float32) < 0.001
        out.append((base + big * mask).to(torch.bfloat16))
    return Inputs(*out)


def hadamard_signs(d: int, seed: int) -> torch.Tensor:
    """A seeded random +-1 vector of length d (fp32), the diagonal of the incoherent transform."""
    g = torch.Generator(device="cpu").manual_seed(seed + 4242)
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.float32)


@dataclass
class BlockScaledInputs:
    """e4m3 codes with one fp32 descale per 128-row block of each head ([B, H, nblk])."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dq: torch.Tensor
    dk: torch.Tensor
    dv: torch.Tensor

    def raw(self, name: str):
        return getattr(self, name).contiguous().view(torch.uint8).numpy()


def blockscaled_inputs(B: int, H: int, N: int, d: int, seed: int = 0,
                       spread_log2: float = 0.5, v_spread_log2: float = 1.0,
                       v_pow2: bool = True) -> BlockScaledInputs:
    """Random operands for the block-scaled fp8 path: the per-tensor e4m3 codes of
    ``random_inputs`` and, for every 128-row block, a descale equal to the per-tensor one times
    2^u, u uniform in [-spread, spread] (seeded; Q, K, V in that order; ``v_spread_log2`` for
    V).  With ``v_pow2`` the value descales are rounded to the nearest power of two."""
    base = random_inputs(B, H, N, d, "e4m3", seed)
    g = torch.Generator(device="cpu").manual_seed(seed + 9191)
    nblk = -(-N // 128)
    ds = []
    for i, d0 in enumerate((base.descale_q, base.descale_k, base.descale_v)):
        spread = v_spread_log2 if i == 2 else spread_log2
        u = (torch.rand((B, H, nblk), generator=g, dtype=torch.float64) * 2 - 1) * spread
        e = math.log2(d0) + u
        if i == 2 and v_pow2:
            e = torch.round(e)
        ds.append(torch.exp2(e).to(torch.float32))
    return BlockScaledInputs(base.q, base.k, base.v, *ds)


@dataclass
class BwdInputs:
    """Operands of the backward pass: Q, K, V and the output gradient dO, bf16 [B, H, N, d]."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor

    def raw(self, name: str):
        return getattr(self, name).contiguous().view(torch.int16).numpy().view("uint16")


def random_bwd_inputs(B: int, H: int, N: int, d: int, seed: int = 0) -> BwdInputs:
    """iid N(0,1) draws for Q, K, V, then dO (in that order), rounded to bf16."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q, k, v, do = (torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
                   for _ in range(4))
    return BwdInputs(q, k, v, do)


def make_inputs(w: Workload) -> Inputs:
    return random_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, w.q_mult)


def sample_rows(N: int, seed: int, extra: int = 56):
    """Deterministic query rows checked one by one at full size: tile edges plus seeded picks."""
    fixed = {0, 1, 2, 127, 128, 255, 256, N - 1}
    rows = {r for r in fixed if 0 <= r < N}
    g = torch.Generator(device="cpu").manual_seed(seed + 7777)
    if N > len(rows):
        pick = torch.randperm(N, generator=g)[: extra + len(rows)].tolist()
        for r in pick:
            if len(rows) >= len(fixed) + extra:
                break
            rows.add(int(r))
    return sorted(rows)
