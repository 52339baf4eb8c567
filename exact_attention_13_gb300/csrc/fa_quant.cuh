// fa_quant.cuh -- fp8 (e4m3) block quantiser for the attention operands, with optional
// incoherent processing.
//
// Block quantisation ("FlashAttention · InkStack", section 3.3.1 "Block Quantization", and
// section 3.3.3 "Scaling"): each block of 128 consecutive rows of one head -- the attention
// kernel's tile -- gets its own descale amax(|X_blk|) / 448 and codes e4m3(X / descale).
// Incoherent processing (same page, section 3.3.2): before quantising, rows may be multiplied
// by M = diag(s) H / sqrt(d), s a +-1 vector and H the Sylvester-Hadamard matrix, evaluated with
// the fast Walsh-Hadamard transform in O(d log d); applied to Q and K alike it leaves QK^T
// unchanged.
//
// One CTA per (128-row block, head): 8 warps of 16 rows.  A row is spread over d / 16 lanes
// holding 16 consecutive elements each (two 16-byte loads, one 16-byte store, every access
// coalesced), so the transform's first four butterfly levels stay in registers and the rest
// (three for d = 128, two for d = 64) are lane shuffles within the row's lane group.  The
// butterflies and the final scaling run two at a time in packed f32x2 instructions, each rounded
// as its scalar form (+2 % with the transform; the shuffles, not the arithmetic, bound it: 32
// elements per lane, one shuffle level fewer, measured 18 % slower, its 64-byte lane runs no
// longer coalesced).  The block's values stay in registers between the amax pass and
// the conversion pass: the operand is read once and the codes written once.
//
// Arithmetic (fp32): descale = amax / 448 and scale = 448 / amax, both correctly rounded
// quotients, once per block; then x * scale and round-to-nearest-even onto e4m3 with saturation
// at 448 (cvt.rn.satfinite).  A block whose amax is 0 gets descale and scale 1.  Without the
// transform this is exactly the reference definition.  With it, the butterflies run on the
// unnormalised +-1 matrix and the 1/sqrt(d) factor multiplies the block amax and the scale, so
// values agree with the fp64 transform to a few fp32 ulps and a code can differ only where the
// scaled value lies that close to a rounding midpoint.
// On request the descale is raised to the next power of two: e4m3's relative precision does not
// depend on the scale, the largest code then lies in (224, 448], and the attention kernel folds
// power-of-two value descales into P without any rounding.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace exattn {

constexpr int kQuantRows = 128;     // rows per block (one descale each)
constexpr int kQuantThreads = 256;  // 8 warps x 16 rows

template <int D, bool HADAMARD>
__global__ void __launch_bounds__(kQuantThreads, 3)
    quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                         float* __restrict__ descales, const float* __restrict__ signs, int n,
                         int nblk, bool pow2) {
  constexpr int kElems = 16;                        // consecutive elements per lane
  constexpr int kLanesPerRow = D / kElems;          // 8 (d = 128) or 4 (d = 64)
  constexpr int kRowsPerStep = 32 / kLanesPerRow;
  constexpr int kSteps = 16 / kRowsPerStep;         // a warp covers 16 rows
  __shared__ float warp_amax[kQuantThreads / 32];

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int blk = blockIdx.x;
  const size_t bh = blockIdx.y;
  const int col = (lane % kLanesPerRow) * kElems;
  const int row_base = blk * kQuantRows + warp * 16 + lane / kLanesPerRow;
  const size_t head = bh * static_cast<size_t>(n) * D;

  float v[kSteps][kElems];
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int row = row_base + st * kRowsPerStep;
    uint4 raw[kElems / 8];
#pragma unroll
    for (int q = 0; q < kElems / 8; ++q) raw[q] = make_uint4(0u, 0u, 0u, 0u);
    if (row < n) {
      const uint4* src = reinterpret_cast<const uint4*>(x + head + static_cast<size_t>(row) * D + col);
#pragma unroll
      for (int q = 0; q < kElems / 8; ++q) raw[q] = __ldg(src + q);
    }
#pragma unroll
    for (int q = 0; q < kElems / 8; ++q) {
      const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[st][8 * q + 2 * i] = __uint_as_float(w[i] << 16);
        v[st][8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  }

  // The transform runs unnormalised (entries of H are +-1); its 1/sqrt(d) is folded into the
  // block's amax and into the final multiplier.
  float norm = 1.f;
  if constexpr (HADAMARD) {
    // 1 / sqrt(d): exact for d = 64; the fp32 value nearest 2^-3.5 for d = 128
    norm = D == 64 ? 0.125f : 0.0883883461356163f;
    float sg[kElems];
#pragma unroll
    for (int q = 0; q < kElems / 4; ++q) {
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(signs + col) + q);
      sg[4 * q] = s4.x;
      sg[4 * q + 1] = s4.y;
      sg[4 * q + 2] = s4.z;
      sg[4 * q + 3] = s4.w;
    }
    // Two butterflies per packed f32x2 instruction, each rounded as its scalar form: a s + b
    // and a s - b (s = +-1, so a s is exact), a + b and a - b (as b (-1) + a), own s + other.
    const float2 neg1 = f32x2(-1.f, -1.f);
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
      // level 1 with the sign flip folded in: (a s_a + b s_b, a s_a - b s_b), pairs (e, e + 1)
      // and (e + 2, e + 3) side by side
#pragma unroll
      for (int e = 0; e < kElems; e += 4) {
        const float2 b2 = mul_f32x2(f32x2(v[st][e + 1], v[st][e + 3]), f32x2(sg[e + 1], sg[e + 3]));
        const float2 a2 = mul_f32x2(f32x2(v[st][e], v[st][e + 2]), f32x2(sg[e], sg[e + 2]));
        const float2 lo = add_f32x2(a2, b2);
        const float2 hi = fma_f32x2(b2, neg1, a2);
        v[st][e] = f32x2_lo(lo);
        v[st][e + 2] = f32x2_hi(lo);
        v[st][e + 1] = f32x2_lo(hi);
        v[st][e + 3] = f32x2_hi(hi);
      }
      // element index = col + e: bits 1-3 of e in registers (butterflies e and e + 1 side by
      // side), the higher bits across lanes
#pragma unroll
      for (int hb = 2; hb < kElems; hb *= 2)
#pragma unroll
        for (int e = 0; e < kElems; e += 2)
          if (!(e & hb)) {
            const float2 a2 = f32x2(v[st][e], v[st][e + 1]);
            const float2 b2 = f32x2(v[st][e + hb], v[st][e + hb + 1]);
            const float2 sum = add_f32x2(a2, b2);
            const float2 dif = fma_f32x2(b2, neg1, a2);
            v[st][e] = f32x2_lo(sum);
            v[st][e + 1] = f32x2_hi(sum);
            v[st][e + hb] = f32x2_lo(dif);
            v[st][e + hb + 1] = f32x2_hi(dif);
          }
#pragma unroll
      for (int hl = 1; hl < kLanesPerRow; hl *= 2) {
        // lower partner: own + other; upper partner: other - own
        const float ls = (lane & hl) ? -1.f : 1.f;
        const float2 ls2 = f32x2(ls, ls);
#pragma unroll
        for (int e = 0; e < kElems; e += 2) {
          const float o0 = __shfl_xor_sync(0xffffffffu, v[st][e], hl);
          const float o1 = __shfl_xor_sync(0xffffffffu, v[st][e + 1], hl);
          const float2 r2 = fma_f32x2(f32x2(v[st][e], v[st][e + 1]), ls2, f32x2(o0, o1));
          v[st][e] = f32x2_lo(r2);
          v[st][e + 1] = f32x2_hi(r2);
        }
      }
    }
  }

  float amax = 0.f;
#pragma unroll
  for (int st = 0; st < kSteps; ++st)
#pragma unroll
    for (int e = 0; e < kElems; ++e) amax = fmaxf(amax, fabsf(v[st][e]));
#pragma unroll
  for (int off = 16; off >= 1; off /= 2) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) warp_amax[warp] = amax;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, warp_amax[w]);
  amax *= norm;
  float descale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  float scale = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
  if (pow2) {
    // the smallest power of two >= the quotient (2^-126 for a subnormal quotient)
    const uint32_t b = __float_as_uint(descale);
    descale = __uint_as_float((b & 0x007FFFFFu) ? ((b & 0x7F800000u) + 0x00800000u) : b);
    scale = __fdiv_rn(1.f, descale);  // exact: a power of two
  }
  if (threadIdx.x == 0) descales[bh * nblk + blk] = descale;
  const float mult = scale * norm;  // norm = 1 without the transform: exact

#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int row = row_base + st * kRowsPerStep;
    uint32_t packed[kElems / 4];
    const float2 mult2 = f32x2(mult, mult);
#pragma unroll
    for (int i = 0; i < kElems / 4; ++i) {
      const float2 x01 = mul_f32x2(f32x2(v[st][4 * i], v[st][4 * i + 1]), mult2);
      const float2 x23 = mul_f32x2(f32x2(v[st][4 * i + 2], v[st][4 * i + 3]), mult2);
      packed[i] = pack_e4m3x4(f32x2_lo(x01), f32x2_hi(x01), f32x2_lo(x23), f32x2_hi(x23));
    }
    if (row < n)
      *reinterpret_cast<uint4*>(codes + head + static_cast<size_t>(row) * D + col) =
          make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

}  // namespace exattn
