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
// One CTA per (128-row block, head): 8 warps of 16 rows.  A row is spread over d / 8 lanes
// holding 8 consecutive elements each (16-byte loads, 8-byte stores, every access coalesced), so
// the transform's first three butterfly levels stay in registers and the rest are lane shuffles
// within the row's lane group.  The block's values stay in registers between the amax pass and
// the conversion pass: the operand is read once and the codes written once.
//
// Arithmetic (fp32): the transform's butterflies and its 1/sqrt(d) factor, descale =
// amax / 448 and the quotient x / descale, both correctly rounded; then round-to-nearest-even
// onto e4m3 with saturation at 448 (cvt.rn.satfinite).  A block whose amax is 0 gets descale 1.
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
__global__ void __launch_bounds__(kQuantThreads)
    quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                         float* __restrict__ descales, const float* __restrict__ signs, int n,
                         int nblk, bool pow2) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerStep = 32 / kLanesPerRow;
  constexpr int kSteps = 16 / kRowsPerStep;
  __shared__ float warp_amax[kQuantThreads / 32];

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int blk = blockIdx.x;
  const size_t bh = blockIdx.y;
  const int col = (lane % kLanesPerRow) * 8;
  const int row_base = blk * kQuantRows + warp * 16 + lane / kLanesPerRow;
  const size_t head = bh * static_cast<size_t>(n) * D;

  float v[kSteps][8];
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int row = row_base + st * kRowsPerStep;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (row < n) raw = __ldg(reinterpret_cast<const uint4*>(x + head + static_cast<size_t>(row) * D + col));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[st][2 * i] = __uint_as_float(w[i] << 16);
      v[st][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }

  if constexpr (HADAMARD) {
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(signs + col));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(signs + col + 4));
    const float sg[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    // 1 / sqrt(d): exact for d = 64; the fp32 value nearest 2^-3.5 for d = 128
    constexpr float kNorm = D == 64 ? 0.125f : 0.0883883461356163f;
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[st][e] *= sg[e];
      // element index = col + e: bits 0-2 live in registers, the higher bits across lanes
#pragma unroll
      for (int hb = 1; hb < 8; hb *= 2)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (!(e & hb)) {
            const float a = v[st][e], b = v[st][e + hb];
            v[st][e] = a + b;
            v[st][e + hb] = a - b;
          }
#pragma unroll
      for (int hl = 1; hl < kLanesPerRow; hl *= 2) {
        const bool upper = (lane & hl) != 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float other = __shfl_xor_sync(0xffffffffu, v[st][e], hl);
          v[st][e] = upper ? other - v[st][e] : v[st][e] + other;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) v[st][e] *= kNorm;
    }
  }

  float amax = 0.f;
#pragma unroll
  for (int st = 0; st < kSteps; ++st)
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[st][e]));
#pragma unroll
  for (int off = 16; off >= 1; off /= 2) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) warp_amax[warp] = amax;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, warp_amax[w]);
  float descale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (pow2) {
    // the smallest power of two >= the quotient (2^-126 for a subnormal quotient)
    const uint32_t b = __float_as_uint(descale);
    descale = __uint_as_float((b & 0x007FFFFFu) ? ((b & 0x7F800000u) + 0x00800000u) : b);
  }
  if (threadIdx.x == 0) descales[bh * nblk + blk] = descale;

#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int row = row_base + st * kRowsPerStep;
    uint32_t packed[2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
      packed[i] = pack_e4m3x4(__fdiv_rn(v[st][4 * i], descale), __fdiv_rn(v[st][4 * i + 1], descale),
                              __fdiv_rn(v[st][4 * i + 2], descale),
                              __fdiv_rn(v[st][4 * i + 3], descale));
    if (row < n)
      *reinterpret_cast<uint2*>(codes + head + static_cast<size_t>(row) * D + col) =
          make_uint2(packed[0], packed[1]);
  }
}

}  // namespace exattn
