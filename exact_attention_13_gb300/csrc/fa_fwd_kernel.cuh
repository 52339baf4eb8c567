// fa_fwd_kernel.cuh -- fused exact-attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// One CTA owns 256 query rows of one (batch, head): two 128-row Q tiles, h = 0, 1.  It streams
// the head's K/V in 128-row blocks through a ring of shared-memory slots and keeps, per row, the
// online-softmax state (running max m, running sum l) in registers and the unnormalised output
// in tensor memory ("FlashAttention · InkStack", sections 1.1.2 "Online Softmax" and 2.1; the
// two-tile ping-pong and TMEM plan of "FlashAttention4 精读", section "新pipeline来overlap matmul
// 和softmax").  Warp roles (384 threads; a separate correction warpgroup was measured and is
// slower on GB300, see the rescale note below):
//
//   warps 0-3  softmax, Q tile 0     one thread per query row: reads its S row from TMEM,
//   warps 4-7  softmax, Q tile 1     updates (m, l), rescales its O row when m grew (bf16: by more
//                                    than the lazy threshold), writes the
//                                    bf16/f16/e4m3 probabilities back into the S columns, and at the
//                                    end normalises O, stores it and the row's log-sum-exp
//   warp  8    TMA producer          Q tiles once, then K_j, V_j into the ring (full/empty
//                                    mbarriers, "FlashAttention · InkStack", section 3.2.1)
//   warp  9    MMA issuer            one elected lane issues S_h = Q_h K_j^T (both operands in smem)
//                                    and O_h += P_h V_j (P from TMEM, V from smem), and owns the
//                                    TMEM allocation
//   warps 10-11 V converters         (fp8 operands with an f16 P V product only) widen each
//                                    e4m3 V block to f16 in shared memory for the PV MMAs;
//                                    otherwise idle
//
// TMEM (512 columns x 128 lanes, fp32 cells): S_0 at columns 0-127, S_1 at 128-255 (P_h is
// written over S_h), O_0 at 256.., O_1 at 384.. .  Lane i holds row i of each tile.
//
// MMA issue order (tcgen05 MMAs from one thread execute in order):
//   S0(0) S1(0) | PV0(0) S0(1) PV1(0) S1(1) | PV0(1) S0(2) PV1(1) S1(2) | ...
// so the tensor core works on one tile while the other tile's softmax runs.  S_h(j+1) is issued
// after PV_h(j), which makes it safe to overwrite P_h; the commit that signals S_h(j+1) also
// proves PV_h(j) complete, so the softmax may rescale O_h right after it.
//
// Every mbarrier wait is bounded in time (globaltimer).  A wait that runs out sets a CTA-wide
// abort flag and the status word; all roles then leave their loops, the MMA thread drains its
// outstanding MMAs, the producer waits (bounded) for its outstanding copies, and the TMEM is
// freed before the CTA exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace exattn {

// Optional timeline trace (build with -DEXATTN_TRACE): one CTA records clock64() at the role
// hand-offs into a device buffer of 11 x 2 x kTraceMaxJ int64, for profiling the pipeline.
// Compiled out by default.
#ifdef EXATTN_TRACE
__device__ long long* g_trace_buf;
__device__ int g_trace_cta;
constexpr int kTraceMaxJ = 512;
#define EXATTN_TRACE_SETUP                                                                 \
  long long* const trace_buf =                                                             \
      ((int)(blockIdx.x + gridDim.x * blockIdx.y) == g_trace_cta) ? g_trace_buf : nullptr
#define EXATTN_TRACE_EVENT(kind, h, j)                                                     \
  do {                                                                                     \
    if (trace_buf && (j) < kTraceMaxJ) trace_buf[((kind) * 2 + (h)) * kTraceMaxJ + (j)] = clock64(); \
  } while (0)
#else
#define EXATTN_TRACE_SETUP \
  do {                     \
  } while (0)
#define EXATTN_TRACE_EVENT(kind, h, j) \
  do {                                 \
  } while (0)
#endif

constexpr int kThreads = 384;
// Warp roles: softmax warps 0-7, then the control warpgroup 8-11 (producer, MMA issuer, two V
// converters).  With the control warpgroup in warps 0-3 instead, the headline shape measured
// 2 % slower and the causal d128 shape 3 % slower (fp8 +1 %).
constexpr int kCtlWarp0 = 8;
constexpr int kProducerWarp = kCtlWarp0;
constexpr int kMmaWarp = kCtlWarp0 + 1;
constexpr int kConvWarp0 = kCtlWarp0 + 2;
constexpr int kSoftmaxWarp0 = 0;
// setmaxnreg split of the 384 x 168 launch registers: 128 x (2 kSoftmaxRegs + kCtlRegs)
#ifndef EXATTN_SOFTMAX_REGS
#define EXATTN_SOFTMAX_REGS 216
#endif
constexpr int kSoftmaxRegs = EXATTN_SOFTMAX_REGS;
constexpr int kCtlRegs = (384 * 168 - 256 * kSoftmaxRegs) / 128;
static_assert(kCtlRegs % 8 == 0 && kCtlRegs >= 24, "setmaxnreg takes multiples of 8");
constexpr int kTileRows = 128;       // query rows per Q tile, keys per K/V block
constexpr int kCtaRows = 2 * kTileRows;
constexpr int kStatusTimeout = 5;    // FA_ERR_DEVICE_TIMEOUT
#ifndef EXATTN_WAIT_LIMIT_NS
#define EXATTN_WAIT_LIMIT_NS 4000000000ull
#endif
constexpr uint64_t kWaitLimitNs = EXATTN_WAIT_LIMIT_NS;  // per wait (4 s in the library)
// Fault injection for the test of the timeout path (test builds only, never in the library):
// the producer loads the Q tiles and then stops, so the first K/V wait runs out and every role
// must leave through the abort path.
#ifndef EXATTN_INJECT_STALL
#define EXATTN_INJECT_STALL 0
#endif
constexpr float kLn2 = 0.6931471805599453f;
// Fraction of exponentials evaluated by the FMA polynomial instead of MUFU: one column in every
// EXATTN_EMU_EVERY of an unmasked block (0 = MUFU only).  On GB300 MUFU does 32 ex2/clk/SM and
// the softmax is issue-bound, so emulation costs time (1-in-8 measured -5..-7 %); off by default.
#ifndef EXATTN_EMU_EVERY
#define EXATTN_EMU_EVERY 0
#endif
// e4m3 P: exponentials two at a time by ex2.approx.f16x2 (unmasked blocks).  f16x2 ex2 runs at
// half the instruction rate of f32 ex2 (the same 32 results/clk/SM), so it saves issue slots
// but not MUFU time; off by default.
#ifndef EXATTN_EX2_F16X2
#define EXATTN_EX2_F16X2 0
#endif

// Format of the probabilities P handed to the P V product.
enum class PFmt { kBf16, kF16, kE4m3 };

template <bool FP8, bool PV16>
__host__ __device__ constexpr PFmt p_fmt() {
  return !FP8 ? PFmt::kBf16 : (PV16 ? PFmt::kF16 : PFmt::kE4m3);
}

// e4m3 probabilities are stored as 2^8 * p: the largest is 256 (< 448, the format's largest
// finite value) and p down to 2^-14 stays out of the subnormal range.  O and l carry the same
// factor, so it cancels in O / l; the LSE takes it back out.  bf16 and f16 P need no offset.
template <PFmt PF>
__host__ __device__ constexpr float p_offset_log2() {
  return PF == PFmt::kE4m3 ? 8.f : 0.f;
}

// Lazy rescale ("FlashAttention4 精读", section 3.1.4): a row's O and l are rescaled only when
// some row of the warp grew its max by more than this threshold (log2 units); otherwise the
// stale max stays and probabilities may reach 2^threshold.  bf16 and f16 P take the page's 8
// (p <= 256).  e4m3 P, stored with the offset 2^8, takes 0.8: its largest probability stays
// below 2^8.8 < 448, e4m3's largest finite value, and since a row's max mostly grows by less than
// that once a few blocks are in, most rescales are still skipped.  Builds with the FMA
// exponential (EXATTN_EMU_EVERY > 0) take 0: the normaliser correction below recomputes a
// block's largest probability with MUFU, which matches the loop's value only where the loop used
// MUFU for that column (at threshold 0 the row max is 2^offset exactly on both units).  The
// softmax warps rescale O themselves: a separate correction warpgroup (16 warps; the softmax
// posts alpha, four warps rescale O while the exponentials run) measured 9-16 % slower on GB300,
// because the 512-thread register split leaves the softmax 168 registers and the alpha -> O-ready
// hand-off lands on the MMA's path.  EXATTN_RESCALE_LOG2 overrides the bf16 threshold (test
// builds).
template <PFmt PF>
__host__ __device__ constexpr float rescale_log2() {
#if defined(EXATTN_RESCALE_LOG2)
  constexpr float kBf16 = EXATTN_RESCALE_LOG2;
#else
  constexpr float kBf16 = 8.f;
#endif
  return EXATTN_EMU_EVERY != 0 ? 0.f
                               : (PF == PFmt::kBf16 ? kBf16 : (PF == PFmt::kF16 ? 8.f : 0.8f));
}

// p rounded to P's format, as the conversions that write P round it (nearest even; e4m3
// saturating), back in fp32.
template <PFmt PF>
__device__ __forceinline__ float round_p(float p) {
  if constexpr (PF == PFmt::kBf16) {
    return __uint_as_float(pack_bf16x2(p, 0.f) << 16);
  } else if constexpr (PF == PFmt::kF16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(pack_f16x2(p, 0.f) & 0xFFFFu)));
  } else {
    const uint32_t h = e4m3x2_to_f16x2(static_cast<uint16_t>(pack_e4m3x4(p, 0.f, 0.f, 0.f) & 0xFFFFu));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
  }
}

// Design knobs (compile-time).  The defaults are the measured best on GB300 (A/B over whole
// launches of the headline shapes): bf16 prefers a short L2 prefetch, e4m3 (softmax-bound) a
// deeper one.  -D overrides apply to both operand types.
#ifndef EXATTN_KV_SLOTS_D128
#define EXATTN_KV_SLOTS_D128 4
#endif
#ifndef EXATTN_KV_SLOTS_PV16
#define EXATTN_KV_SLOTS_PV16 6
#endif
template <bool FP8>
__host__ __device__ constexpr int l2_prefetch_blocks() {
#ifdef EXATTN_L2_PREFETCH_BLOCKS
  return EXATTN_L2_PREFETCH_BLOCKS;
#else
  return FP8 ? 6 : 2;
#endif
}
// P is published in two parts of 64 keys: the P V MMAs of the first part run while the softmax
// computes the second.  (For bf16 P this measured -3 % while the MMA issue was the bottleneck;
// with the issue loop run by the whole warp it is +6 % on the headline shape.  Four parts of
// 32 keys measured 9-18 % slower: every part adds a hand-off to both sides.)
__host__ __device__ constexpr int p_parts() { return 2; }

struct KernelArgs {
  __nv_bfloat16* o;   // [BH, N, d]            (one key split)
  float* lse;         // [BH, N]               (one key split)
  float* o_part;      // [splits, BH, N, d]    (several key splits: O of each split, fp32)
  float* lse_part;    // [splits, BH, N]       (several key splits: LSE of each split)
  int* status;        // device status word (never null when launched by the library)
  int n;              // keys = queries per head
  int bh;             // batch * heads
  int mblock0;        // first 256-row query block of this launch (launches may cover a range)
  float c;            // scale * log2(e) * descale_q * descale_k
  float out_mult;     // descale_v (1 for bf16)
  // fp8 block scaling (null for per-tensor descales): one fp32 descale per 128-row block of
  // each head, [BH, nblk]; c and out_mult then carry no descale of their own
  const float* dq_blk;
  const float* dk_blk;
  const float* dv_blk;
  int nblk;
};

// Compile-time geometry of one instance.  PV16 (fp8 operands only): the P V product runs in
// f16 -- P rounded to f16 instead of e4m3, V widened from e4m3 to f16 in shared memory by a
// converter warp -- while S = Q K^T stays an fp8 product.
template <int D, bool FP8, bool PV16 = false>
struct Geo {
  static constexpr int kElem = FP8 ? 1 : 2;                 // bytes per operand element
  static constexpr int kRowBytes = D * kElem;               // bytes of one operand row
  static constexpr int kSwBytes = kRowBytes >= 128 ? 128 : kRowBytes;  // swizzle span
  static constexpr int kBoxes = kRowBytes / kSwBytes;       // TMA boxes per 128-row tile
  static constexpr int kBoxElems = kSwBytes / kElem;        // inner box extent (elements)
  static constexpr int kTileBytes = kTileRows * kRowBytes;  // one 128-row operand tile
  static constexpr bool kPv16 = FP8 && PV16;
  static constexpr bool kPE4m3 = FP8 && !PV16;              // P stored as e4m3
  static constexpr int kSlots = (FP8 && D == 128 && PV16)
                                    ? EXATTN_KV_SLOTS_PV16
                                    : ((FP8 || D == 64) ? 8 : EXATTN_KV_SLOTS_D128);  // ring depth
  static constexpr int kQBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kSlots * kTileBytes;
  // f16 copies of V (PV16): two buffers, each 128 keys x D in 128-byte swizzled boxes of 64
  // columns, the layout of a bf16 V tile
  static constexpr int kV16TileBytes = kTileRows * D * 2;
  static constexpr int kV16Bytes = kPv16 ? 2 * kV16TileBytes : 0;
  static constexpr uint32_t kSwMode = kSwBytes == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kKStepBytes = 32;                    // K extent of one MMA, in bytes
  static constexpr int kKStepsS = kRowBytes / kKStepBytes;  // MMAs per S = Q K^T
  static constexpr int kKeysPerPv = kPE4m3 ? 32 : 16;       // keys per PV MMA
  static constexpr int kPvSteps = kTileRows / kKeysPerPv;   // MMAs per O += P V
  static constexpr int kPCols = kPE4m3 ? 32 : 64;           // TMEM columns of one P row
  static constexpr int kPvSwBytes = kPv16 ? 128 : kSwBytes; // swizzle span of the PV B tile
  static constexpr uint32_t kIdescS = instr_desc(128, 128, FP8 ? 0 : 1, false, false);
  static constexpr uint32_t kIdescPV = instr_desc(128, D, FP8 ? 0 : 1, false, true);
  // descriptor offset (16-byte units) of K step kb of an S operand tile; 0 past the last step
  __host__ __device__ static constexpr int s_off(int kb) {
    return kb >= kKStepsS ? 0
                          : ((kb * kKStepBytes / kSwBytes) * kTileRows * kSwBytes +
                             (kb * kKStepBytes) % kSwBytes) >> 4;
  }
  // descriptor step (16-byte units) between the V key groups of consecutive PV MMAs
  static constexpr int kPvStep = (kKeysPerPv * kPvSwBytes) >> 4;
};

// Shared-memory control block (after the operand tiles).
template <int kSlots>
struct Ctrl {
  uint64_t q_full;
  uint64_t kv_full[kSlots];
  uint64_t kv_empty[kSlots];
  uint64_t s_full[2];
  uint64_t p_full[2][p_parts()];  // [tile][published part of the keys]
  uint64_t o_full[2];
  uint64_t s_read[2];     // the softmax warps of tile h have read S_h (head dim 64)
  uint64_t pv_done[2];    // P V of tile h's current block complete (head dim 64)
  uint64_t v16_full[2];   // f16 V buffer b written (PV16)
  uint64_t v16_empty[2];  // f16 V buffer b no longer read by the MMAs (PV16)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float dv_max[8];        // fp8 block scaling: the largest value descale, per softmax warp
};

template <int D, bool FP8, bool PV16 = false>
constexpr int smem_bytes() {
  using G = Geo<D, FP8, PV16>;
  return G::kQBytes + G::kRingBytes + G::kV16Bytes + (int)sizeof(Ctrl<G::kSlots>) + 1024;
}

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or the wait ran out.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, int* abort_flag,
                                           int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 127u) == 0) {
      if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
        atomicExch(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Key blocks Q tile h must visit: all of them, or (causal) those up to its diagonal block.
// A tile whose first row is past the end of the sequence visits none.
template <bool CAUSAL>
__device__ __forceinline__ int kv_blocks_for_tile(int row0, int n) {
  if (row0 >= n) return 0;
  const int total = (n + kTileRows - 1) / kTileRows;
  return CAUSAL ? (row0 / kTileRows + 1) : total;
}

// Softmax numerator of one row: p_i = 2^(s_i c - m) for the 128 keys of the block (keys >= lim
// are masked to 0 when MASKED; with EMU_EVERY > 0 one column in EMU_EVERY of an unmasked block
// uses the FMA polynomial, "FlashAttention4 精读", section 3.1.3 "partial emulation"), rounded
// to bf16 (or f16 or e4m3) and written to P's TMEM columns (t_s) in two parts of 64 keys; after
// each part the warp publishes on that part's P barrier.  pre_store() runs before the first store.
// Returns the fp32 sum of the unrounded p.
template <bool MASKED, PFmt PF, int P_PARTS, int EMU_EVERY, typename PreStore>
__device__ __forceinline__ float exp_and_publish(float (&s)[128], float c, float m, int lim,
                                                 uint32_t t_s, uint32_t bar0, int lane,
                                                 PreStore&& pre_store) {
  static_assert(P_PARTS == 2, "P is published in two parts of 64 keys");
  constexpr int kKeys = 128 / P_PARTS;   // keys per published part
#if EXATTN_EX2_F16X2
  if constexpr (PF == PFmt::kE4m3 && !MASKED && EMU_EVERY == 0) {
    // Two exponentials per MUFU instruction (ex2.approx.f16x2).  The argument leaves out P's
    // 2^8 offset, so it is at most 0.8 and its f16 rounding stays below 2^-11 absolute; p is
    // then scaled by 2^8 in f16 (exact) and converted to e4m3.  The row sum takes p pairwise in
    // f16 (one rounding) and accumulates in fp32.
    const float2 c2 = f32x2(c, c), nm2 = f32x2(-(m + 8.f), -(m + 8.f));
    float2 ps2[4] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f), f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
    for (int part = 0; part < P_PARTS; ++part) {
      uint32_t r[kKeys / 4];
#pragma unroll
      for (int q = 0; q < kKeys / 4; ++q) {
        const int i = kKeys * part + 4 * q;
        const float2 xa = fma_f32x2(f32x2(s[i], s[i + 1]), c2, nm2);
        const float2 xb = fma_f32x2(f32x2(s[i + 2], s[i + 3]), c2, nm2);
        uint32_t ha = pack_f16x2(f32x2_lo(xa), f32x2_hi(xa));
        uint32_t hb = pack_f16x2(f32x2_lo(xb), f32x2_hi(xb));
        ha = ex2_f16x2(ha);
        hb = ex2_f16x2(hb);
        r[q] = e4m3x4_from_f16x2_scaled256(ha, hb);
        const uint32_t hs = hadd_f16x2(ha, hb);
        ps2[q % 4] = add_f32x2(ps2[q % 4], f16x2_to_f32x2(hs));
      }
      if (part == 0) pre_store();
      tmem_st16(t_s + 16 * part, r);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar0 + 8 * part);
    }
    float ps[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ps[2 * k] = f32x2_lo(ps2[k]);
      ps[2 * k + 1] = f32x2_hi(ps2[k]);
    }
#pragma unroll
    for (int w = 4; w >= 1; w /= 2)
#pragma unroll
      for (int k = 0; k < w; ++k) ps[k] += ps[k + w];
    return ps[0] * 256.f;
  }
#endif
  // eight partial sums (element i goes to sum i % 8), kept as four packed pairs; the exponent
  // arguments s c - m are formed two at a time (same rounding as the scalar fma)
  float2 ps2[4] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f), f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
  const float2 c2 = f32x2(c, c), nm2 = f32x2(-m, -m);
#pragma unroll
  for (int part = 0; part < P_PARTS; ++part) {
#pragma unroll
    for (int i = kKeys * part; i < kKeys * part + kKeys; i += 2) {
      const float2 x2 = fma_f32x2(f32x2(s[i], s[i + 1]), c2, nm2);
      const float x0 = f32x2_lo(x2), x1 = f32x2_hi(x2);
      float p0, p1;
      if constexpr (MASKED) {
        p0 = i < lim ? ex2_mufu(x0) : 0.f;
        p1 = i + 1 < lim ? ex2_mufu(x1) : 0.f;
      } else if constexpr (EMU_EVERY > 0) {
        p0 = (i % EMU_EVERY == EMU_EVERY - 1) ? ex2_poly(x0) : ex2_mufu(x0);
        p1 = ((i + 1) % EMU_EVERY == EMU_EVERY - 1) ? ex2_poly(x1) : ex2_mufu(x1);
      } else {
        p0 = ex2_mufu(x0);
        p1 = ex2_mufu(x1);
      }
      s[i] = p0;
      s[i + 1] = p1;
      ps2[(i / 2) % 4] = add_f32x2(ps2[(i / 2) % 4], f32x2(p0, p1));
    }
    if (part == 0) pre_store();   // P's columns may still be read by the previous P V
    if constexpr (PF == PFmt::kE4m3) {
      // four keys per TMEM column
      uint32_t r[kKeys / 4];
#pragma unroll
      for (int i = 0; i < kKeys / 4; ++i) {
        const int k = kKeys * part + 4 * i;
        r[i] = pack_e4m3x4(s[k], s[k + 1], s[k + 2], s[k + 3]);
      }
      tmem_st16(t_s + 16 * part, r);
    } else {
      // two keys per TMEM column
      uint32_t r[kKeys / 2];
#pragma unroll
      for (int i = 0; i < kKeys / 2; ++i) {
        const int k = kKeys * part + 2 * i;
        r[i] = PF == PFmt::kF16 ? pack_f16x2(s[k], s[k + 1]) : pack_bf16x2(s[k], s[k + 1]);
      }
      tmem_st32(t_s + 32 * part, r);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar0 + 8 * part);   // p_full[h][part]
  }
  float ps[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ps[2 * k] = f32x2_lo(ps2[k]);
    ps[2 * k + 1] = f32x2_hi(ps2[k]);
  }
#pragma unroll
  for (int w = 4; w >= 1; w /= 2)
#pragma unroll
    for (int k = 0; k < w; ++k) ps[k] += ps[k + w];
  return ps[0];
}

template <int D, bool FP8, bool CAUSAL, bool PV16 = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                  const KernelArgs args) {
  using G = Geo<D, FP8, PV16>;
  constexpr PFmt kPFmt = p_fmt<FP8, PV16>();
  constexpr int kPHalves = p_parts();
  // Head dim 64 (not with the f16 P V product, whose converter warps need warps 10-11): O_h takes
  // 64 of its 128 TMEM columns and P_h the other 64, so S_h is free again as soon as the softmax
  // has read it, and each tile gets an issuing warp of its own (warps 9 and 10).  Measured on
  // B1 H16 N32768 d64 causal: 1017 -> 1084 TFLOPS.  (The two tiles' softmaxes then run in phase
  // and share MUFU; a single issuer polling both tiles without blocking measured 608: each probe
  // is a shared-memory round trip, so it reacted ~2000 cycles late.)
  constexpr bool kSepP = D == 64 && !G::kPv16;
  constexpr int kL2PrefetchBlocks = l2_prefetch_blocks<FP8>();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* s_q = smem;                          // two Q tiles
  uint8_t* s_ring = smem + G::kQBytes;          // K/V slots
  uint8_t* s_v16 = s_ring + G::kRingBytes;      // f16 V buffers (PV16)
  Ctrl<G::kSlots>* ctl = reinterpret_cast<Ctrl<G::kSlots>*>(s_v16 + G::kV16Bytes);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int n = args.n;
  EXATTN_TRACE_SETUP;
  // Launch order.  Non-causal: query blocks of one head are adjacent (x), so the CTAs sharing
  // that head's K/V run together and re-read it from L2.  Causal: heads are adjacent (x) and
  // query blocks run from the last (heaviest: it sees every key block) to the first (y), i.e.
  // longest-processing-time-first over the whole grid ("FlashAttention4 精读", section 3.3).
  const int bh = CAUSAL ? blockIdx.x : blockIdx.y;
  const int mblock = args.mblock0 + (CAUSAL ? (gridDim.y - 1 - blockIdx.y) : blockIdx.x);
  const int row0 = mblock * kCtaRows;
  const int nkv0_all = kv_blocks_for_tile<CAUSAL>(row0, n);
  const int nkv1_all = kv_blocks_for_tile<CAUSAL>(row0 + kTileRows, n);
  // Key split (blockIdx.z of gridDim.z): this CTA visits key blocks [jb, jb + nkv_h) of tile h;
  // a tile whose range is empty in this split only reports an empty partial result.
  const int nsplit = gridDim.z;
  const int nkv_all = nkv0_all > nkv1_all ? nkv0_all : nkv1_all;
  const int jb = static_cast<int>(static_cast<long long>(blockIdx.z) * nkv_all / nsplit);
  const int je = static_cast<int>(static_cast<long long>(blockIdx.z + 1) * nkv_all / nsplit);
  const int nkv0 = max(0, min(je, nkv0_all) - jb);
  const int nkv1 = max(0, min(je, nkv1_all) - jb);
  const int nkv_load = nkv0 > nkv1 ? nkv0 : nkv1;

  // ---------------------------------------------------------------- setup
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->q_full), 1);
    for (int s = 0; s < G::kSlots; ++s) {
      mbar_init(smem_u32(&ctl->kv_full[s]), 1);
      mbar_init(smem_u32(&ctl->kv_empty[s]), kSepP ? 2 : 1);   // head dim 64: one per tile
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&ctl->s_full[h]), 1);
      for (int q = 0; q < p_parts(); ++q)
        mbar_init(smem_u32(&ctl->p_full[h][q]), 4);  // one arrival per softmax warp
      mbar_init(smem_u32(&ctl->o_full[h]), 1);
      mbar_init(smem_u32(&ctl->s_read[h]), 4);   // one arrival per softmax warp
      mbar_init(smem_u32(&ctl->pv_done[h]), 1);
      mbar_init(smem_u32(&ctl->v16_full[h]), 2);  // one arrival per converter warp
      mbar_init(smem_u32(&ctl->v16_empty[h]), 1);
    }
    mbar_init(smem_u32(&ctl->drain), kSepP ? 2 : 1);   // head dim 64: one issuer per tile
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  int* abort_flag = &ctl->abort;

  // registers: the producer/MMA warpgroup gives most of its share to the softmax warpgroups
  // (384 threads x 168 at launch = 128 x (216 + 216 + 72))
  if (warp >= kCtlWarp0 && warp < kCtlWarp0 + 4) {
    regs_dec<kCtlRegs>();
  if (warp == kProducerWarp) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      const uint64_t keep = l2_policy_evict_last();   // K/V are re-read by other CTAs
      const uint64_t once = l2_policy_evict_first();  // Q is read once
      const uint32_t qbar = smem_u32(&ctl->q_full);
      const int ntiles = (nkv0 > 0) + (nkv1 > 0);
      if (ntiles > 0) {
        mbar_arrive_expect_tx(qbar, ntiles * G::kTileBytes);
        for (int h = 0; h < 2; ++h) {
          if ((h == 0 ? nkv0 : nkv1) == 0) continue;
          for (int b = 0; b < G::kBoxes; ++b)
            tma_load_3d_hint(smem_u32(s_q + h * G::kTileBytes + b * kTileRows * G::kSwBytes),
                             &map_q, qbar, b * G::kBoxElems, row0 + h * kTileRows, bh, once);
        }
      }
      // L2 warm-up of the first K/V blocks; the loop keeps it kL2PrefetchBlocks ahead
      for (int j = 0; j < kL2PrefetchBlocks && j < nkv_load; ++j)
        for (int b = 0; b < G::kBoxes; ++b) {
          tma_prefetch_l2_3d(&map_k, b * G::kBoxElems, (jb + j) * kTileRows, bh);
          tma_prefetch_l2_3d(&map_v, b * G::kBoxElems, (jb + j) * kTileRows, bh);
        }
      int issued = 0;
      bool ok = true;
      const int n_loads = EXATTN_INJECT_STALL ? 0 : 2 * nkv_load;
      for (int t = 0; t < n_loads && ok; ++t) {
        const int slot = t % G::kSlots;
        const int round = t / G::kSlots;
        if (round > 0) {
          ok = wait_phase(smem_u32(&ctl->kv_empty[slot]), (round - 1) & 1, abort_flag,
                          args.status);
          if (!ok) break;
        }
        const uint32_t fbar = smem_u32(&ctl->kv_full[slot]);
        EXATTN_TRACE_EVENT(9, t & 1, t >> 1);
        mbar_arrive_expect_tx(fbar, G::kTileBytes);
        const CUtensorMap* map = (t & 1) ? &map_v : &map_k;
        uint8_t* dst = s_ring + slot * G::kTileBytes;
        for (int b = 0; b < G::kBoxes; ++b)
          tma_load_3d_hint(smem_u32(dst + b * kTileRows * G::kSwBytes), map, fbar,
                           b * G::kBoxElems, (jb + (t >> 1)) * kTileRows, bh, keep);
        const int jp = (t >> 1) + kL2PrefetchBlocks;
        if (jp < nkv_load)
          for (int b = 0; b < G::kBoxes; ++b)
            tma_prefetch_l2_3d(map, b * G::kBoxElems, (jb + jp) * kTileRows, bh);
        ++issued;
      }
      if (!ok) {
        // abort: let the copies already issued land before the CTA's smem goes away
        if (ntiles > 0) wait_phase(smem_u32(&ctl->q_full), 0, abort_flag, args.status);
        const int first = issued > G::kSlots ? issued - G::kSlots : 0;
        for (int t = first; t < issued; ++t) {
          const uint32_t fbar = smem_u32(&ctl->kv_full[t % G::kSlots]);
          const uint32_t par = (t / G::kSlots) & 1;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(fbar, par) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == kMmaWarp || (kSepP && warp == kMmaWarp + 1)) {
    // ============================================================ MMA issuer(s)
    if (nkv_load > 0) {
      // The whole warp runs the issue loop, so the descriptor arithmetic is warp-uniform; one
      // lane, elected from the converged warp, issues each product and commit.  (With the loop
      // in lane 0 alone the same MMAs went out measurably slower: headline shape -7 %, causal
      // head-dim-64 shape -11 %.)
      auto issuer = []() -> bool { return elect_one(); };
      // a wait whose outcome every lane agrees on (an abort racing a phase completion could
      // otherwise split the warp), which also reconverges it
      auto mwait = [&](uint32_t bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, args.status));
      };
      bool ok = mwait(smem_u32(&ctl->q_full), 0);
      tc_fence_after();
      const uint32_t q_base = smem_u32(s_q);
      const uint32_t ring_base = smem_u32(s_ring);
      const int nkv[2] = {nkv0, nkv1};

      // The tensor core holds only a couple of MMAs in its queue, so any time this thread spends
      // between two products (waits, descriptor arithmetic, issue slots lost to the softmax
      // warps of its SMSP) leaves the pipe idle.  Each step therefore does its waits first, then
      // issues P V and the next S back to back with descriptors formed from per-tile bases.
      auto wait_kv = [&](int t) -> bool {
        return mwait(smem_u32(&ctl->kv_full[t % G::kSlots]), (t / G::kSlots) & 1);
      };
      const uint64_t q_desc = smem_desc(q_base, 16, 8 * G::kSwBytes, G::kSwMode);
      const uint64_t ring_desc = smem_desc(ring_base, 16, 8 * G::kSwBytes, G::kSwMode);
      // S_h = Q_h K_j^T into TMEM columns [128h, 128h + 128); K_j has landed
      auto issue_s = [&](int h, int j) {
        const int t = 2 * j;
        const uint64_t qd = q_desc + static_cast<uint64_t>(h * (G::kTileBytes >> 4));
        const uint64_t kd = ring_desc + static_cast<uint64_t>((t % G::kSlots) * (G::kTileBytes >> 4));
        if (issuer()) {
          mma_chain_ss_off<G::kKStepsS, FP8 ? 1 : 0, G::s_off(1), G::s_off(2), G::s_off(3),
                           G::s_off(4), G::s_off(5), G::s_off(6), G::s_off(7)>(
              tmem + h * 128, G::kIdescS, 0u, qd, kd);
          tc_commit(smem_u32(&ctl->s_full[h]));
        }
        __syncwarp();
        EXATTN_TRACE_EVENT(6, h, j);
      };
      // O_h += P_h V_j, P_h read from TMEM over S_h's columns.  The softmax may publish P in two
      // halves of 64 keys; the MMAs of the first half start while the second is computed.
      auto issue_pv_part = [&](int h, int j, int half, uint64_t vd) {
        constexpr int kN = G::kPvSteps / kPHalves;   // MMAs per published part of P
        // A: 8 TMEM columns of P per MMA; B: the next key group of V
        const uint32_t acc = (j > 0 || half > 0) ? 1u : 0u;
        const uint32_t a_tm = tmem + (kSepP ? 256 + h * 128 + 64 : h * 128) + half * kN * 8;
        const uint64_t b_desc = vd + static_cast<uint64_t>(half * kN * G::kPvStep);
        if (issuer())
          mma_chain_ts_off<kN, G::kPE4m3 ? 1 : 0, G::kPvStep, 8, 16, 24, 32, 40, 48, 56>(
              tmem + 256 + h * 128, G::kIdescPV, acc, a_tm, b_desc);
        __syncwarp();
      };
      // one step of tile h: P V of block j, then S of block j + 1 (which overwrites P_h).  It
      // needs V_j (or its f16 copy), K_{j+1} and (the first part of) P_h(j); the first two have
      // almost always landed and P_h(j) is often published already, so one probe checks all
      // three at once and the waits run one by one only when one of them is still open.
      auto step = [&](int h, int j) -> bool {
        const bool more = j + 1 < nkv[h];
        const int tv = 2 * j + 1, tk = 2 * j + 2;
        const uint32_t bar_v = G::kPv16 ? smem_u32(&ctl->v16_full[j & 1])
                                        : smem_u32(&ctl->kv_full[tv % G::kSlots]);
        const uint32_t par_v = G::kPv16 ? (j >> 1) & 1 : (tv / G::kSlots) & 1;
        const uint32_t bar_k = more ? smem_u32(&ctl->kv_full[tk % G::kSlots]) : bar_v;
        const uint32_t par_k = more ? (tk / G::kSlots) & 1 : par_v;
        const uint32_t bar_p = smem_u32(&ctl->p_full[h][0]);
        const uint32_t par_p = j & 1;
        if (!__all_sync(0xffffffffu, mbar_try_wait3(bar_v, par_v, bar_k, par_k, bar_p, par_p))) {
          if (!mwait(bar_v, par_v) || !mwait(bar_k, par_k) || !mwait(bar_p, par_p)) return false;
        }
        EXATTN_TRACE_EVENT(8, h, j);
        uint64_t vd;
        if constexpr (G::kPv16) {
          vd = smem_desc(smem_u32(s_v16) + (j & 1) * G::kV16TileBytes, kTileRows * G::kPvSwBytes,
                         8 * G::kPvSwBytes, kSwizzle128B);
          // both converter warps are done with the e4m3 copy: hand its slot back
          const bool first_user = (h == 0) || (j >= nkv[0]);
          if (first_user && lane == 0) mbar_arrive(smem_u32(&ctl->kv_empty[tv % G::kSlots]));
        } else {
          vd = smem_desc(ring_base + (tv % G::kSlots) * G::kTileBytes, kTileRows * G::kPvSwBytes,
                         8 * G::kPvSwBytes, G::kSwMode);
        }
        EXATTN_TRACE_EVENT(7, h, j + 1);
#pragma unroll
        for (int half = 0; half < kPHalves; ++half) {
          if (half > 0 && !mwait(smem_u32(&ctl->p_full[h][half]), j & 1)) return false;
          tc_fence_after();
          if (half == 0) EXATTN_TRACE_EVENT(4, h, j);
          issue_pv_part(h, j, half, vd);
        }
        EXATTN_TRACE_EVENT(5, h, j);
        if (j == nkv[h] - 1) {
          if (issuer()) tc_commit(smem_u32(&ctl->o_full[h]));
          __syncwarp();
        }
        if (more) issue_s(h, j + 1);
        return true;
      };

      ok = ok && wait_kv(0);
      if constexpr (!kSepP) {
        if (ok) {
          tc_fence_after();
          if (nkv0 > 0) issue_s(0, 0);
          if (nkv1 > 0) issue_s(1, 0);
        }
        for (int j = 0; j < nkv_load && ok; ++j) {
#pragma unroll
          for (int h = 0; h < 2 && ok; ++h)
            if (j < nkv[h]) ok = step(h, j);
        }
      } else {
        // Head dim 64: warp 9 issues tile 0's products and warp 10 tile 1's.  Per tile the events
        // come in a fixed order -- the softmax reads S_h(j), then publishes the two parts of
        // P_h(j) -- so each issuer waits for them one by one (blocking, bounded waits) and the
        // two tiles never wait for each other.  S_h(j+1) goes in as soon as the softmax has
        // read S_h(j); P V of block j as soon as its part of P_h(j) is published.  Ring slots
        // go back by tcgen05.commit from each tile that reads them (two arrivals per slot; a
        // tile alone on a block commits twice).
        const int h = warp - kMmaWarp;
        const int o = 1 - h;
        auto commit_to = [&](uint32_t bar, int times) {
          if (issuer())
            for (int i = 0; i < times; ++i) tc_commit(bar);
          __syncwarp();
        };
        if (ok && nkv[h] > 0) {
          tc_fence_after();
          issue_s(h, 0);
          commit_to(smem_u32(&ctl->kv_empty[0]), 0 < nkv[o] ? 1 : 2);
          for (int j = 0; j < nkv[h] && ok; ++j) {
            const int tv = 2 * j + 1, tk = 2 * j + 2;
            if (j + 1 < nkv[h]) {
              ok = mwait(smem_u32(&ctl->s_read[h]), j & 1) && wait_kv(tk);
              if (!ok) break;
              tc_fence_after();
              issue_s(h, j + 1);
              commit_to(smem_u32(&ctl->kv_empty[tk % G::kSlots]), j + 1 < nkv[o] ? 1 : 2);
            }
            const uint64_t vd = smem_desc(ring_base + (tv % G::kSlots) * G::kTileBytes,
                                          kTileRows * G::kPvSwBytes, 8 * G::kPvSwBytes,
                                          G::kSwMode);
#pragma unroll
            for (int part = 0; part < kPHalves; ++part) {
              ok = mwait(smem_u32(&ctl->p_full[h][part]), j & 1) && (part > 0 || wait_kv(tv));
              if (!ok) break;
              tc_fence_after();
              if (part == 0) EXATTN_TRACE_EVENT(4, h, j);
              issue_pv_part(h, j, part, vd);
            }
            if (!ok) break;
            EXATTN_TRACE_EVENT(5, h, j);
            commit_to(smem_u32(&ctl->pv_done[h]), 1);
            if (j == nkv[h] - 1) commit_to(smem_u32(&ctl->o_full[h]), 1);
            commit_to(smem_u32(&ctl->kv_empty[tv % G::kSlots]), j < nkv[o] ? 1 : 2);
          }
        }
      }
      // make sure nothing this thread issued is still running before TMEM is released
      __syncwarp();
      if (issuer()) tc_commit(smem_u32(&ctl->drain));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    if constexpr (G::kPv16) {
      // ========================================================== V converters (PV16)
      // Warps 10 and 11 widen each e4m3 V block to f16 (rows [0, 64) and [64, 128)) in one of
      // two buffers; the MMA thread frees the e4m3 ring slot once both halves are written.
      // Source: 128 rows of D bytes, swizzled over spans of kSwBytes (128 B for D = 128, 64 B
      // for D = 64).  Destination: boxes of 64 columns (128-byte rows, 128-byte swizzle).  Each
      // lane moves 16-element chunks: one 16-byte load, eight exact widenings, two 16-byte
      // stores.
      constexpr int kChunks = D / 16;            // 16-element chunks per row
      constexpr int kRowsPerPass = 32 / kChunks;
      const int row_begin = (warp - kConvWarp0) * (kTileRows / 2);
      const int c = lane % kChunks;
      const int box_off = (c / 4) * (kTileRows * 128);
      const int cc = 2 * (c % 4);
      bool ok = true;
      for (int j = 0; j < nkv_load && ok; ++j) {
        const int t = 2 * j + 1;
        const int slot = t % G::kSlots;
        ok = wait_phase(smem_u32(&ctl->kv_full[slot]), (t / G::kSlots) & 1, abort_flag,
                        args.status);
        if (ok && j >= 2)
          ok = wait_phase(smem_u32(&ctl->v16_empty[j & 1]), ((j >> 1) - 1) & 1, abort_flag,
                          args.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        fence_proxy_async_smem();
        const uint8_t* src = s_ring + slot * G::kTileBytes;
        uint8_t* dst = s_v16 + (j & 1) * G::kV16TileBytes + box_off;
#pragma unroll 2
        for (int r = row_begin + lane / kChunks; r < row_begin + kTileRows / 2;
             r += kRowsPerPass) {
          const int c_phys = D == 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
          const uint4 raw = *reinterpret_cast<const uint4*>(src + r * G::kRowBytes + c_phys * 16);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hx[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            hx[2 * i] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] & 0xFFFFu));
            hx[2 * i + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] >> 16));
          }
          // elements 16c .. 16c+15 = box c / 4, 16-byte chunks cc and cc + 1 of the row
          uint8_t* row = dst + r * 128;
          *reinterpret_cast<uint4*>(row + ((cc ^ (r & 7)) * 16)) =
              make_uint4(hx[0], hx[1], hx[2], hx[3]);
          *reinterpret_cast<uint4*>(row + (((cc + 1) ^ (r & 7)) * 16)) =
              make_uint4(hx[4], hx[5], hx[6], hx[7]);
        }
        // the MMAs read the f16 copy through the async proxy
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->v16_full[j & 1]));
      }
    }
  }
  } else {
    regs_inc<kSoftmaxRegs>();
    // ============================================================ softmax / epilogue
    const int h = (warp - kSoftmaxWarp0) / 4;
    const int w4 = warp % 4;
    const int nkv_h = h == 0 ? nkv0 : nkv1;
    const int nkv_h_all = h == 0 ? nkv0_all : nkv1_all;
    const int r_local = w4 * 32 + lane;        // TMEM lane == row within the tile
    const int row = row0 + h * kTileRows + r_local;
    const uint32_t lane_addr = static_cast<uint32_t>(w4 * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + h * 128;        // S_h
    const uint32_t t_o = tmem + lane_addr + 256 + h * 128;  // O_h
    const uint32_t t_p = kSepP ? t_o + 64 : t_s;             // P_h (over S_h for head dim 128)
    float c = args.c;
    float m_run = -INFINITY;  // running max of scaled logits, log2 units
    float l_run = 0.f;        // running sum of 2^(x - m_run) (times 2^p_offset_log2)
    float l_fix = 0.f;        // sum over blocks of (rounded - unrounded) largest probability
    bool ok = true;
    // fp8 block scaling ("FlashAttention · InkStack", section 3.3.1 "Block Quantization"): the
    // score block (i, j) is scaled by dq_i dk_j, folded into the exponent's multiplier; the value
    // block's dv_j is folded into P as the factor dv_j / dv_max <= 1 (a shift of the exponent),
    // l takes the inverse factor and the output multiplier is dv_max.  With power-of-two value
    // descales the fold is exact; otherwise the factor shares P's e4m3 rounding.
    // With fp8 P V, dv_max is kept in shared memory and the descales' index formed where it is
    // used, so that neither occupies a register through the key-block loop (C5's shape: +1 %;
    // the f16 P V instances measured 2 % slower that way and keep both in registers).
    const bool blockscaled = FP8 && args.dk_blk != nullptr;
    float* const dv_max_w = &ctl->dv_max[warp - kSoftmaxWarp0];
    float dv_max_r = 1.f;
    const size_t blk_base = static_cast<size_t>(bh) * args.nblk;
    if (blockscaled) {
      float mx = 0.f;
      for (int t = lane; t < args.nblk; t += 32) mx = fmaxf(mx, __ldg(args.dv_blk + blk_base + t));
#pragma unroll
      for (int off = 16; off >= 1; off /= 2) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane == 0) *dv_max_w = mx;
      __syncwarp();
      dv_max_r = mx;
      const int qblk = mblock * 2 + h;
      if (qblk < args.nblk) c *= __ldg(args.dq_blk + blk_base + qblk);
    }

    for (int j = 0; j < nkv_h; ++j) {
      float c_j = c;                             // multiplier of this key block's raw scores
      float bias_j = p_offset_log2<kPFmt>();     // added to every exponent of the block
      float l_mult = 1.f;                        // l gathers rowsum * l_mult
      if (blockscaled) {
        const size_t blk = (G::kPv16 ? blk_base : static_cast<size_t>(bh) * args.nblk) + jb + j;
        const float dk = __ldg(args.dk_blk + blk);
        const float dv = __ldg(args.dv_blk + blk);
        const float dv_max = G::kPv16 ? dv_max_r : *dv_max_w;
        c_j = c * dk;
        // log2(dv / dv_max) as exponent + log2(mantissa): exact when the ratio is a power of
        // two, so P then carries no rounding beyond its own e4m3 rounding
        const uint32_t rb = __float_as_uint(dv / dv_max);
        const float mant = __uint_as_float((rb & 0x007FFFFFu) | 0x3F800000u);
        bias_j += static_cast<float>(static_cast<int>((rb >> 23) & 0xFFu) - 127) +
                  (mant == 1.f ? 0.f : lg2_mufu(mant));
        l_mult = dv_max / dv;
      }
      ok = wait_phase(smem_u32(&ctl->s_full[h]), j & 1, abort_flag, args.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      if (threadIdx.x % 128 == 0) EXATTN_TRACE_EVENT(0, h, j);
      // Ring slots go back to the producer from here rather than by tcgen05.commit from the MMA
      // thread, whose commits would sit between two products.  Tile 1 (tile 0 when tile 1 has
      // no rows) visits every loaded block, and its MMAs are issued after tile 0's, so S_h(j)
      // complete means both tiles are done with K_j, and (S_h(j) following P V of block j - 1)
      // with V_{j-1} (or its f16 copy).
      // (head dim 64: the MMA warp hands the slots back itself)
      if (!kSepP && threadIdx.x % 128 == 0 && h == (nkv1 > 0 ? 1 : 0)) {
        mbar_arrive(smem_u32(&ctl->kv_empty[(2 * j) % G::kSlots]));
        if (j > 0)
          mbar_arrive(smem_u32(G::kPv16 ? &ctl->v16_empty[(j - 1) & 1]
                                        : &ctl->kv_empty[(2 * j - 1) % G::kSlots]));
      }

      // the row of S: four TMEM loads in flight, one wait
      float s[128];
      {
        uint32_t r[4][32];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) tmem_ld32(t_s + cb * 32, r[cb]);
        tmem_ld_wait();
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
          for (int i = 0; i < 32; ++i) s[cb * 32 + i] = __uint_as_float(r[cb][i]);
      }
      if constexpr (kSepP) {
        // S_h(j) is in registers: the MMA warp may compute S_h(j+1) over it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->s_read[h]));
      }
      // head dim 64: P V of block j - 1 must be complete before O_h is rescaled or P_h(j) is
      // written over P_h(j - 1)
      bool pv_prev_done = !kSepP || j == 0;
      auto wait_pv_prev = [&]() {
        if (pv_prev_done) return;
        ok = __all_sync(0xffffffffu, wait_phase(smem_u32(&ctl->pv_done[h]), (j - 1) & 1,
                                                abort_flag, args.status));
        tc_fence_after();
        pv_prev_done = true;
      };
      // masks: keys past the end of the sequence, and the causal diagonal block
      const int jg = jb + j;  // block index within the head
      const int key0 = jg * kTileRows;
      const bool diag = CAUSAL && jg == nkv_h_all - 1;
      const bool masked = (key0 + kTileRows > n) || diag;
      int lim = kTileRows;  // keys < lim are visible to this row
      if (masked) {
        const int lim_c = diag ? r_local + 1 : kTileRows;
        lim = min(n - key0, lim_c);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) s[i] = -INFINITY;
      }
      // row max: eight independent partial maxima folding two columns per instruction, then a
      // tree
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mp[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
      for (int i = 16; i < 128; i += 2) mp[(i / 2) % 8] = max3f(mp[(i / 2) % 8], s[i], s[i + 1]);
#pragma unroll
      for (int w = 4; w >= 1; w /= 2)
#pragma unroll
        for (int k = 0; k < w; ++k) mp[k] = fmaxf(mp[k], mp[k + w]);
      const float m_cand = fmaxf(m_run, mp[0] * c_j);
      if (threadIdx.x % 128 == 0) EXATTN_TRACE_EVENT(1, h, j);

      // Rescale O and l when some row of the warp grew its max by more than the lazy threshold
      // (the decision is warp-uniform because tcgen05.ld/st are warp-collective; rows whose max
      // did not move get alpha = 1).
      if (j == 0) {
        m_run = m_cand;
      } else if (__any_sync(0xffffffffu, m_cand - m_run > rescale_log2<kPFmt>())) {
        wait_pv_prev();
        const float alpha = ex2_mufu(m_run - m_cand);
        uint32_t r[32];
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          tmem_ld32(t_o + cb * 32, r);
          tmem_ld_wait();
          const float2 a2 = f32x2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 v = mul_f32x2(f32x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), a2);
            r[i] = __float_as_uint(f32x2_lo(v));
            r[i + 1] = __float_as_uint(f32x2_hi(v));
          }
          tmem_st32(t_o + cb * 32, r);
        }
        l_run *= alpha;
        l_fix *= alpha;
        m_run = m_cand;
      }
      if (threadIdx.x % 128 == 0) EXATTN_TRACE_EVENT(10, h, j);

      // probabilities p = 2^(s c - m), written over S (masked keys give exactly 0); the mask
      // test lives in its own instantiation so unmasked blocks run a select-free loop
      const uint32_t pb0 = smem_u32(&ctl->p_full[h][0]);
      const float m_shift = m_run - bias_j;
      // The P V product sums the probabilities as rounded to P's format, l_run sums them
      // unrounded.  Where a row's weight sits on one key, that key's rounding would reach O
      // undiluted, and under the lazy rescale the largest probability is no longer exactly
      // 2^0.  So O is divided by l_run plus, per block, the rounding of the block's largest
      // probability (the same fma and ex2 as in the loop below give the same value), which
      // makes O exact for a single dominant key; the LSE keeps l_run.  (Without the lazy
      // rescale the row's largest probability is exactly 2^offset and needs no correction.)
      if constexpr (rescale_log2<kPFmt>() > 0.f) {
        float p_top = ex2_mufu(fmaf(mp[0], c_j, -m_shift));
#if EXATTN_EX2_F16X2
        // unmasked e4m3 blocks take p through f16 (see exp_and_publish)
        if (kPFmt == PFmt::kE4m3 && !masked) {
          const float x = fmaf(mp[0], c_j, -(m_shift + 8.f));
          p_top = f16x2_to_f32x2(ex2_f16x2(pack_f16x2(x, x))).x * 256.f;
        }
#endif
        l_fix = fmaf(round_p<kPFmt>(p_top) - p_top, l_mult, l_fix);
      }
      const float rowsum =
          masked ? exp_and_publish<true, kPFmt, kPHalves, 0>(s, c_j, m_shift, lim, t_p, pb0, lane,
                                                             wait_pv_prev)
                 : exp_and_publish<false, kPFmt, kPHalves, EXATTN_EMU_EVERY>(
                       s, c_j, m_shift, lim, t_p, pb0, lane, wait_pv_prev);
      if (threadIdx.x % 128 == 0) EXATTN_TRACE_EVENT(3, h, j);
      l_run = fmaf(rowsum, l_mult, l_run);
    }

    if (ok && nkv_h > 0) {
      ok = wait_phase(smem_u32(&ctl->o_full[h]), 0, abort_flag, args.status);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const float inv_l =
            (blockscaled ? (G::kPv16 ? dv_max_r : *dv_max_w) : args.out_mult) / (l_run + l_fix);
        const bool live = row < n;
        const float lse_row = (m_run + lg2_mufu(l_run) - p_offset_log2<kPFmt>()) * kLn2;
        if (!FP8 && D == 128 && nsplit == 1) {
          // Bulk-store epilogue (bf16 operands, head dim 128, one key split): the warp's 32 rows
          // of O, scaled and rounded to bf16, go into its tile's Q buffer -- free, since every S
          // of the tile has completed -- laid out as the 128-byte-swizzled boxes of 64 columns
          // the O tensor map describes, and one lane stores them.  With a 16-byte store per lane
          // and row from registers (each warp instruction touching 32 rows) the epilogue took
          // 2300-2900 cycles on B4 H16 N2048 causal, this way 1900-2150: that shape +2 %, the
          // headline +1 %.  At head dim 64 the same epilogue measured 8 % slower on B1 H16
          // N32768 causal and the register stores stay; fp8 operands leave a Q tile too small
          // for bf16 O.
          uint32_t r[D / 32][32];
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) tmem_ld32(t_o + cb * 32, r[cb]);
          tmem_ld_wait();
          const uint32_t stage = smem_u32(s_q + h * G::kTileBytes);
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t pk[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                pk[i] = pack_bf16x2(__uint_as_float(r[cb][8 * q4 + 2 * i]) * inv_l,
                                    __uint_as_float(r[cb][8 * q4 + 2 * i + 1]) * inv_l);
              const int g = cb * 4 + q4;          // 16-byte chunk of the row (8 columns)
              const int box = g / 8, c = g % 8;   // box of 64 columns, chunk within its row
              st_shared_v4(stage + box * (kTileRows * 128) + r_local * 128 + ((c ^ (r_local & 7)) * 16),
                           pk[0], pk[1], pk[2], pk[3]);
            }
          fence_proxy_async_smem();
          __syncwarp();
          const int wrow = row0 + h * kTileRows + w4 * 32;   // the warp's first row
          if (lane == 0 && wrow < n) {
#pragma unroll
            for (int box = 0; box < D / 64; ++box)
              tma_store_3d(&map_o, stage + box * (kTileRows * 128) + w4 * 32 * 128, box * 64, wrow,
                           bh);
            bulk_commit_group();
            bulk_wait_group_read0();   // the CTA's shared memory must outlive the reads
          }
          __syncwarp();
          if (live) args.lse[static_cast<size_t>(bh) * n + row] = lse_row;
        } else if (nsplit == 1) {
          __nv_bfloat16* orow = args.o + (static_cast<size_t>(bh) * n + (live ? row : 0)) * D;
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t r[32];
            tmem_ld32(t_o + cb * 32, r);
            tmem_ld_wait();
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l,
                                      __uint_as_float(r[2 * i + 1]) * inv_l);
            if (live) {
              uint4* dst = reinterpret_cast<uint4*>(orow + cb * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                    packed[4 * i + 3]);
            }
          }
          if (live) args.lse[static_cast<size_t>(bh) * n + row] = lse_row;
        } else {
          // this split's normalised output and log-sum-exp, merged later by the combine kernel
          const size_t prow = (static_cast<size_t>(blockIdx.z) * args.bh + bh) * n + (live ? row : 0);
          float* orow = args.o_part + prow * D;
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t r[32];
            tmem_ld32(t_o + cb * 32, r);
            tmem_ld_wait();
            if (live) {
              float4* dst = reinterpret_cast<float4*>(orow + cb * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv_l,
                                     __uint_as_float(r[4 * i + 1]) * inv_l,
                                     __uint_as_float(r[4 * i + 2]) * inv_l,
                                     __uint_as_float(r[4 * i + 3]) * inv_l);
            }
          }
          if (live) args.lse_part[prow] = lse_row;
        }
      }
    } else if (ok && nsplit > 1 && row < n) {
      // empty key range in this split: contributes nothing to the merge
      const size_t prow = (static_cast<size_t>(blockIdx.z) * args.bh + bh) * n + row;
      float4* dst = reinterpret_cast<float4*>(args.o_part + prow * D);
#pragma unroll
      for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      args.lse_part[prow] = -INFINITY;
    }
    tc_fence_before();
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


}  // namespace exattn
