// fa_bwd_kernel.cuh -- attention backward for sm_103a (tcgen05 + TMEM + TMA), bf16 operands.
//
// Gradients of exact attention ("FlashAttention · InkStack", section 1.2 "反向传播"): with P
// recomputed from the forward pass's log-sum-exp (P_ij = exp(scale q_i.k_j - LSE_i), the
// recomputation of section 1.2.2) and D_i = rowsum(dO_i * O_i):
//
//   dV_j = sum_i P_ij^T dO_i          dP_ij = dO_i V_j^T          dS_ij = P_ij * (dP_ij - D_i)
//   dK_j = scale sum_i dS_ij^T Q_i    dQ_i  = scale sum_j dS_ij K_j
//
// Three launches:
//   bwd_delta_kernel   D_i = dO_i . O_i (fp32), one warp per row;
//   bwd_dkdv_kernel    one CTA per (head, 128-key block j): K_j and V_j stay in shared memory,
//                      the query blocks i stream through a two-stage ring; per i the tensor core
//                      computes S^T = K_j Q_i^T and dP^T = V_j dO_i^T into TMEM, the softmax warps
//                      turn them into P^T and dS^T (bf16, written back over S^T and dP^T), and the
//                      tensor core accumulates dV_j += P^T dO_i and dK_j += dS^T Q_i in TMEM;
//   bwd_dq_kernel      one CTA per (head, 128-query block i): Q_i and dO_i stay, the key blocks
//                      stream; per j S = Q_i K_j^T and dP = dO_i V_j^T, the softmax warps form dS,
//                      and dQ_i += dS K_j accumulates in TMEM.
// Splitting dQ from dK/dV recomputes S and dP once more (7 products instead of 5) but needs no
// atomics and no fp32 dQ accumulator in global memory.
//
// The MMAs are the forward kernel's: S-type products have both operands K-major in shared memory
// (128-byte swizzled TMA tiles), the accumulating products take their A operand (P^T, dS^T or dS,
// bf16) from TMEM and their B operand MN-major from the same tiles.  Warp roles (384 threads):
// warps 0-7 one half-row of S each (warp w: TMEM lanes 32 (w % 4) .., columns 64 (w / 4) ..),
// warp 8 TMA, warp 9 MMA issue and TMEM owner, warp 10 (dK/dV only) stages LSE and D of each query
// block in shared memory.  Every wait is bounded as in the forward kernel (and a test build with
// EXATTN_INJECT_STALL stops each producer after the CTA's fixed tiles, so the first streamed wait
// runs out and every role leaves through the abort path).
#pragma once

#include "fa_fwd_kernel.cuh"

namespace exattn {

constexpr int kBwdThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdGeo {
  static constexpr int kBoxes = D / 64;                     // 64-column (128-byte) TMA boxes
  static constexpr int kTileBytes = kTileRows * D * 2;      // one 128-row bf16 tile
  static constexpr int kKSteps = D / 16;                    // MMAs per S-type product
  static constexpr uint32_t kIdescS = instr_desc(128, 128, 1, false, false);
  static constexpr uint32_t kIdescAcc = instr_desc(128, D, 1, false, true);
  static constexpr int kHalfCols = D / 2;                   // output columns per thread
};

struct BwdArgs {
  __nv_bfloat16* g0;      // dkdv: dK out; dq: dQ out            [BH, N, d]
  __nv_bfloat16* g1;      // dkdv: dV out                         [BH, N, d]
  const float* lse;       // forward log-sum-exp (natural log)    [BH, N]
  const float* delta;     // D                                    [BH, N]
  int* status;
  int n;
  float c;                // scale * log2(e)
  float scale;
};

struct BwdCtrl {
  uint64_t fix_full;      // the CTA's fixed pair of tiles (dK/dV: K_j, V_j; dQ: Q_i, dO_i)
  uint64_t ring_full[2];  // streamed pair (dK/dV: Q_i, dO_i; dQ: K_j, V_j)
  uint64_t ring_empty[2];
  uint64_t vec_full[2];   // LSE and D of the query block (dK/dV)
  uint64_t s_full;        // S (dK/dV: S^T) of the step is in TMEM
  uint64_t dp_full;       // dP (dP^T) of the step is in TMEM
  uint64_t p_full;        // dK/dV: P^T written back in bf16; dQ: S read (eight warps)
  uint64_t ds_full;       // dS (dS^T) written back in bf16 (eight warps)
  uint64_t o_full;        // the last accumulating product is done
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  alignas(16) float lse2[2][kTileRows];   // LSE * log2(e) of the stage's 128 queries
  alignas(16) float dlt[2][kTileRows];    // D of the stage's 128 queries
};

// two fixed tiles + two ring stages of two tiles + the control block
template <int D>
constexpr int bwd_smem_bytes() {
  return 6 * BwdGeo<D>::kTileBytes + static_cast<int>(sizeof(BwdCtrl)) + 1024;
}

// The dQ kernel streams K_j and V_j as separate tiles through a five-slot ring: V_j is released
// once dP has read it and K_j once dQ has, so each load starts two to three products before it
// is needed (a stage of both tiles, released after dQ, left one product for a 64 KB load).
constexpr int kDqSlots = 5;

struct DqCtrl {
  uint64_t fix_full;                 // Q_i and dO_i
  uint64_t tile_full[kDqSlots];      // tile t (K_j for t = 2j, V_j for t = 2j + 1) in slot t % 5
  uint64_t tile_empty[kDqSlots];
  uint64_t s_full;                   // S of the step is in TMEM
  uint64_t dp_full;                  // dP of the step is in TMEM
  uint64_t p_full;                   // the softmax has read S (eight warps)
  uint64_t ds_full;                  // dS written back in bf16 (eight warps)
  uint64_t o_full;                   // the last dQ product is done
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// two fixed tiles + the five-slot ring + the control block
template <int D>
constexpr int dq_smem_bytes() {
  return (2 + kDqSlots) * BwdGeo<D>::kTileBytes + static_cast<int>(sizeof(DqCtrl)) + 1024;
}

// D_i = sum_t dO_it O_it in fp32, one warp per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta, long long rows) {
  constexpr int kPer = D / 32;
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x % 32;
  const __nv_bfloat16* a = o + row * D + lane * kPer;
  const __nv_bfloat16* b = dout + row * D + lane * kPer;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; i += 2) {
    const uint32_t wa = *reinterpret_cast<const uint32_t*>(a + i);
    const uint32_t wb = *reinterpret_cast<const uint32_t*>(b + i);
    acc = fmaf(__uint_as_float(wa << 16), __uint_as_float(wb << 16), acc);
    acc = fmaf(__uint_as_float(wa & 0xFFFF0000u), __uint_as_float(wb & 0xFFFF0000u), acc);
  }
#pragma unroll
  for (int off = 16; off >= 1; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

// A operand of an accumulating product: the softmax warps of column half 0 write their 64 bf16
// values to TMEM columns [0, 32), those of half 1 to [64, 96), each inside the S columns it read
// itself (so no warp overwrites S another warp has not read yet); k-step kb (16 keys) reads 8
// columns at kb < 4 ? 8 kb : 64 + 8 (kb - 4).

// S-type product into TMEM columns [col, col + 128): A and B both 128 x D K-major tiles.  The
// K steps of 32 bytes advance 2 descriptor units inside a 128-byte swizzle span and 1024 units
// (one 128-row box) past it.
template <int D>
__device__ __forceinline__ void mma_s_type(uint32_t tmem_d, uint32_t a_tile, uint32_t b_tile) {
  using G = BwdGeo<D>;
  mma_chain_ss_off<G::kKSteps, 0, 2, 4, 6, 1024, 1026, 1028, 1030>(
      tmem_d, G::kIdescS, 0u, smem_desc(a_tile, 16, 1024, kSwizzle128B),
      smem_desc(b_tile, 16, 1024, kSwizzle128B));
}

// Accumulating product D += A (128 x 128 bf16 from TMEM, columns as above) * B (128 x D tile,
// MN-major, 16 keys = 128 descriptor units per step).
template <int D>
__device__ __forceinline__ void mma_acc(uint32_t tmem_d, uint32_t tmem_a, uint32_t b_tile,
                                        bool accumulate) {
  using G = BwdGeo<D>;
  mma_chain_ts_off<8, 0, 128, 8, 16, 24, 64, 72, 80, 88>(
      tmem_d, G::kIdescAcc, accumulate ? 1u : 0u, tmem_a,
      smem_desc(b_tile, kTileRows * 128, 1024, kSwizzle128B));
}

// Half-row softmax steps shared by both kernels, for the 64 columns of this thread's row.
// softmax_p: P = 2^(s c - LSE log2 e) from the S columns into p[] (fp32), and, when STORE, as
// bf16 over the S columns (dK/dV kernel: the A operand of dV += P^T dO).  softmax_ds:
// dS = P (dP - D) from the dP columns, as bf16 over them.  Both run in two passes of 32 columns;
// the bf16 results of pass 0 land in columns 0-15 and of pass 1 in columns 16-31 of the thread's
// range, whose fp32 values were read in pass 0.  PER_COLUMN (dK/dV kernel): column q has its own
// LSE * log2(e) and D, read as float4 from the shared arrays; otherwise (dQ kernel) the row's
// own values apply to every column.  MASKED (a separate instantiation, so the unmasked blocks
// carry no per-column select): `visible` decides which columns keep their probability.
template <bool PER_COLUMN, bool STORE, bool MASKED, typename VisFn>
__device__ __forceinline__ void softmax_p(uint32_t t_s, float c, const float* l2, float l2_row,
                                          VisFn visible, float (&p)[64]) {
  // pass 1's TMEM load is issued before pass 0's arithmetic, so its latency overlaps it
  uint32_t rs[2][32];
  tmem_ld32(t_s, rs[0]);
  tmem_ld_wait();
  tmem_ld32(t_s + 32, rs[1]);
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    float lv[32];
    if constexpr (PER_COLUMN) {
      const float4* l4 = reinterpret_cast<const float4*>(l2 + 32 * pass);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 a = l4[i];
        lv[4 * i] = a.x;
        lv[4 * i + 1] = a.y;
        lv[4 * i + 2] = a.z;
        lv[4 * i + 3] = a.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) lv[i] = l2_row;
    }
    if (pass == 1) tmem_ld_wait();
    const float2 c2 = f32x2(c, c);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      // s c - LSE log2(e) for two columns in one packed fma
      const float2 x2 = fma_f32x2(f32x2(__uint_as_float(rs[pass][i]), __uint_as_float(rs[pass][i + 1])),
                                    c2, f32x2(-lv[i], -lv[i + 1]));
      float x0 = ex2_mufu(f32x2_lo(x2)), x1 = ex2_mufu(f32x2_hi(x2));
      if constexpr (MASKED) {
        x0 = visible(32 * pass + i) ? x0 : 0.f;
        x1 = visible(32 * pass + i + 1) ? x1 : 0.f;
      }
      p[32 * pass + i] = x0;
      p[32 * pass + i + 1] = x1;
    }
    if constexpr (STORE) {
      uint32_t pp[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) pp[i] = pack_bf16x2(p[32 * pass + 2 * i], p[32 * pass + 2 * i + 1]);
      tmem_st16(t_s + 16 * pass, pp);
    }
  }
  if constexpr (STORE) tmem_st_wait();
}

template <bool PER_COLUMN>
__device__ __forceinline__ void softmax_ds(uint32_t t_dp, const float* dl, float dl_row,
                                           const float (&p)[64]) {
  uint32_t rd[2][32];
  tmem_ld32(t_dp, rd[0]);
  tmem_ld_wait();
  tmem_ld32(t_dp + 32, rd[1]);
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    float dv[32];
    if constexpr (PER_COLUMN) {
      const float4* d4 = reinterpret_cast<const float4*>(dl + 32 * pass);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 b = d4[i];
        dv[4 * i] = b.x;
        dv[4 * i + 1] = b.y;
        dv[4 * i + 2] = b.z;
        dv[4 * i + 3] = b.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) dv[i] = dl_row;
    }
    if (pass == 1) tmem_ld_wait();
    uint32_t pd[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int q = 32 * pass + 2 * i;
      // dS = P (dP - D), two columns per packed add and multiply
      const float2 t2 = add_f32x2(f32x2(__uint_as_float(rd[pass][2 * i]), __uint_as_float(rd[pass][2 * i + 1])),
                                    f32x2(-dv[2 * i], -dv[2 * i + 1]));
      const float2 d2 = mul_f32x2(f32x2(p[q], p[q + 1]), t2);
      pd[i] = pack_bf16x2(f32x2_lo(d2), f32x2_hi(d2));
    }
    tmem_st16(t_dp + 16 * pass, pd);
  }
  tmem_st_wait();
}

// ------------------------------------------------------------------------------------------
// dK, dV: one CTA per (head, key block).  Grid (key blocks, BH); causal: (BH, key blocks) with
// the key blocks in increasing order, i.e. the CTAs with the most query blocks first.
// ------------------------------------------------------------------------------------------
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_g0, const __grid_constant__ CUtensorMap map_g1,
                    const BwdArgs args) {
  using G = BwdGeo<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* s_k = smem;
  uint8_t* s_v = smem + G::kTileBytes;
  uint8_t* s_ring = smem + 2 * G::kTileBytes;  // stage s: Q at 2s, dO at 2s + 1 (tiles)
  BwdCtrl* ctl = reinterpret_cast<BwdCtrl*>(smem + 6 * G::kTileBytes);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int n = args.n;
  const int bh = CAUSAL ? blockIdx.x : blockIdx.y;
  const int jblk = CAUSAL ? blockIdx.y : blockIdx.x;
  const int nblk = (n + kTileRows - 1) / kTileRows;
  const int i0 = CAUSAL ? jblk : 0;   // first query block that sees this key block
  const int nq = nblk - i0;           // query blocks visited (>= 1)
  int* const status = args.status;

  if (warp == 9) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->fix_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ctl->ring_full[s]), 1);
      mbar_init(smem_u32(&ctl->ring_empty[s]), 1);
      mbar_init(smem_u32(&ctl->vec_full[s]), 1);
    }
    mbar_init(smem_u32(&ctl->s_full), 1);
    mbar_init(smem_u32(&ctl->dp_full), 1);
    mbar_init(smem_u32(&ctl->p_full), 8);
    mbar_init(smem_u32(&ctl->ds_full), 8);
    mbar_init(smem_u32(&ctl->o_full), 1);
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  int* abort_flag = &ctl->abort;

  if (warp >= 8) {
    regs_dec<72>();
    if (warp == 8) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_map(&map_q);
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
        tma_prefetch_map(&map_do);
        const uint32_t fb = smem_u32(&ctl->fix_full);
        mbar_arrive_expect_tx(fb, 2 * G::kTileBytes);
        for (int b = 0; b < G::kBoxes; ++b) {
          tma_load_3d(smem_u32(s_k + b * kTileRows * 128), &map_k, fb, b * 64, jblk * kTileRows, bh);
          tma_load_3d(smem_u32(s_v + b * kTileRows * 128), &map_v, fb, b * 64, jblk * kTileRows, bh);
        }
        bool ok = true;
        int issued = 0;
        const int n_stream = EXATTN_INJECT_STALL ? 0 : nq;   // test builds: stop after K_j, V_j
        for (int u = 0; u < n_stream && ok; ++u) {
          const int s = u & 1;
          if (u >= 2) {
            ok = wait_phase(smem_u32(&ctl->ring_empty[s]), ((u >> 1) - 1) & 1, abort_flag, status);
            if (!ok) break;
          }
          const uint32_t rb = smem_u32(&ctl->ring_full[s]);
          mbar_arrive_expect_tx(rb, 2 * G::kTileBytes);
          uint8_t* dq = s_ring + (2 * s) * G::kTileBytes;
          uint8_t* ddo = s_ring + (2 * s + 1) * G::kTileBytes;
          const int row = (i0 + u) * kTileRows;
          for (int b = 0; b < G::kBoxes; ++b) {
            tma_load_3d(smem_u32(dq + b * kTileRows * 128), &map_q, rb, b * 64, row, bh);
            tma_load_3d(smem_u32(ddo + b * kTileRows * 128), &map_do, rb, b * 64, row, bh);
          }
          ++issued;
        }
        if (!ok) {
          // abort: let the copies already issued land before the CTA's smem goes away
          wait_phase(fb, 0, abort_flag, status);
          for (int u = issued > 2 ? issued - 2 : 0; u < issued; ++u) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&ctl->ring_full[u & 1]), (u >> 1) & 1) &&
                   globaltimer_ns() - t0 < kWaitLimitNs) {
            }
          }
        }
      }
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the issue loop (warp-uniform descriptor arithmetic); one elected
      // lane issues each product and commit.  Wait outcomes are made warp-uniform.
      {
        auto mwait = [&](uint32_t bar, uint32_t parity) -> bool {
          return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, status));
        };
        bool ok = mwait(smem_u32(&ctl->fix_full), 0);
        tc_fence_after();
        const uint32_t k_tile = smem_u32(s_k), v_tile = smem_u32(s_v);
        // Issue order per step u: dV(u), S(u+1), dK(u), dP(u+1).  S(u+1) overwrites P^T(u)
        // only after dV(u) has read it (the tensor core runs one thread's MMAs in order), and
        // dP(u+1) overwrites dS^T(u) after dK(u); so the softmax forms P^T(u+1) while dK(u)
        // and dP(u+1) run, and dS^T(u+1) while dV(u+1) and S(u+2) run.
        auto tile = [&](int u, int which) {
          return smem_u32(s_ring + (2 * (u & 1) + which) * G::kTileBytes);
        };
        ok = ok && mwait(smem_u32(&ctl->ring_full[0]), 0);
        if (ok) {
          tc_fence_after();
          if (elect_one()) {
            mma_s_type<D>(tmem, k_tile, tile(0, 0));          // S^T  = K_j Q_i^T
            tc_commit(smem_u32(&ctl->s_full));
            mma_s_type<D>(tmem + 128, v_tile, tile(0, 1));    // dP^T = V_j dO_i^T
            tc_commit(smem_u32(&ctl->dp_full));
          }
          __syncwarp();
        }
        for (int u = 0; u < nq && ok; ++u) {
          const bool more = u + 1 < nq;
          ok = mwait(smem_u32(&ctl->p_full), u & 1);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) mma_acc<D>(tmem + 256, tmem, tile(u, 1), u > 0);   // dV += P^T dO_i
          __syncwarp();
          if (more) {
            ok = mwait(smem_u32(&ctl->ring_full[(u + 1) & 1]), ((u + 1) >> 1) & 1);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
              mma_s_type<D>(tmem, k_tile, tile(u + 1, 0));
              tc_commit(smem_u32(&ctl->s_full));
            }
            __syncwarp();
          }
          ok = mwait(smem_u32(&ctl->ds_full), u & 1);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
            mma_acc<D>(tmem + 384, tmem + 128, tile(u, 0), u > 0);   // dK += dS^T Q_i
            tc_commit(smem_u32(&ctl->ring_empty[u & 1]));
            if (more) {
              mma_s_type<D>(tmem + 128, v_tile, tile(u + 1, 1));
              tc_commit(smem_u32(&ctl->dp_full));
            }
          }
          __syncwarp();
        }
        if (elect_one()) {
          if (ok) tc_commit(smem_u32(&ctl->o_full));
          tc_commit(smem_u32(&ctl->drain));
        }
        __syncwarp();
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    } else if (warp == 10) {
      // ------------------------------------------------------------ LSE / D stager
      // The values of query block u + 1 are loaded into registers while block u's stage is
      // being waited for and written, so the global-load latency is off the softmax's path.
      constexpr int kPer = kTileRows / 32;
      float lv[kPer], dv[kPer];
      const float* lse_h = args.lse + static_cast<size_t>(bh) * n;
      const float* dlt_h = args.delta + static_cast<size_t>(bh) * n;
      auto fetch = [&](int u) {
        const int row0 = (i0 + u) * kTileRows + lane;
#pragma unroll
        for (int t = 0; t < kPer; ++t) {
          const int row = row0 + 32 * t;
          lv[t] = row < n ? __ldg(lse_h + row) : 0.f;
          dv[t] = row < n ? __ldg(dlt_h + row) : 0.f;
        }
      };
      fetch(0);
      bool ok = true;
      for (int u = 0; u < nq && ok; ++u) {
        const int s = u & 1;
        if (u >= 2)
          ok = wait_phase(smem_u32(&ctl->ring_empty[s]), ((u >> 1) - 1) & 1, abort_flag, status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
#pragma unroll
        for (int t = 0; t < kPer; ++t) {
          ctl->lse2[s][lane + 32 * t] = lv[t] * kLog2e;
          ctl->dlt[s][lane + 32 * t] = dv[t];
        }
        if (u + 1 < nq) fetch(u + 1);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->vec_full[s]));
      }
    }
  } else {
    regs_inc<216>();
    // ------------------------------------------------------------ softmax warps
    const int w4 = warp % 4, hc = warp / 4;
    const int r = w4 * 32 + lane;                  // key row within the block (TMEM lane)
    const int key = jblk * kTileRows + r;
    const uint32_t lane_addr = static_cast<uint32_t>(w4 * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + 64 * hc;
    const uint32_t t_dp = tmem + lane_addr + 128 + 64 * hc;
    bool ok = true;
    for (int u = 0; u < nq && ok; ++u) {
      const int s = u & 1;
      const int qblk = i0 + u;
      ok = wait_phase(smem_u32(&ctl->vec_full[s]), (u >> 1) & 1, abort_flag, status);
      if (ok) ok = wait_phase(smem_u32(&ctl->s_full), u & 1, abort_flag, status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* l2 = ctl->lse2[s] + 64 * hc;
      const float* dl = ctl->dlt[s] + 64 * hc;
      const int q0 = qblk * kTileRows + 64 * hc;   // first query column of this half
      const bool any_masked = (CAUSAL && qblk == jblk) || (qblk + 1) * kTileRows > n;
      float p[64];
      const auto vis = [&](int q) { return q0 + q < n && (!CAUSAL || key <= q0 + q); };
      if (any_masked)
        softmax_p<true, true, true>(t_s, args.c, l2, 0.f, vis, p);
      else
        softmax_p<true, true, false>(t_s, args.c, l2, 0.f, vis, p);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full));
      ok = wait_phase(smem_u32(&ctl->dp_full), u & 1, abort_flag, status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      softmax_ds<true>(t_dp, dl, 0.f, p);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->ds_full));
    }
    if (ok) {
      ok = wait_phase(smem_u32(&ctl->o_full), 0, abort_flag, status);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok && D == 128) {
      // Bulk-store epilogue (head dim 128): the warp's 32 key rows x 64 columns of dV and dK,
      // rounded to bf16, go into the V and K tiles (free: every product has completed) in the
      // 128-byte-swizzled layout of the output tensor maps' boxes, and one lane stores them
      // (rows past N are clipped by the maps).
      tc_fence_after();
#pragma unroll
      for (int which = 0; which < 2; ++which) {   // 0: dV (cols 256..), 1: dK (cols 384..)
        const uint32_t t_acc = tmem + lane_addr + (which ? 384 : 256) + G::kHalfCols * hc;
        const float mult = which ? args.scale : 1.f;
        uint32_t rr[2][32];
        tmem_ld32(t_acc, rr[0]);
        tmem_ld32(t_acc + 32, rr[1]);
        tmem_ld_wait();
        const uint32_t box = smem_u32(which ? s_k : s_v) + hc * (kTileRows * 128);
#pragma unroll
        for (int g = 0; g < 8; ++g) {   // 16-byte chunk (8 columns) of the row's 64
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(rr[g / 4][8 * (g % 4) + 2 * i]) * mult,
                                __uint_as_float(rr[g / 4][8 * (g % 4) + 2 * i + 1]) * mult);
          st_shared_v4(box + r * 128 + ((g ^ (r & 7)) * 16), pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int wrow = jblk * kTileRows + w4 * 32;   // the warp's first key row
      if (lane == 0 && wrow < n) {
        const uint32_t slab = hc * (kTileRows * 128) + w4 * 32 * 128;
        tma_store_3d(&map_g1, smem_u32(s_v) + slab, 64 * hc, wrow, bh);
        tma_store_3d(&map_g0, smem_u32(s_k) + slab, 64 * hc, wrow, bh);
        bulk_commit_group();
        bulk_wait_group_read0();   // the CTA's shared memory must outlive the reads
      }
      __syncwarp();
    } else if (ok) {
      tc_fence_after();
      const bool live = key < n;
      const size_t row_off = (static_cast<size_t>(bh) * n + (live ? key : 0)) * D + G::kHalfCols * hc;
#pragma unroll
      for (int which = 0; which < 2; ++which) {   // 0: dV (cols 256..), 1: dK (cols 384..)
        const uint32_t t_acc = tmem + lane_addr + (which ? 384 : 256) + G::kHalfCols * hc;
        const float mult = which ? args.scale : 1.f;
        __nv_bfloat16* dst = (which ? args.g0 : args.g1) + row_off;
#pragma unroll
        for (int cb = 0; cb < G::kHalfCols / 32; ++cb) {
          uint32_t rr[32];
          tmem_ld32(t_acc + cb * 32, rr);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * mult,
                                __uint_as_float(rr[2 * i + 1]) * mult);
          if (live) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cb * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// dQ: one CTA per (head, query block).  Grid (query blocks, BH); causal: (BH, query blocks) with
// the query blocks in decreasing order (the heaviest first).
// ------------------------------------------------------------------------------------------
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                  const __grid_constant__ CUtensorMap map_g0, const BwdArgs args) {
  using G = BwdGeo<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* s_q = smem;
  uint8_t* s_do = smem + G::kTileBytes;
  uint8_t* s_ring = smem + 2 * G::kTileBytes;  // slot i at tile i
  DqCtrl* ctl = reinterpret_cast<DqCtrl*>(smem + (2 + kDqSlots) * G::kTileBytes);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int n = args.n;
  const int nblk = (n + kTileRows - 1) / kTileRows;
  const int bh = CAUSAL ? blockIdx.x : blockIdx.y;
  const int iblk = CAUSAL ? (nblk - 1 - static_cast<int>(blockIdx.y)) : blockIdx.x;
  const int nk = CAUSAL ? iblk + 1 : nblk;   // key blocks visited
  int* const status = args.status;

  if (warp == 9) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->fix_full), 1);
    for (int i = 0; i < kDqSlots; ++i) {
      mbar_init(smem_u32(&ctl->tile_full[i]), 1);
      mbar_init(smem_u32(&ctl->tile_empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl->s_full), 1);
    mbar_init(smem_u32(&ctl->dp_full), 1);
    mbar_init(smem_u32(&ctl->p_full), 8);
    mbar_init(smem_u32(&ctl->ds_full), 8);
    mbar_init(smem_u32(&ctl->o_full), 1);
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  int* abort_flag = &ctl->abort;
  const int ntiles = 2 * nk;

  if (warp >= 8) {
    regs_dec<72>();
    if (warp == 8) {
      if (lane == 0) {
        tma_prefetch_map(&map_q);
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
        tma_prefetch_map(&map_do);
        const uint32_t fb = smem_u32(&ctl->fix_full);
        mbar_arrive_expect_tx(fb, 2 * G::kTileBytes);
        for (int b = 0; b < G::kBoxes; ++b) {
          tma_load_3d(smem_u32(s_q + b * kTileRows * 128), &map_q, fb, b * 64, iblk * kTileRows, bh);
          tma_load_3d(smem_u32(s_do + b * kTileRows * 128), &map_do, fb, b * 64, iblk * kTileRows, bh);
        }
        bool ok = true;
        int issued = 0;
        const int n_load = EXATTN_INJECT_STALL ? 0 : ntiles;   // test builds: stop after Q_i, dO_i
        for (int t = 0; t < n_load && ok; ++t) {
          const int slot = t % kDqSlots;
          if (t >= kDqSlots) {
            ok = wait_phase(smem_u32(&ctl->tile_empty[slot]), (t / kDqSlots - 1) & 1, abort_flag,
                            status);
            if (!ok) break;
          }
          const uint32_t tb = smem_u32(&ctl->tile_full[slot]);
          mbar_arrive_expect_tx(tb, G::kTileBytes);
          uint8_t* dst = s_ring + slot * G::kTileBytes;
          const CUtensorMap* map = (t & 1) ? &map_v : &map_k;
          for (int b = 0; b < G::kBoxes; ++b)
            tma_load_3d(smem_u32(dst + b * kTileRows * 128), map, tb, b * 64, (t >> 1) * kTileRows,
                        bh);
          ++issued;
        }
        if (!ok) {
          // abort: let the copies still in flight land before the CTA's smem goes away
          wait_phase(fb, 0, abort_flag, status);
          for (int t = issued > kDqSlots ? issued - kDqSlots : 0; t < issued; ++t) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&ctl->tile_full[t % kDqSlots]), (t / kDqSlots) & 1) &&
                   globaltimer_ns() - t0 < kWaitLimitNs) {
            }
          }
        }
      }
    } else if (warp == 9) {
      // The whole warp runs the issue loop; one elected lane issues (as in the dK/dV kernel).
      {
        auto mwait = [&](uint32_t bar, uint32_t parity) -> bool {
          return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, status));
        };
        bool ok = mwait(smem_u32(&ctl->fix_full), 0);
        tc_fence_after();
        const uint32_t q_tile = smem_u32(s_q), do_tile = smem_u32(s_do);
        // Issue order per step u: S(u+1) once the softmax has read S(u), then dQ(u), dP(u+1);
        // the tensor core computes S(u+1) while the softmax forms dS(u).  V_j's slot is handed
        // back behind dP, K_j's behind dQ.
        auto tile = [&](int t) { return smem_u32(s_ring + (t % kDqSlots) * G::kTileBytes); };
        auto tile_ready = [&](int t) {
          const bool r = mwait(smem_u32(&ctl->tile_full[t % kDqSlots]), (t / kDqSlots) & 1);
          tc_fence_after();
          return r;
        };
        auto release = [&](int t) { tc_commit(smem_u32(&ctl->tile_empty[t % kDqSlots])); };
        ok = ok && tile_ready(0);
        if (ok) {
          if (elect_one()) {
            mma_s_type<D>(tmem, q_tile, tile(0));           // S  = Q_i K_j^T
            tc_commit(smem_u32(&ctl->s_full));
          }
          __syncwarp();
          ok = tile_ready(1);
        }
        if (ok) {
          if (elect_one()) {
            mma_s_type<D>(tmem + 128, do_tile, tile(1));    // dP = dO_i V_j^T
            tc_commit(smem_u32(&ctl->dp_full));
            release(1);
          }
          __syncwarp();
        }
        for (int u = 0; u < nk && ok; ++u) {
          const bool more = u + 1 < nk;
          if (more) {
            ok = mwait(smem_u32(&ctl->p_full), u & 1);
            if (ok) ok = tile_ready(2 * u + 2);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
              mma_s_type<D>(tmem, q_tile, tile(2 * u + 2));
              tc_commit(smem_u32(&ctl->s_full));
            }
            __syncwarp();
          }
          ok = mwait(smem_u32(&ctl->ds_full), u & 1);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
            mma_acc<D>(tmem + 256, tmem + 128, tile(2 * u), u > 0);   // dQ += dS K_j
            release(2 * u);
          }
          __syncwarp();
          if (more) {
            ok = tile_ready(2 * u + 3);
            if (!ok) break;
            if (elect_one()) {
              mma_s_type<D>(tmem + 128, do_tile, tile(2 * u + 3));
              tc_commit(smem_u32(&ctl->dp_full));
              release(2 * u + 3);
            }
            __syncwarp();
          }
        }
        if (elect_one()) {
          if (ok) tc_commit(smem_u32(&ctl->o_full));
          tc_commit(smem_u32(&ctl->drain));
        }
        __syncwarp();
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    regs_inc<216>();
    const int w4 = warp % 4, hc = warp / 4;
    const int r = w4 * 32 + lane;                  // query row within the block (TMEM lane)
    const int row = iblk * kTileRows + r;
    const bool live = row < n;
    const size_t ridx = static_cast<size_t>(bh) * n + (live ? row : 0);
    const float lse2_row = live ? args.lse[ridx] * kLog2e : 0.f;
    const float d_row = live ? args.delta[ridx] : 0.f;
    const uint32_t lane_addr = static_cast<uint32_t>(w4 * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + 64 * hc;
    const uint32_t t_dp = tmem + lane_addr + 128 + 64 * hc;
    bool ok = true;
    for (int u = 0; u < nk && ok; ++u) {
      ok = wait_phase(smem_u32(&ctl->s_full), u & 1, abort_flag, status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int k0 = u * kTileRows + 64 * hc;      // first key column of this half
      const bool any_masked = (CAUSAL && u == iblk) || (u + 1) * kTileRows > n;
      float p[64];
      const auto vis = [&](int k) { return k0 + k < n && (!CAUSAL || k0 + k <= row); };
      if (any_masked)
        softmax_p<false, false, true>(t_s, args.c, nullptr, lse2_row, vis, p);
      else
        softmax_p<false, false, false>(t_s, args.c, nullptr, lse2_row, vis, p);
      // S has been read into registers: the tensor core may overwrite it with the next S
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full));
      ok = wait_phase(smem_u32(&ctl->dp_full), u & 1, abort_flag, status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // dS lands over the dP columns (tmem + 128), where the dQ product takes its A operand
      softmax_ds<false>(t_dp, nullptr, d_row, p);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->ds_full));
    }
    if (ok) {
      ok = wait_phase(smem_u32(&ctl->o_full), 0, abort_flag, status);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok && D == 128) {
      // bulk-store epilogue, as in the dK/dV kernel: the warp's rows of dQ through the Q tile
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_addr + 256 + G::kHalfCols * hc;
      uint32_t rr[2][32];
      tmem_ld32(t_acc, rr[0]);
      tmem_ld32(t_acc + 32, rr[1]);
      tmem_ld_wait();
      const uint32_t box = smem_u32(s_q) + hc * (kTileRows * 128);
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(rr[g / 4][8 * (g % 4) + 2 * i]) * args.scale,
                              __uint_as_float(rr[g / 4][8 * (g % 4) + 2 * i + 1]) * args.scale);
        st_shared_v4(box + r * 128 + ((g ^ (r & 7)) * 16), pk[0], pk[1], pk[2], pk[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int wrow = iblk * kTileRows + w4 * 32;   // the warp's first query row
      if (lane == 0 && wrow < n) {
        tma_store_3d(&map_g0, box + w4 * 32 * 128, 64 * hc, wrow, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      __syncwarp();
    } else if (ok) {
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_addr + 256 + G::kHalfCols * hc;
      __nv_bfloat16* dst = args.g0 + ridx * D + G::kHalfCols * hc;
#pragma unroll
      for (int cb = 0; cb < G::kHalfCols / 32; ++cb) {
        uint32_t rr[32];
        tmem_ld32(t_acc + cb * 32, rr);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * args.scale,
                              __uint_as_float(rr[2 * i + 1]) * args.scale);
        if (live) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + cb * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace exattn
