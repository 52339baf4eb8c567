// unit_probe.cu -- standalone diagnostic for the sm_103a building blocks the attention kernel
// relies on.  Not part of libexattn.so; tests/test_gpu_unit_probe.py builds and runs it.
//
//  1. Exactness of the tcgen05 operand conventions: S = Q K^T with both operands K-major in
//     128B/64B-swizzled shared memory written by TMA, and O = P V with P read from tensor memory
//     and V MN-major in shared memory; bf16 and e4m3, head dims 64 and 128; small integer data so
//     the fp32 results must match the CPU exactly.
//  2. Per-SM issue rates: MUFU ex2 (f32, bf16x2, f16x2), FFMA, and tcgen05.mma cycles per
//     instruction for the shapes and the issue order the attention kernel uses.
// Prints one line per measurement and "PROBE PASS" / "PROBE FAIL".
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>
#include <cmath>
#include "sm103_ptx.cuh"

using namespace exattn;

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e), __FILE__, __LINE__); exit(1);} } while (0)

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeFn g_encode = nullptr;

static void make_map(CUtensorMap* m, void* ptr, int esize, int d, int rows, int box_inner, CUtensorMapSwizzle sw) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, 1};
  cuuint64_t strides[2] = {(cuuint64_t)d * esize, (cuuint64_t)d * esize * rows};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, ptr, dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) { printf("encode failed %d\n", (int)r); exit(1); }
}

// One CTA, 128 threads. Q,K: [128, D] ; V: [128 keys, D]; P: [128, 128] (given in global, as raw 32-bit words)
// S out [128,128] f32; O out [128, D] f32.
// FP8: 0 -> bf16, 1 -> e4m3
template <int D, int FP8>
__global__ void __launch_bounds__(128, 1) k_probe(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, const uint32_t* __restrict__ pwords,
                        float* __restrict__ s_out, float* __restrict__ o_out, int* err) {
  constexpr int ES = FP8 ? 1 : 2;
  constexpr int ROWB = D * ES;                       // bytes per row
  constexpr int SWB = ROWB >= 128 ? 128 : ROWB;      // swizzle span bytes
  constexpr int NBOX = ROWB / SWB;                   // boxes per tile row
  constexpr int TILE = 128 * ROWB;                   // bytes per 128-row tile
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm; uint8_t* sK = sm + TILE; uint8_t* sV = sm + 2 * TILE;
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x, warp = tid / 32;
  if (warp == 0) { tmem_alloc(smem_u32(&tbase), 512); tmem_relinquish(); }
  if (tid == 0) { mbar_init(smem_u32(&bars[0]), 1); mbar_init(smem_u32(&bars[1]), 1); fence_mbar_init(); }
  tc_fence_before(); __syncthreads(); tc_fence_after();
  const uint32_t tm = tbase;
  if (tid == 0) {
    uint32_t b = smem_u32(&bars[0]);
    mbar_arrive_expect_tx(b, 3 * TILE);
    for (int i = 0; i < NBOX; ++i) {
      int el = i * SWB / ES;
      tma_load_3d(smem_u32(sQ + i * 128 * SWB), &mq, b, el, 0, 0);
      tma_load_3d(smem_u32(sK + i * 128 * SWB), &mk, b, el, 0, 0);
      tma_load_3d(smem_u32(sV + i * 128 * SWB), &mv, b, el, 0, 0);
    }
  }
  // P row into TMEM columns [256, 256 + PCOLS)
  constexpr int PCOLS = FP8 ? 32 : 64;
  {
    uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int c = 0; c < PCOLS; c += 16) {
      uint32_t r[16];
      for (int i = 0; i < 16; ++i) r[i] = pwords[tid * PCOLS + c + i];
      tmem_st16(tm + lane_base + 256 + c, r);
    }
    tmem_st_wait();
  }
  tc_fence_before(); __syncthreads(); tc_fence_after();
  if (tid == 0) {
    uint32_t b = smem_u32(&bars[0]);
    int spins = 0;
    while (!mbar_try_wait(b, 0)) { if (++spins > (1 << 24)) { atomicExch(err, 1); break; } }
    tc_fence_after();
    const uint32_t swmode = SWB == 128 ? kSwizzle128B : kSwizzle64B;
    const uint32_t sbo = 8 * SWB;
    // S = Q K^T, M=128 N=128 K=D
    constexpr int KSTEP_B = 32;                       // bytes of K per MMA (16 bf16 / 32 e4m3)
    const uint32_t idS = instr_desc(128, 128, FP8 ? 0 : 1, false, false);
    for (int kb = 0; kb < ROWB / KSTEP_B; ++kb) {
      int box = (kb * KSTEP_B) / SWB, within = (kb * KSTEP_B) % SWB;
      uint64_t da = smem_desc(smem_u32(sQ + box * 128 * SWB + within), 16, sbo, swmode);
      uint64_t db = smem_desc(smem_u32(sK + box * 128 * SWB + within), 16, sbo, swmode);
      if (FP8) mma_f8_ss(tm + 0, da, db, idS, kb > 0); else mma_f16_ss(tm + 0, da, db, idS, kb > 0);
    }
    // O = P V, M=128 N=D K=128 keys; V MN-major: row = key (SWB bytes per row per box)
    const uint32_t idO = instr_desc(128, D, FP8 ? 0 : 1, false, true);
    constexpr int KEYS_PER_MMA = FP8 ? 32 : 16;
    for (int kb = 0; kb < 128 / KEYS_PER_MMA; ++kb) {
      uint64_t dv = smem_desc(smem_u32(sV + kb * KEYS_PER_MMA * SWB), 128 * SWB, sbo, swmode);
      uint32_t a = tm + 256 + kb * 8;
      if (FP8) mma_f8_ts(tm + 128, a, dv, idO, kb > 0); else mma_f16_ts(tm + 128, a, dv, idO, kb > 0);
    }
    tc_commit(smem_u32(&bars[1]));
    spins = 0;
    while (!mbar_try_wait(smem_u32(&bars[1]), 0)) { if (++spins > (1 << 24)) { atomicExch(err, 2); break; } }
  }
  tc_fence_before(); __syncthreads(); tc_fence_after();
  {
    uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int c = 0; c < 128; c += 32) {
      uint32_t r[32];
      tmem_ld32(tm + lane_base + c, r);
      tmem_ld_wait();
      for (int i = 0; i < 32; ++i) s_out[tid * 128 + c + i] = __uint_as_float(r[i]);
    }
    for (int c = 0; c < D; c += 32) {
      uint32_t r[32];
      tmem_ld32(tm + lane_base + 128 + c, r);
      tmem_ld_wait();
      for (int i = 0; i < 32; ++i) o_out[tid * D + c + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before(); __syncthreads(); tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, 512);
}

static uint16_t f2bf(float f) { uint32_t u; memcpy(&u, &f, 4); return (uint16_t)(u >> 16); }  // exact for small ints
static float e4m3_val(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  float v = e == 0 ? ldexpf(m / 8.0f, -6) : ldexpf(1 + m / 8.0f, e - 7);
  return s ? -v : v;
}

template <int D, int FP8>
static bool run_probe(const char* name) {
  const int ES = FP8 ? 1 : 2;
  std::vector<float> q(128 * D), k(128 * D), v(128 * D), p(128 * 128);
  std::vector<uint8_t> qb(128 * D * ES), kb(128 * D * ES), vb(128 * D * ES);
  srand(1234 + D + FP8);
  // small exact values
  const float vals8[] = {-2, -1.5f, -1, -0.5f, 0, 0.5f, 1, 1.5f, 2};
  const uint8_t codes8[] = {0xC0, 0xBC, 0xB8, 0xB0, 0x00, 0x30, 0x38, 0x3C, 0x40};
  auto fill = [&](std::vector<float>& f, std::vector<uint8_t>& raw) {
    for (size_t i = 0; i < f.size(); ++i) {
      int j = rand() % 9;
      f[i] = vals8[j];
      if (FP8) raw[i] = codes8[j];
      else { uint16_t b = f2bf(vals8[j]); memcpy(&raw[2 * i], &b, 2); }
    }
  };
  fill(q, qb); fill(k, kb); fill(v, vb);
  for (int i = 0; i < 128; ++i) if (std::fabs(e4m3_val(codes8[i % 9]) - vals8[i % 9]) > 0) { printf("code table wrong\n"); }
  // P: values in {0, 0.25, 0.5, 1}
  const float pv[] = {0, 0.25f, 0.5f, 1.0f};
  const uint8_t pc8[] = {0x00, 0x28, 0x30, 0x38};
  std::vector<uint32_t> pw(128 * (FP8 ? 32 : 64));
  for (int r = 0; r < 128; ++r)
    for (int c = 0; c < 128; ++c) {
      int j = rand() % 4;
      p[r * 128 + c] = pv[j];
      if (FP8) { uint32_t& w = pw[r * 32 + c / 4]; if (c % 4 == 0) w = 0; w |= (uint32_t)pc8[j] << (8 * (c % 4)); }
      else { uint32_t& w = pw[r * 64 + c / 2]; if (c % 2 == 0) w = 0; w |= (uint32_t)f2bf(pv[j]) << (16 * (c % 2)); }
    }
  void *dq, *dk, *dv; uint32_t* dp; float *ds, *dout; int* derr;
  CK(cudaMalloc(&dq, qb.size())); CK(cudaMalloc(&dk, kb.size())); CK(cudaMalloc(&dv, vb.size()));
  CK(cudaMalloc(&dp, pw.size() * 4)); CK(cudaMalloc(&ds, 128 * 128 * 4)); CK(cudaMalloc(&dout, 128 * D * 4));
  CK(cudaMalloc(&derr, 4)); CK(cudaMemset(derr, 0, 4));
  CK(cudaMemcpy(dq, qb.data(), qb.size(), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dk, kb.data(), kb.size(), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dv, vb.data(), vb.size(), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dp, pw.data(), pw.size() * 4, cudaMemcpyHostToDevice));
  CUtensorMap mq, mk, mv;
  int rowb = D * ES, swb = rowb >= 128 ? 128 : rowb;
  CUtensorMapSwizzle sw = swb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  make_map(&mq, dq, ES, D, 128, swb / ES, sw);
  make_map(&mk, dk, ES, D, 128, swb / ES, sw);
  make_map(&mv, dv, ES, D, 128, swb / ES, sw);
  size_t smem = 3 * 128 * rowb + 1024;
  CK(cudaFuncSetAttribute(k_probe<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  k_probe<D, FP8><<<1, 128, smem>>>(mq, mk, mv, dp, ds, dout, derr);
  CK(cudaGetLastError());
  CK(cudaDeviceSynchronize());
  int herr; CK(cudaMemcpy(&herr, derr, 4, cudaMemcpyDeviceToHost));
  std::vector<float> s(128 * 128), o(128 * D);
  CK(cudaMemcpy(s.data(), ds, s.size() * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(o.data(), dout, o.size() * 4, cudaMemcpyDeviceToHost));
  double es = 0, eo = 0;
  int bad_s = 0, bad_o = 0;
  for (int i = 0; i < 128; ++i)
    for (int j = 0; j < 128; ++j) {
      double ref = 0; for (int t = 0; t < D; ++t) ref += (double)q[i * D + t] * k[j * D + t];
      double e = std::fabs(ref - s[i * 128 + j]); if (e > es) es = e; if (e > 0) ++bad_s;
    }
  for (int i = 0; i < 128; ++i)
    for (int t = 0; t < D; ++t) {
      double ref = 0; for (int j = 0; j < 128; ++j) ref += (double)p[i * 128 + j] * v[j * D + t];
      double e = std::fabs(ref - o[i * D + t]); if (e > eo) eo = e; if (e > 0) ++bad_o;
    }
  printf("[%s] err_flag=%d  S: max_err=%g bad=%d   O: max_err=%g bad=%d   sample S00=%g O00=%g\n", name, herr, es, bad_s, eo, bad_o, s[0], o[0]);
  cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dp); cudaFree(ds); cudaFree(dout); cudaFree(derr);
  return es == 0 && eo == 0 && herr == 0;
}

// ---------------- throughput probes ----------------
template <int KIND>
__global__ void __launch_bounds__(1024, 1) k_rate(float* out, long long* cyc, int iters) {
  float x[8];
  for (int i = 0; i < 8; ++i) x[i] = -1.0f - 0.001f * (threadIdx.x + i);
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (KIND == 0) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(x[i]));
      else if (KIND == 1) asm volatile("fma.rn.f32 %0, %0, 0f3F7FFFFF, 0f3A83126F;" : "+f"(x[i]));
      else if (KIND == 2) { uint32_t& u = reinterpret_cast<uint32_t&>(x[i]); asm volatile("ex2.approx.ftz.bf16x2 %0, %0;" : "+r"(u)); }
      else { uint32_t& u = reinterpret_cast<uint32_t&>(x[i]); asm volatile("ex2.approx.f16x2 %0, %0;" : "+r"(u)); }
    }
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0; for (int i = 0; i < 8; ++i) s += x[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

static void run_rates(int nsm) {
  float* out; long long* cyc;
  CK(cudaMalloc(&out, (size_t)nsm * 1024 * 4)); CK(cudaMalloc(&cyc, nsm * 8));
  const char* names[] = {"ex2.f32", "ffma.f32", "ex2.bf16x2", "ex2.f16x2"};
  for (int kind = 0; kind < 4; ++kind) {
    int iters = 4096;
    for (int rep = 0; rep < 2; ++rep) {
      if (kind == 0) k_rate<0><<<nsm, 1024>>>(out, cyc, iters);
      if (kind == 1) k_rate<1><<<nsm, 1024>>>(out, cyc, iters);
      if (kind == 2) k_rate<2><<<nsm, 1024>>>(out, cyc, iters);
      if (kind == 3) k_rate<3><<<nsm, 1024>>>(out, cyc, iters);
      CK(cudaGetLastError()); CK(cudaDeviceSynchronize());
    }
    std::vector<long long> c(nsm); CK(cudaMemcpy(c.data(), cyc, nsm * 8, cudaMemcpyDeviceToHost));
    double mean = 0; for (auto v : c) mean += v; mean /= nsm;
    double ops = 1024.0 * iters * 8;
    printf("[rate] %-10s  %.2f instr/clk/SM (mean cycles %.0f)\n", names[kind], ops / mean, mean);
  }
  cudaFree(out); cudaFree(cyc);
}

// MODE 0: SS N128 Kmajor; 1: SS N256; 2: TS N128 (A tmem) B MN-major; 3: SS N128 B MN-major;
// 4: alternate SS N128 (S) and TS N128 (PV) like the kernel; 5: fp8 SS N128 K32; 6: fp8 TS N128
template <int MODE>
__global__ void __launch_bounds__(384, 1) k_mma(long long* cyc, int nmma, int* err) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar;
  __shared__ uint64_t dummy[4];
  __shared__ uint32_t tbase;
  int tid = threadIdx.x;
  for (int i = tid; i < 98304 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3C003C00u;
  __shared__ volatile int done;
  if (tid == 0) done = 0;
  if (tid < 32) { tmem_alloc(smem_u32(&tbase), 512); tmem_relinquish(); }
  if (tid == 0) { mbar_init(smem_u32(&bar), 1); for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&dummy[q]), 1); fence_mbar_init(); }
  fence_proxy_async_smem();
  tc_fence_before(); __syncthreads(); tc_fence_after();
  uint32_t tm = tbase;
  if (tid == 0) {
    const uint32_t idS = instr_desc(128, 128, 1, false, false);
    const uint32_t idS256 = instr_desc(128, 256, 1, false, false);
    const uint32_t idPV = instr_desc(128, 128, 1, false, true);
    const uint32_t idS8 = instr_desc(128, 128, 0, false, false);
    const uint32_t idPV8 = instr_desc(128, 128, 0, false, true);
    uint64_t da = smem_desc(smem_u32(sm), 16, 1024, kSwizzle128B);
    uint64_t db = smem_desc(smem_u32(sm + 32768), 16, 1024, kSwizzle128B);
    uint64_t dv = smem_desc(smem_u32(sm + 65536), 16384, 1024, kSwizzle128B);
    long long t0 = clock64();
    for (int i = 0; i < nmma; ++i) {
      uint32_t acc = i > 3;
      if (MODE == 0) mma_f16_ss(tm + (i & 1) * 128, da + (i & 3) * 2, db + (i & 3) * 2, idS, acc);
      if (MODE == 1) mma_f16_ss(tm + (i & 1) * 256, da + (i & 3) * 2, db + (i & 3) * 2, idS256, acc);
      if (MODE == 2) mma_f16_ts(tm + 256 + (i & 1) * 128, tm + (i & 1) * 128 + (i & 7) * 8, dv + (i & 7) * 128, idPV, acc);
      if (MODE == 3) mma_f16_ss(tm + (i & 1) * 128, da + (i & 3) * 2, dv + (i & 7) * 128, idPV, acc);
      if (MODE == 4) {
        if ((i >> 3) & 1) mma_f16_ts(tm + 256 + ((i >> 4) & 1) * 128, tm + ((i >> 4) & 1) * 128 + (i & 7) * 8, dv + (i & 7) * 128, idPV, acc);
        else mma_f16_ss(tm + ((i >> 4) & 1) * 128, da + (i & 3) * 2, db + (i & 3) * 2, idS, acc);
      }
      if (MODE == 5) mma_f8_ss(tm + (i & 1) * 128, da + (i & 3) * 2, db + (i & 3) * 2, idS8, acc);
      if (MODE == 6) mma_f8_ts(tm + 256 + (i & 1) * 128, tm + (i & 1) * 128 + (i & 3) * 8, dv + (i & 3) * 256, idPV8, acc);
      if (MODE == 7 || MODE == 10 || MODE >= 30) {  // kernel order: PV0 S0 PV1 S1, P aliased over S
        const int g = (i >> 3) & 3, k = i & 7, h = g >> 1;
        if ((g & 1) == 0) mma_f16_ts(tm + 256 + h * 128, tm + h * 128 + k * 8, dv + k * 128, idPV, 1);
        else mma_f16_ss(tm + h * 128, da + (k & 3) * 2, db + (k & 3) * 2, idS, k > 0);
        if (MODE == 33 && k == 7) tc_commit(smem_u32(&dummy[g]));
        if (MODE == 34 && k == 7) { tc_commit(smem_u32(&dummy[g])); if (g & 1) tc_commit(smem_u32(&dummy[(g + 1) & 3])); }
        if (MODE == 35 && k == 7 && g == 3) tc_commit(smem_u32(&dummy[0]));
      }
      if (MODE == 8 || MODE == 9) {  // same order, PV N=64; 8: P aliased over S, 9: P separate
        const uint32_t idPV64 = instr_desc(128, 64, 1, false, true);
        const int g = (i >> 3) & 3, k = i & 7, h = g >> 1;
        const uint32_t pcol = MODE == 8 ? h * 128 : 256 + h * 64;
        if ((g & 1) == 0) mma_f16_ts(tm + 384 + h * 64, tm + pcol + k * 8, dv + k * 128, idPV64, 1);
        else mma_f16_ss(tm + h * 128, da + (k & 3) * 2, db + (k & 3) * 2, idS, k > 0);
      }
      if (MODE == 11) mma_f16_ss(tm + ((i >> 3) & 1) * 128, da + (i & 3) * 2, db + (i & 3) * 2, idS, (i & 7) > 0);
      if (MODE == 12) mma_f16_ss(tm + ((i >> 3) & 1) * 256, da + (i & 3) * 2, db + (i & 3) * 2, idS256, (i & 7) > 0);
      if (MODE == 13) {  // S0 and S1 k-steps interleaved (two chains), then PV0/PV1 interleaved
        const int g = (i >> 4) & 1, k = (i >> 1) & 7, h = i & 1;
        if (g == 1) mma_f16_ts(tm + 256 + h * 128, tm + h * 128 + k * 8, dv + k * 128, idPV, 1);
        else mma_f16_ss(tm + h * 128, da + (k & 3) * 2, db + (k & 3) * 2, idS, k > 0);
      }
      if (MODE >= 15 && MODE <= 19) {  // SS/TS alternation with no TMEM overlap: group size G
        const int G = MODE == 15 ? 1 : MODE == 16 ? 4 : MODE == 17 ? 8 : MODE == 18 ? 16 : 64;
        const int k = i & 7;
        if ((i / G) & 1) mma_f16_ts(tm + 384, tm + 256 + k * 8, dv + k * 128, instr_desc(128, 128, 1, false, true), 1);
        else mma_f16_ss(tm + 0, da + (k & 3) * 2, db + (k & 3) * 2, idS, 1);
      }
      if (MODE == 20) mma_f16_ts(tm + 384 + ((i >> 3) & 1) * 64, tm + 256 + (i & 7) * 8, dv + (i & 7) * 128, instr_desc(128, 64, 1, false, true), 1);
      if (MODE == 14) {  // same-D chain of TS N128
        mma_f16_ts(tm + 256 + ((i >> 3) & 1) * 128, tm + (i & 7) * 8, dv + (i & 7) * 128, idPV, 1);
      }
    }
    done = 1;
    tc_commit(smem_u32(&bar));
    int spins = 0;
    while (!mbar_try_wait(smem_u32(&bar), 0)) { if (++spins > (1 << 26)) { atomicExch(err, 3); break; } }
    long long t1 = clock64();
    cyc[blockIdx.x] = t1 - t0;
  } else if ((MODE == 30 || MODE == 32) && tid >= 128 && tid < 384) {
    // softmax-like TMEM traffic at the real kernel's pace: one S row read + P row write per ~1400 cycles
    const int w = (tid / 32) % 4, h = (tid / 128) - 1;
    const uint32_t base = tm + ((uint32_t)(w * 32) << 16) + h * 128;
    uint32_t r[32];
    for (int it = 0; it < (1 << 16) && !done; ++it) {
      for (int c = 0; c < 4; ++c) tmem_ld32(base + c * 32, r);
      tmem_ld_wait();
      for (int c = 0; c < 2; ++c) tmem_st32(base + c * 32, r);
      tmem_st_wait();
      long long t0 = clock64();
      while (clock64() - t0 < 1200) {}
    }
  } else if ((MODE == 31 || MODE == 32) && tid >= 64 && tid < 128) {
    // TMA-like smem writes: 2 warps store 16 B per lane into a 16 KB scratch area, ~32 B/clk total
    uint4* dst = reinterpret_cast<uint4*>(sm + 98304);
    const int l = tid - 64;
    for (int it = 0; it < (1 << 20) && !done; ++it) {
      dst[(it * 64 + l) & 1023] = make_uint4(it, it, it, it);
      long long t0 = clock64();
      while (clock64() - t0 < 20) {}
    }
  } else if (MODE == 10 && tid >= 128 && tid < 384) {
    // 8 warps hammer TMEM like the softmax: load 128 S columns, store 64 P columns
    const int w = (tid / 32) % 4, h = (tid / 128) - 1;
    const uint32_t base = tm + ((uint32_t)(w * 32) << 16) + h * 128;
    uint32_t r[32];
    for (int it = 0; it < (1 << 20) && !done; ++it) {
      for (int c = 0; c < 4; ++c) tmem_ld32(base + c * 32, r);
      tmem_ld_wait();
      for (int c = 0; c < 2; ++c) tmem_st32(base + c * 32, r);
      tmem_st_wait();
    }
  }
  tc_fence_before(); __syncthreads(); tc_fence_after();
  if (tid < 32) tmem_dealloc(tm, 512);
}

template <int MODE>
int run_mma_mode(const char* name, int nsm, double flop_per_mma) {
  long long* cyc; int* err;
  CK(cudaMalloc(&cyc, nsm * 8)); CK(cudaMalloc(&err, 4)); CK(cudaMemset(err, 0, 4));
  CK(cudaFuncSetAttribute(k_mma<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024));
  int nmma = 4096;
  const int nthr = (MODE == 10 || MODE == 30 || MODE == 32) ? 384 : 128;
  for (int rep = 0; rep < 2; ++rep) { k_mma<MODE><<<nsm, nthr, 120 * 1024>>>(cyc, nmma, err); CK(cudaGetLastError()); CK(cudaDeviceSynchronize()); }
  std::vector<long long> c(nsm); CK(cudaMemcpy(c.data(), cyc, nsm * 8, cudaMemcpyDeviceToHost));
  int herr; CK(cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost));
  double mean = 0; for (auto v : c) mean += v; mean /= nsm;
  printf("%-34s %7.1f cycles/mma  %6.0f flop/clk/SM  err=%d\n", name, mean / nmma, flop_per_mma * nmma / mean, herr);
  cudaFree(cyc); cudaFree(err);
  return 0;
}


// The attention order with each product issued as one asm block (mma_chain_*_off, the form the
// kernels use), one tcgen05.commit per product.  MODE 0: nothing else; 1: per product also a
// try_wait on a completed barrier, a tcgen05 fence, a second commit and a clock store (the
// issuing thread's bookkeeping); 2: warps 4-11 run independent FMA/ex2 work meanwhile (busy
// softmax-like warps on every SMSP); 3: warps 4-11 move S, P and O through TMEM at the
// softmax's pace.
template <int MODE>
__global__ void __launch_bounds__(384, 1) k_chain(long long* cyc, int nmma, int* err, float* sink) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar, done_bar;
  __shared__ uint64_t dummy[4];
  __shared__ uint32_t tbase;
  __shared__ volatile int done;
  const int tid = threadIdx.x;
  for (int i = tid; i < 98304 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3C003C00u;
  if (tid == 0) done = 0;
  if (tid < 32) { tmem_alloc(smem_u32(&tbase), 512); tmem_relinquish(); }
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_init(smem_u32(&done_bar), 1);
    for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&dummy[q]), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  tc_fence_before(); __syncthreads(); tc_fence_after();
  const uint32_t tm = tbase;
  if (tid == 0) {
    mbar_arrive(smem_u32(&done_bar));  // phase 0 complete: the MODE 1 try_wait always succeeds
    const uint32_t idS = instr_desc(128, 128, 1, false, false);
    const uint32_t idPV = instr_desc(128, 128, 1, false, true);
    const uint64_t da = smem_desc(smem_u32(sm), 16, 1024, kSwizzle128B);
    const uint64_t db = smem_desc(smem_u32(sm + 32768), 16, 1024, kSwizzle128B);
    const uint64_t dv = smem_desc(smem_u32(sm + 65536), 16384, 1024, kSwizzle128B);
    const long long t0 = clock64();
    for (int i = 0; i < nmma; i += 8) {
      const int g = (i >> 3) & 3, h = g >> 1;
      if (MODE == 1) {
        if (!mbar_try_wait(smem_u32(&done_bar), 0)) atomicExch(err, 5);
        tc_fence_after();
      }
      if ((g & 1) == 0)
        mma_chain_ts_off<8, 0, 128, 8, 16, 24, 32, 40, 48, 56>(tm + 256 + h * 128, idPV, 1u,
                                                              tm + h * 128, dv);
      else
        mma_chain_ss_off<8, 0, 2, 4, 6, 1024, 1026, 1028, 1030>(tm + h * 128, idS, 0u, da, db);
      tc_commit(smem_u32(&dummy[g]));
      if (MODE == 1) {
        tc_commit(smem_u32(&dummy[(g + 1) & 3]));
        reinterpret_cast<long long*>(sink)[(i >> 3) & 63] = clock64();
      }
    }
    tc_commit(smem_u32(&bar));
    int spins = 0;
    while (!mbar_try_wait(smem_u32(&bar), 0)) { if (++spins > (1 << 26)) { atomicExch(err, 3); break; } }
    cyc[blockIdx.x] = clock64() - t0;
    done = 1;
  } else if (tid >= 128 && MODE == 2) {
    float a[8];
    for (int k = 0; k < 8; ++k) a[k] = tid + k;
    for (int it = 0; it < (1 << 20) && !done; ++it) {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          a[q] = (q == 4 || q == 7) ? ex2_mufu(a[q] * -1e-3f) : fmaf(a[q], 0.999f, 0.5f);
      }
    }
    float t = 0.f;
    for (int k = 0; k < 8; ++k) t += a[k];
    if (t == 12345.f) sink[tid] = t;
  } else if (tid >= 128 && MODE == 3) {
    const int w = (tid / 32) % 4, h = (tid / 128) - 1;
    const uint32_t sb = tm + (static_cast<uint32_t>(w * 32) << 16) + h * 128, ob = sb + 256;
    float acc = tid * 1e-3f;
    for (int it = 0; it < (1 << 16) && !done; ++it) {
      uint32_t r[4][32];
      for (int c = 0; c < 4; ++c) tmem_ld32(sb + c * 32, r[c]);
      tmem_ld_wait();
      float a2[8];
      for (int k = 0; k < 8; ++k) a2[k] = __uint_as_float(r[0][k] & 0x3FFFFFFFu) * 1e-9f + acc;
#pragma unroll 4
      for (int k = 0; k < 64; ++k)
        for (int q = 0; q < 8; ++q) a2[q] = fmaf(ex2_mufu(a2[q] * -1e-3f), 1e-3f, a2[q]);
      for (int q = 0; q < 8; ++q) acc += a2[q];
      uint32_t o[32];
      for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(acc + k);
      tmem_st32(sb, o);
      tmem_st32(sb + 32, o);
      tmem_st_wait();
      if (it & 1) {
        for (int c = 0; c < 4; ++c) {
          uint32_t x[32];
          tmem_ld32(ob + c * 32, x);
          tmem_ld_wait();
          for (int k = 0; k < 32; ++k) x[k] = __float_as_uint(__uint_as_float(x[k]) * 0.999f);
          tmem_st32(ob + c * 32, x);
        }
        tmem_st_wait();
      }
    }
    if (acc == 12345.f) sink[tid] = acc;
  }
  tc_fence_before(); __syncthreads(); tc_fence_after();
  if (tid < 32) tmem_dealloc(tm, 512);
}

template <int MODE>
void run_chain_mode(const char* name, int nsm) {
  long long* cyc; int* err; float* sink;
  CK(cudaMalloc(&cyc, nsm * 8)); CK(cudaMalloc(&err, 4)); CK(cudaMemset(err, 0, 4));
  CK(cudaMalloc(&sink, 384 * 4)); CK(cudaMemset(sink, 0, 384 * 4));
  CK(cudaFuncSetAttribute(k_chain<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024));
  const int nmma = 4096;
  for (int rep = 0; rep < 2; ++rep) {
    k_chain<MODE><<<nsm, 384, 120 * 1024>>>(cyc, nmma, err, sink);
    CK(cudaGetLastError()); CK(cudaDeviceSynchronize());
  }
  std::vector<long long> c(nsm); CK(cudaMemcpy(c.data(), cyc, nsm * 8, cudaMemcpyDeviceToHost));
  int herr; CK(cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost));
  double mean = 0; for (auto v : c) mean += v; mean /= nsm;
  printf("%-34s %7.1f cycles/mma  err=%d\n", name, mean / nmma, herr);
  cudaFree(cyc); cudaFree(err); cudaFree(sink);
}

// mbarrier hand-off latency: warp 4 arrives at a recorded clock, thread 0 polls with try_wait
// (MODE 0) or test_wait (MODE 1) and records when it sees the phase complete.
template <int MODE>
__global__ void __launch_bounds__(256, 1) k_wake(long long* out, int* err) {
  __shared__ uint64_t bar;
  __shared__ long long t_arr;
  const int tid = threadIdx.x;
  if (tid == 0) { mbar_init(smem_u32(&bar), 1); fence_mbar_init(); }
  __syncthreads();
  long long sum = 0;
  for (int it = 0; it < 64; ++it) {
    if (tid == 128) {
      const long long s0 = clock64();
      while (clock64() - s0 < 2000) {}
      t_arr = clock64();
      mbar_arrive(smem_u32(&bar));
    } else if (tid == 0) {
      int spins = 0;
      for (;;) {
        uint32_t ok;
        if (MODE == 0) {
          ok = mbar_try_wait(smem_u32(&bar), it & 1);
        } else {
          asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                       "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(smem_u32(&bar)), "r"(it & 1) : "memory");
        }
        if (ok) break;
        if (++spins > (1 << 26)) { atomicExch(err, 1); break; }
      }
      sum += clock64();
    }
    __syncthreads();
    if (tid == 0) sum -= t_arr;
    __syncthreads();
  }
  if (tid == 0) out[blockIdx.x] = sum / 64;
}

template <int MODE>
void run_wake(const char* name, int nsm) {
  long long* out; int* err;
  CK(cudaMalloc(&out, nsm * 8)); CK(cudaMalloc(&err, 4)); CK(cudaMemset(err, 0, 4));
  k_wake<MODE><<<nsm, 256>>>(out, err); CK(cudaGetLastError()); CK(cudaDeviceSynchronize());
  std::vector<long long> c(nsm); CK(cudaMemcpy(c.data(), out, nsm * 8, cudaMemcpyDeviceToHost));
  int herr; CK(cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost));
  double mean = 0; for (auto v : c) mean += v; mean /= nsm;
  printf("%-34s %7.1f cycles arrive -> seen  err=%d\n", name, mean, herr);
  cudaFree(out); cudaFree(err);
}


int main() {
  cudaDeviceProp prop; CK(cudaGetDeviceProperties(&prop, 0));
  printf("device %s  SMs %d  cc %d.%d  smem/block optin %zu  L2 %d\n", prop.name, prop.multiProcessorCount, prop.major, prop.minor,
         prop.sharedMemPerBlockOptin, prop.l2CacheSize);
  cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&g_encode, 12000, cudaEnableDefault, &q));
  bool ok = true;
  ok &= run_probe<128, 0>("bf16 d128");
  ok &= run_probe<64, 0>("bf16 d64");
  ok &= run_probe<128, 1>("e4m3 d128");
  ok &= run_probe<64, 1>("e4m3 d64");
  const int nsm = prop.multiProcessorCount;
  run_rates(nsm);
  const double f128 = 2.0 * 128 * 128 * 16;
  run_mma_mode<0>("mma SS bf16 M128 N128 K16", nsm, f128);
  run_mma_mode<1>("mma SS bf16 M128 N256 K16", nsm, 2 * f128);
  run_mma_mode<2>("mma TS bf16 M128 N128 K16 (B MN)", nsm, f128);
  run_mma_mode<5>("mma SS e4m3 M128 N128 K32", nsm, 2 * f128);
  run_mma_mode<6>("mma TS e4m3 M128 N128 K32 (B MN)", nsm, 2 * f128);
  run_mma_mode<11>("same-D chains of 8, SS N128", nsm, f128);
  run_mma_mode<14>("same-D chains of 8, TS N128", nsm, f128);
  run_mma_mode<15>("SS/TS alternate every 1", nsm, f128);
  run_mma_mode<17>("SS/TS alternate every 8", nsm, f128);
  run_mma_mode<7>("attention order PV0 S0 PV1 S1", nsm, f128);
  run_mma_mode<35>("attention order + 1 commit/32", nsm, f128);
  run_mma_mode<33>("attention order + commit/group", nsm, f128);
  run_mma_mode<30>("attention order + TMEM ld/st", nsm, f128);
  run_chain_mode<0>("chains: attention order + commit", nsm);
  run_chain_mode<1>("chains + issuer bookkeeping", nsm);
  run_chain_mode<2>("chains + busy warps on every SMSP", nsm);
  run_chain_mode<3>("chains + softmax-paced TMEM S/P/O", nsm);
  run_wake<0>("mbarrier hand-off, try_wait", nsm);
  run_wake<1>("mbarrier hand-off, test_wait", nsm);
  printf("PROBE %s\n", ok ? "PASS" : "FAIL");
  return 0;
}
