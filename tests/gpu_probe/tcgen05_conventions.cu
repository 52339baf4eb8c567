// tcgen05_conventions.cu -- exactness of the tcgen05 operand conventions the attention kernels
// rely on (test infrastructure: built and run by tests/test_gpu_tcgen05_conventions.py, not part
// of libexattn.so).
//
// One CTA computes S = Q K^T with both operands K-major in 128B/64B-swizzled shared memory
// written by TMA, and O = P V with P read from tensor memory and V MN-major in shared memory,
// for bf16 and e4m3 operands at head dims 64 and 128, with the descriptor and instruction-
// descriptor helpers of sm103_ptx.cuh.  The data are small integers and binary fractions, so
// every fp32 result must equal the CPU's exactly.  Prints one line per case and "PROBE PASS" /
// "PROBE FAIL".
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>
#include <cmath>
#include "../../exact_attention_13_gb300/csrc/sm103_ptx.cuh"

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

int main() {
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, 0));
  printf("device %s  SMs %d  cc %d.%d\n", prop.name, prop.multiProcessorCount, prop.major,
         prop.minor);
  cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&g_encode, 12000,
                                      cudaEnableDefault, &q));
  bool ok = true;
  ok &= run_probe<128, 0>("bf16 d128");
  ok &= run_probe<64, 0>("bf16 d64");
  ok &= run_probe<128, 1>("e4m3 d128");
  ok &= run_probe<64, 1>("e4m3 d64");
  printf("PROBE %s\n", ok ? "PASS" : "FAIL");
  return ok ? 0 : 1;
}
