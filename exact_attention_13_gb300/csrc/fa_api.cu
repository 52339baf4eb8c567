// fa_api.cu -- host side of libexattn.so: argument checks, TMA tensor maps, kernel launch, and
// the C ABI declared in include/exact_attention.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/exact_attention.h"
#include "fa_fwd_kernel.cuh"
#include "fa_quant.cuh"
#include "fa_bwd_kernel.cuh"

namespace exattn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 16;

// Bytes of the key-split partials: O_s [splits, B*H, N, d] and LSE_s [splits, B*H, N], fp32.
size_t split_workspace_bytes(int B, int H, int N, int d, int splits) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t bytes = static_cast<size_t>(splits) * rows * (static_cast<size_t>(d) + 1) * 4;
  return (bytes + 255) / 256 * 256;
}

// Per-device status word the kernel writes when a bounded wait runs out (fa_fwd callers that
// pass no status pointer of their own).
__device__ int g_device_status;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Device-side address of g_device_status for the current device, looked up once per device.
int* library_status_ptr(int dev) {
  static std::atomic<int*> cache[kMaxDevices];
  int* p = cache[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return nullptr;
  cache[dev].store(static_cast<int*>(addr), std::memory_order_release);
  return static_cast<int*>(addr);
}

// [B*H, N, d] view of one operand, tiles of box_rows (128) rows x (one swizzle span) with the
// swizzle the MMA descriptors expect.  Rows past N (per head) read as zero (loads) or are clipped
// (stores).
bool encode_operand_map(CUtensorMap* map, const void* ptr, int elem_bytes, int d, int n,
                        int bh, int box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int row_bytes = d * elem_bytes;
  const int sw_bytes = row_bytes >= 128 ? 128 : row_bytes;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n),
                        static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes),
                           static_cast<cuuint64_t>(row_bytes) * static_cast<cuuint64_t>(n)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(sw_bytes / elem_bytes),
                       static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                  3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Per-block fp8 descales, [B*H, ceil(N / 128)] each (null: per-tensor descales).
struct BlockScales {
  const float* dq;
  const float* dk;
  const float* dv;
};

// One launch over the 256-row query blocks [mblock0, mblock0 + mblocks) of every head.
template <int D, bool FP8, bool CAUSAL, bool PV16>
int launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           float c, float out_mult, int* status, int splits, float* o_part, float* lse_part,
           const BlockScales* bs, int mblock0, int mblocks, cudaStream_t stream) {
  constexpr int elem = FP8 ? 1 : 2;
  CUtensorMap mq, mk, mv, mo;
  const int bh = B * H;
  // O (bf16 for every operand type): boxes of one softmax warp's 32 rows, for the bulk-store
  // epilogue
  if (!encode_operand_map(&mq, q, elem, D, N, bh) || !encode_operand_map(&mk, k, elem, D, N, bh) ||
      !encode_operand_map(&mv, v, elem, D, N, bh) || !encode_operand_map(&mo, o, 2, D, N, bh, 32))
    return FA_ERR_CUDA;
  auto kern = fa_fwd_kernel<D, FP8, CAUSAL, PV16>;
  constexpr int smem = smem_bytes<D, FP8, PV16>();
  static_assert(smem <= 227 * 1024, "shared memory per CTA");
  // one CTA per SM (the kernel takes all 512 TMEM columns): ask for > half the SM's smem
  constexpr int smem_request = smem > 120 * 1024 ? smem : 120 * 1024;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  static std::atomic<uint64_t> attr_done{0};
  if (!(attr_done.load(std::memory_order_acquire) & (1ull << dev))) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_request) !=
        cudaSuccess)
      return FA_ERR_CUDA;
    attr_done.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  KernelArgs args;
  args.o = static_cast<__nv_bfloat16*>(o);
  args.lse = lse;
  args.status = status ? status : library_status_ptr(dev);
  if (!args.status) return FA_ERR_CUDA;
  args.o_part = o_part;
  args.lse_part = lse_part;
  args.n = N;
  args.bh = bh;
  args.c = c;
  args.out_mult = out_mult;
  args.dq_blk = bs ? bs->dq : nullptr;
  args.dk_blk = bs ? bs->dk : nullptr;
  args.dv_blk = bs ? bs->dv : nullptr;
  args.nblk = (N + kTileRows - 1) / kTileRows;
  args.mblock0 = mblock0;
  const unsigned mb = static_cast<unsigned>(mblocks);
  const unsigned z = static_cast<unsigned>(splits);
  const dim3 grid = CAUSAL ? dim3(static_cast<unsigned>(bh), mb, z)
                           : dim3(mb, static_cast<unsigned>(bh), z);
  kern<<<grid, kThreads, smem_request, stream>>>(mq, mk, mv, mo, args);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Every query block of every head.  fp8 operands with fp8 P V and the causal mask: causal rows
// near the start of a sequence see only a few keys, so the e4m3 rounding of each probability
// (up to 2^-4 relative) reaches O almost undiluted there; the first query block of every head
// (rows 0-255, at most 256 keys each) therefore runs the instance with the f16 P V product, and
// the other query blocks the fp8 one.
template <int D, bool FP8, bool PV16 = false>
int launch_mask(int causal, const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int N, float c, float om, int* st, int splits, float* op,
                float* lp, const BlockScales* bs, cudaStream_t s) {
  const int mtotal = (N + kCtaRows - 1) / kCtaRows;
  if (!causal)
    return launch<D, FP8, false, PV16>(q, k, v, o, lse, B, H, N, c, om, st, splits, op, lp, bs,
                                       0, mtotal, s);
  if (!FP8 || PV16)
    return launch<D, FP8, true, PV16>(q, k, v, o, lse, B, H, N, c, om, st, splits, op, lp, bs,
                                      0, mtotal, s);
  int rc = launch<D, true, true, true>(q, k, v, o, lse, B, H, N, c, om, st, splits, op, lp, bs, 0,
                                       1, s);
  if (rc == FA_OK && mtotal > 1)
    rc = launch<D, true, true, false>(q, k, v, o, lse, B, H, N, c, om, st, splits, op, lp, bs, 1,
                                      mtotal - 1, s);
  return rc;
}

// Merge of key splits ("FlashAttention · InkStack", section 2.2: key blocks can be processed
// independently and merged associatively).  Each split s left O_s (normalised by its own sum)
// and LSE_s; the merge is LSE = log sum_s e^LSE_s and O = sum_s e^(LSE_s - LSE) O_s, evaluated
// around the largest LSE_s.  One warp per query row, D / 32 consecutive columns per lane.
template <int D>
__global__ void __launch_bounds__(256) combine_splits_kernel(const float* __restrict__ o_part,
                                                             const float* __restrict__ lse_part,
                                                             __nv_bfloat16* __restrict__ o,
                                                             float* __restrict__ lse, int splits,
                                                             long long rows) {
  constexpr int kPer = D / 32;
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x % 32;
  float m = -INFINITY;
  for (int sp = 0; sp < splits; ++sp) m = fmaxf(m, lse_part[sp * rows + row]);
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float l = 0.f;
  for (int sp = 0; sp < splits; ++sp) {
    const float ls = lse_part[sp * rows + row];
    const float w = ls == -INFINITY ? 0.f : expf(ls - m);
    l += w;
    const float* src = o_part + (static_cast<size_t>(sp) * rows + row) * D + lane * kPer;
#pragma unroll
    for (int i = 0; i < kPer; i += 2) {
      const float2 x = *reinterpret_cast<const float2*>(src + i);
      acc[i] = fmaf(w, x.x, acc[i]);
      acc[i + 1] = fmaf(w, x.y, acc[i + 1]);
    }
  }
  const float inv = 1.f / l;
  __nv_bfloat16* dst = o + row * D + lane * kPer;
#pragma unroll
  for (int i = 0; i < kPer; i += 2)
    *reinterpret_cast<uint32_t*>(dst + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
  if (lane == 0) lse[row] = m + logf(l);
}

template <int D>
int launch_combine(const float* o_part, const float* lse_part, void* o, float* lse, int splits,
                   long long rows, cudaStream_t s) {
  const long long blocks = (rows + 7) / 8;
  combine_splits_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      o_part, lse_part, static_cast<__nv_bfloat16*>(o), lse, splits, rows);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bytes of the backward's scratch: D [B*H*N] fp32, rounded up to 256.
size_t bwd_workspace_bytes(int B, int H, int N) {
  const size_t bytes = static_cast<size_t>(B) * H * N * 4;
  return (bytes + 255) / 256 * 256;
}

template <typename K>
bool set_smem_once(K kern, int bytes, int dev, std::atomic<uint64_t>& done) {
  if (done.load(std::memory_order_acquire) & (1ull << dev)) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  done.fetch_or(1ull << dev, std::memory_order_acq_rel);
  return true;
}

// Backward: D, then dK/dV, then dQ, all on `stream`.
template <int D, bool CAUSAL>
int launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, float scale,
               float* delta, int* status, cudaStream_t stream) {
  const int bh = B * H;
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  // outputs: boxes of one softmax warp's 32 rows, for the bulk-store epilogues
  if (!encode_operand_map(&mq, q, 2, D, N, bh) || !encode_operand_map(&mk, k, 2, D, N, bh) ||
      !encode_operand_map(&mv, v, 2, D, N, bh) || !encode_operand_map(&mdo, dout, 2, D, N, bh) ||
      !encode_operand_map(&mdq, dq, 2, D, N, bh, 32) ||
      !encode_operand_map(&mdk, dk, 2, D, N, bh, 32) ||
      !encode_operand_map(&mdv, dv, 2, D, N, bh, 32))
    return FA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  BwdArgs a;
  a.lse = lse;
  a.delta = delta;
  a.status = status ? status : library_status_ptr(dev);
  if (!a.status) return FA_ERR_CUDA;
  a.n = N;
  a.c = scale * 1.4426950408889634f;
  a.scale = scale;
  const long long rows = static_cast<long long>(bh) * N;
  bwd_delta_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta, rows);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  // at least 120 KB each, so that one CTA (which takes all 512 TMEM columns) runs per SM
  constexpr int smem = bwd_smem_bytes<D>(), smem_dq = dq_smem_bytes<D>();
  static_assert(smem <= 227 * 1024 && smem_dq <= 227 * 1024, "shared memory per CTA");
  constexpr int smem_request = smem > 120 * 1024 ? smem : 120 * 1024;
  constexpr int smem_dq_request = smem_dq > 120 * 1024 ? smem_dq : 120 * 1024;
  static std::atomic<uint64_t> done_kv{0}, done_q{0};
  auto kkv = bwd_dkdv_kernel<D, CAUSAL>;
  auto kq = bwd_dq_kernel<D, CAUSAL>;
  if (!set_smem_once(kkv, smem_request, dev, done_kv) ||
      !set_smem_once(kq, smem_dq_request, dev, done_q))
    return FA_ERR_CUDA;
  const unsigned nblk = static_cast<unsigned>((N + kTileRows - 1) / kTileRows);
  const dim3 grid = CAUSAL ? dim3(static_cast<unsigned>(bh), nblk) : dim3(nblk, static_cast<unsigned>(bh));
  a.g0 = static_cast<__nv_bfloat16*>(dk);
  a.g1 = static_cast<__nv_bfloat16*>(dv);
  kkv<<<grid, kBwdThreads, smem_request, stream>>>(mq, mk, mv, mdo, mdk, mdv, a);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  a.g0 = static_cast<__nv_bfloat16*>(dq);
  a.g1 = nullptr;
  kq<<<grid, kBwdThreads, smem_dq_request, stream>>>(mq, mk, mv, mdo, mdq, a);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

__global__ void exp2_probe_kernel(const float* x, float* y, long long n, int mode) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    y[i] = mode == 0 ? ex2_mufu(x[i]) : ex2_poly(x[i]);
}

}  // namespace
}  // namespace exattn

namespace exattn {
namespace {

// Shared argument checks and dispatch of fa_fwd_ex / fa_fwd_split / fa_fwd_fp8_blockscaled.
// splits == 1 writes O and LSE directly; splits > 1 writes per-split partials into
// `workspace`, then merges them.  `bs` (fp8 only) replaces the per-tensor descales.
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int N, int d, float scale, int causal, int dtype, const fa_fwd_opts* opts,
             int splits, void* workspace, size_t workspace_bytes, void* stream,
             const BlockScales* bs = nullptr) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP8_E4M3 && dtype != FA_DTYPE_FP8_E4M3_PV16)
    return FA_ERR_INVALID_ARG;
  const bool fp8 = dtype != FA_DTYPE_BF16;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (splits < 1 || splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  float dq = 1.f, dk = 1.f, dv = 1.f;
  int* status = nullptr;
  if (opts) {
    status = opts->dev_status;
    if (fp8) {
      dq = opts->descale_q;
      dk = opts->descale_k;
      dv = opts->descale_v;
      if (!std::isfinite(dq) || !std::isfinite(dk) || !std::isfinite(dv) || dq <= 0.f ||
          dk <= 0.f || dv <= 0.f)
        return FA_ERR_INVALID_ARG;
    }
  }
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return FA_ERR_UNSUPPORTED;
  if (N > 0x7FFFFFFF - 2 * kCtaRows) return FA_ERR_UNSUPPORTED;
  if (causal && (N + kCtaRows - 1) / kCtaRows > 65535) return FA_ERR_UNSUPPORTED;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  if (splits > 1) {
    const size_t need = split_workspace_bytes(B, H, N, d, splits);
    if (!workspace || workspace_bytes < need) return FA_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return FA_ERR_MISALIGNED;
    o_part = static_cast<float*>(workspace);
    lse_part = o_part + static_cast<size_t>(splits) * B * H * N * d;
  }
  if (bs) {
    if (!fp8 || !bs->dq || !bs->dk || !bs->dv) return FA_ERR_INVALID_ARG;
    if (!aligned(bs->dq, 4) || !aligned(bs->dk, 4) || !aligned(bs->dv, 4))
      return FA_ERR_MISALIGNED;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || (status && !aligned(status, 4)))
    return FA_ERR_MISALIGNED;
  const double c = static_cast<double>(scale) * 1.4426950408889634 * dq * dk;
  if (!std::isfinite(c) || c > 3.0e38) return FA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float cf = static_cast<float>(c);
  int rc;
  if (dtype == FA_DTYPE_BF16) {
    rc = d == 64 ? launch_mask<64, false>(causal, q, k, v, o, lse, B, H, N, cf, 1.f, status,
                                          splits, o_part, lse_part, nullptr, s)
                 : launch_mask<128, false>(causal, q, k, v, o, lse, B, H, N, cf, 1.f, status,
                                           splits, o_part, lse_part, nullptr, s);
  } else if (dtype == FA_DTYPE_FP8_E4M3_PV16) {
    rc = d == 64 ? launch_mask<64, true, true>(causal, q, k, v, o, lse, B, H, N, cf, dv, status,
                                               splits, o_part, lse_part, bs, s)
                 : launch_mask<128, true, true>(causal, q, k, v, o, lse, B, H, N, cf, dv, status,
                                                splits, o_part, lse_part, bs, s);
  } else {
    rc = d == 64 ? launch_mask<64, true, false>(causal, q, k, v, o, lse, B, H, N, cf, dv, status,
                                                splits, o_part, lse_part, bs, s)
                 : launch_mask<128, true, false>(causal, q, k, v, o, lse, B, H, N, cf, dv,
                                                 status, splits, o_part, lse_part, bs, s);
  }
  if (rc != FA_OK || splits == 1) return rc;
  const long long rows = static_cast<long long>(B) * H * N;
  return d == 64 ? launch_combine<64>(o_part, lse_part, o, lse, splits, rows, s)
                 : launch_combine<128>(o_part, lse_part, o, lse, splits, rows, s);
}

}  // namespace
}  // namespace exattn

using namespace exattn;

extern "C" {

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int N, int d, float scale, int causal, int dtype, const fa_fwd_opts* opts,
              void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, opts, 1, nullptr, 0,
                  stream);
}

size_t fa_fwd_split_workspace_bytes(int B, int H, int N, int d, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || num_splits < 1 ||
      num_splits > kMaxSplits)
    return 0;
  return split_workspace_bytes(B, H, N, d, num_splits);
}

int fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, int dtype, int num_splits,
                 void* workspace, size_t workspace_bytes, const fa_fwd_opts* opts,
                 void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, opts, num_splits,
                  workspace, workspace_bytes, stream);
}

int fa_fwd_fp8_blockscaled(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int causal, int dtype,
                           const float* descale_q_blk, const float* descale_k_blk,
                           const float* descale_v_blk, int num_splits, void* workspace,
                           size_t workspace_bytes, int* dev_status, void* stream) {
  if (dtype != FA_DTYPE_FP8_E4M3 && dtype != FA_DTYPE_FP8_E4M3_PV16) return FA_ERR_INVALID_ARG;
  fa_fwd_opts opts;
  opts.descale_q = opts.descale_k = opts.descale_v = 1.f;
  opts.dev_status = dev_status;
  const BlockScales bs{descale_q_blk, descale_k_blk, descale_v_blk};
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, &opts, num_splits,
                  workspace, workspace_bytes, stream, &bs);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  return bwd_workspace_bytes(B, H, N);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, void* workspace, size_t workspace_bytes, int* dev_status,
           void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return FA_ERR_UNSUPPORTED;
  if ((N + kTileRows - 1) / kTileRows > 65535 || N > 0x7FFFFFFF - kTileRows)
    return FA_ERR_UNSUPPORTED;
  if (workspace_bytes < bwd_workspace_bytes(B, H, N)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 16) || (dev_status && !aligned(dev_status, 4)))
    return FA_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* delta = static_cast<float*>(workspace);
  if (d == 64)
    return causal ? launch_bwd<64, true>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, scale, delta,
                                         dev_status, s)
                  : launch_bwd<64, false>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, scale,
                                          delta, dev_status, s);
  return causal ? launch_bwd<128, true>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, scale, delta,
                                        dev_status, s)
                : launch_bwd<128, false>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, scale, delta,
                                         dev_status, s);
}

int fa_quantize_e4m3(const void* x, void* codes, float* descales, int B, int H, int N, int d,
                     const float* signs, int flags, void* stream) {
  if (!x || !codes || !descales || B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (flags & ~FA_QUANT_POW2_DESCALE) return FA_ERR_INVALID_ARG;
  const bool pow2 = (flags & FA_QUANT_POW2_DESCALE) != 0;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return FA_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(descales, 4) ||
      (signs && !aligned(signs, 16)))
    return FA_ERR_MISALIGNED;
  const int nblk = (N + kQuantRows - 1) / kQuantRows;
  const dim3 grid(static_cast<unsigned>(nblk), static_cast<unsigned>(B * H));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* cb = static_cast<uint8_t*>(codes);
  if (d == 64) {
    if (signs)
      quantize_e4m3_kernel<64, true><<<grid, kQuantThreads, 0, s>>>(xb, cb, descales, signs, N, nblk, pow2);
    else
      quantize_e4m3_kernel<64, false><<<grid, kQuantThreads, 0, s>>>(xb, cb, descales, signs, N, nblk, pow2);
  } else {
    if (signs)
      quantize_e4m3_kernel<128, true><<<grid, kQuantThreads, 0, s>>>(xb, cb, descales, signs, N, nblk, pow2);
    else
      quantize_e4m3_kernel<128, false><<<grid, kQuantThreads, 0, s>>>(xb, cb, descales, signs, N, nblk, pow2);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, int dtype, void* stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, nullptr, stream);
}

int fa_device_status(int clear, int* out) {
  if (!out) return FA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  *out = v;
  return FA_OK;
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_MISALIGNED: return "misaligned pointer";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int fa_version(void) { return 100; }

#ifdef EXATTN_TRACE
// Diagnostic builds only: point the timeline trace at a device buffer of
// 11 * 2 * kTraceMaxJ int64 and pick the CTA (blockIdx.x + gridDim.x * blockIdx.y) to record.
FA_API int fa_trace_config(long long* buf, int cta) {
  if (cudaMemcpyToSymbol(g_trace_buf, &buf, sizeof(buf)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_trace_cta, &cta, sizeof(cta)) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}
#endif

int fa_debug_exp2(const float* x, float* y, long long n, int mode, void* stream) {
  if (!x || !y || n < 0 || (mode != 0 && mode != 1)) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  exp2_probe_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      x, y, n, mode);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Key-split forward without any allocation (fa_fwd_split_noalloc).
//
// Some callers cannot allocate device memory at call time: a plug-in running inside a host that
// owns every byte of the GPU's memory and forbids libraries from allocating, or a serving loop
// that must not stall or fail on an allocation in the middle of a request.  For them the split
// partials live in one fixed, file-scope scratch array instead of a caller-provided workspace.
// The array is part of the library's device image: every GPU that loads the library holds its
// 64 MiB until the process exits, whether or not this entry point is ever called.
// ---------------------------------------------------------------------------------------------
namespace exattn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t{64} << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up with cudaGetSymbolAddress, once per
// device, while that device is current; the first call on each device does this set-up.
void* noalloc_scratch(int dev) {
  static std::atomic<void*> cache[kMaxDevices];
  void* p = cache[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) return nullptr;
  cache[dev].store(addr, std::memory_order_release);
  return addr;
}

}  // namespace
}  // namespace exattn

extern "C" {

int fa_fwd_split_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, float scale, int causal, int dtype, int num_splits,
                         const fa_fwd_opts* opts, void* stream) {
  using namespace exattn;
  if (B < 1 || H < 1 || N < 1 || num_splits < 1 || num_splits > kMaxSplits)
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  // the partials must fit in the fixed scratch; larger problems are refused, never truncated
  if (num_splits > 1 && split_workspace_bytes(B, H, N, d, num_splits) > kNoAllocScratchBytes)
    return FA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  void* scratch = noalloc_scratch(dev);
  if (!scratch) return FA_ERR_CUDA;
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, opts, num_splits, scratch,
                  kNoAllocScratchBytes, stream);
}

}  // extern "C"
