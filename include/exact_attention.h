/*
 * exact_attention.h -- C ABI of libexattn.so, the fused exact-attention forward for sm_103a.
 *
 * The operation (problem statement of "FlashAttention · InkStack", opening of "FlashAttention 1:
 * Data Movement", and the stored statistic of its section 2.1 "优化 Online Softmax"):
 *
 *     O   = softmax(scale * Q K^T + mask) V
 *     LSE = log sum_j exp(scale * q_i . k_j)     (natural log, over the keys row i may see)
 *
 * computed in one kernel launch without writing the N x N scores or probabilities anywhere:
 * Q is tiled into 128-row blocks, K/V are streamed in 128-row blocks, and each row keeps the
 * online-softmax state (running max m, running sum l, unnormalised output) on chip, merged with
 * the rescale factor alpha = e^(m_old - m_new) ("FlashAttention · InkStack", section 1.1.2).
 * The causal mask is lower-triangular with the diagonal included (key j visible to query i iff
 * j <= i); fully masked key blocks are skipped.
 *
 * Layout (all row-major, head dimension fastest, no padding between rows):
 *   q, k, v : [B, H, N, d], bf16 or fp8 e4m3fn (all three the same dtype)
 *   o       : [B, H, N, d], bf16 for both operand dtypes
 *   lse     : [B, H, N], fp32
 *
 * Ownership: every pointer is caller-owned device memory.  The library allocates no device
 * memory, frees nothing and keeps no pointer after the call returns.  The kernel runs
 * asynchronously on `stream` (a cudaStream_t, NULL = legacy default stream); the caller keeps
 * the buffers alive until the stream has passed the launch.  No call synchronises the stream.
 *
 * Errors: arguments are checked on the host before anything is launched; a failed check returns
 * a status code and launches nothing.  A launch failure returns FA_ERR_CUDA.  Inside the kernel
 * every wait is bounded in time; a wait that runs out makes the kernel stop early, free its
 * tensor memory and record FA_ERR_DEVICE_TIMEOUT in the device status word (see
 * fa_device_status / fa_fwd_opts.dev_status).  No exception crosses this interface.
 */
#ifndef EXACT_ATTENTION_H
#define EXACT_ATTENTION_H

#include <stddef.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_DTYPE_BF16 = 0,          /* q, k, v are bf16 */
  FA_DTYPE_FP8_E4M3 = 1,      /* q, k, v are fp8 e4m3fn with fp32 descales; both products are
                                 fp8 ("FlashAttention · InkStack", section 3.3): P is rounded to
                                 e4m3, up to 2^-4 relative per probability, so a row whose mass
                                 sits on a few keys carries that error on O.  With the causal
                                 mask the first 256 query rows of every head (which see at most
                                 256 keys) take the f16 P V product of FP8_E4M3_PV16, in a
                                 second, small launch on the same stream */
  FA_DTYPE_FP8_E4M3_PV16 = 2  /* as FP8_E4M3, but the P V product is f16: P rounded to f16, V
                                 widened exactly from e4m3 in shared memory (slower; S = Q K^T
                                 stays an fp8 product) */
} fa_dtype;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* null pointer, non-positive size, bad scale or dtype */
  FA_ERR_UNSUPPORTED = 2,    /* head dim not in {64, 128}, or sizes beyond the kernel's limits */
  FA_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned */
  FA_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed (no device, launch error) */
  FA_ERR_DEVICE_TIMEOUT = 5  /* a bounded wait inside the kernel ran out; outputs are invalid */
} fa_status;

/*
 * Attention forward.
 *   q, k, v : device pointers, [B, H, N, d] of `dtype` (16-byte aligned)
 *   o       : device pointer, [B, H, N, d] bf16 (16-byte aligned)
 *   lse     : device pointer, [B, H, N] fp32 (4-byte aligned)
 *   B, H, N : >= 1, with B * H <= 65535 and N < 2^31 - 512 (causal: N <= 65535 * 256)
 *   d       : head dimension, 64 or 128
 *   scale   : softmax scale applied to q . k, finite and >= 0 (usually 1/sqrt(d))
 *   causal  : 0 = no mask, nonzero = lower-triangular mask (diagonal included)
 *   dtype   : an fa_dtype; FP8_E4M3 uses descales of 1.0 here (see fa_fwd_ex)
 *   stream  : a cudaStream_t
 * Returns an fa_status.
 */
FA_API int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, int dtype, void* stream);

/*
 * Options of fa_fwd_ex.  For fp8 operands the stored values are code * descale: the scores are
 * scale * descale_q * descale_k * (q . k) and the output is descale_v * (P V) (per-tensor
 * scaling of "FlashAttention · InkStack", section 3.3.3 "Scaling").  The descales must be
 * finite and > 0; they are ignored for bf16.  `dev_status`, if not NULL, is a device int the
 * kernel sets to FA_ERR_DEVICE_TIMEOUT when a wait runs out (it never writes FA_OK: clear it
 * before the call); if NULL the library's own per-device status word is used instead.
 */
typedef struct {
  float descale_q;
  float descale_k;
  float descale_v;
  int* dev_status;
} fa_fwd_opts;

/* fa_fwd with options; `opts` may be NULL (descales 1.0, library status word). */
FA_API int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int N, int d, float scale, int causal, int dtype, const fa_fwd_opts* opts,
              void* stream);

/*
 * Key-split ("split-KV") variant of fa_fwd_ex.  The key blocks each query tile visits are
 * divided into `num_splits` contiguous ranges processed by separate CTAs (more parallelism when
 * B * H * ceil(N / 256) is small next to the GPU's SM count); each range leaves its normalised
 * output and log-sum-exp in `workspace`, and a second kernel merges the ranges with the
 * associative log-sum-exp merge ("FlashAttention · InkStack", section 2.2: independent key
 * blocks merged by an associative operation; the (m, l, U) recurrence of section 1.1.2).
 *   num_splits      : 1..16 (1 = fa_fwd_ex; workspace may then be NULL)
 *   workspace       : caller-owned device scratch, 16-byte aligned, at least
 *                     fa_fwd_split_workspace_bytes(B, H, N, d, num_splits) bytes; its contents
 *                     on entry do not matter and are undefined on return
 * Other arguments, layouts and errors as fa_fwd_ex; too small a workspace is
 * FA_ERR_INVALID_ARG.  The result equals fa_fwd_ex's up to fp32 rounding.
 */
FA_API int fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int N, int d, float scale, int causal, int dtype, int num_splits,
                        void* workspace, size_t workspace_bytes, const fa_fwd_opts* opts,
                        void* stream);

/* Workspace bytes fa_fwd_split needs: num_splits * B * H * N * (d + 1) * 4, rounded up to 256;
 * 0 for invalid arguments. */
FA_API size_t fa_fwd_split_workspace_bytes(int B, int H, int N, int d, int num_splits);

/*
 * fa_fwd_split without any allocation, for callers that cannot allocate device memory when they
 * call: a plug-in whose host owns all of the GPU's memory and forbids libraries from allocating,
 * or a serving loop that must not stall or fail on an allocation mid-request.  The paper has no
 * counterpart of this entry point; it is an interface convenience of this library.
 *
 * Instead of a caller workspace, the split partials live in a fixed 64 MiB scratch array inside
 * the library's device image (every GPU that loads the library holds it until the process
 * exits).  The caller still passes inputs and outputs.  No call allocates or frees memory.
 *   - The first call on a device looks up the scratch's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture.
 *   - Problems whose partials need more than 64 MiB, i.e.
 *     fa_fwd_split_workspace_bytes(B, H, N, d, num_splits) > 64 MiB, return FA_ERR_UNSUPPORTED
 *     and launch nothing.  num_splits == 1 needs no scratch and behaves as fa_fwd_ex.
 *   - Every call on a device shares the one array and leaves its last contents there; nothing in
 *     it needs to start at zero (every partial is written before it is read).  Calls whose
 *     kernels overlap on the GPU (concurrent streams on the same device) race on the array and
 *     give undefined results: serialise them.
 * Other arguments, layouts and errors as fa_fwd_split.
 */
FA_API int fa_fwd_split_noalloc(const void* q, const void* k, const void* v, void* o,
                                float* lse, int B, int H, int N, int d, float scale, int causal,
                                int dtype, int num_splits, const fa_fwd_opts* opts,
                                void* stream);

/*
 * fp8 forward with block scaling ("FlashAttention · InkStack", section 3.3.1 "Block
 * Quantization"; "FlashAttention 完全拆解（三）", section on block quantisation): every block of
 * 128 consecutive rows of one head of Q, K and V carries its own descale, so the stored value of
 * row i of head (b, h) is code * descale_X_blk[(b * H + h) * nblk + i / 128], nblk = ceil(N / 128).
 * Score block (i, j) is then scale * dq_i * dk_j * (q . k) and the output sum_j P_ij dv_j V_j.
 *   q, k, v           : device pointers, [B, H, N, d] e4m3fn codes (16-byte aligned)
 *   dtype             : FA_DTYPE_FP8_E4M3 or FA_DTYPE_FP8_E4M3_PV16 (precision of P V)
 *   descale_*_blk     : device pointers, [B, H, nblk] fp32 (4-byte aligned); every descale must
 *                       be finite and > 0 (fa_quantize_e4m3 writes such arrays), otherwise the
 *                       output is undefined (the kernel still runs to completion).  The value
 *                       descales enter P as dv_j / max_j dv_j: exact for powers of two, else
 *                       rounded with P (see FA_QUANT_POW2_DESCALE)
 *   num_splits, workspace, workspace_bytes : as fa_fwd_split (1 and NULL, 0 for no key split)
 *   dev_status        : as fa_fwd_opts.dev_status (NULL = the library's status word)
 * Other arguments, layouts and errors as fa_fwd_split.
 */
FA_API int fa_fwd_fp8_blockscaled(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int H, int N, int d, float scale,
                                  int causal, int dtype, const float* descale_q_blk,
                                  const float* descale_k_blk, const float* descale_v_blk,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  int* dev_status, void* stream);

/* fa_quantize_e4m3 flag: round every descale up to a power of two (recommended for V). */
#define FA_QUANT_POW2_DESCALE 1

/*
 * Block quantiser to fp8 e4m3fn, with optional incoherent processing ("FlashAttention ·
 * InkStack", sections 3.3.1 "Block Quantization", 3.3.2 "Incoherent Processing" and 3.3.3
 * "Scaling").  For every block of 128 consecutive rows of each head:
 *     X'        = X diag(signs) Had / sqrt(d)   if signs != NULL (fast Walsh-Hadamard transform;
 *                 Had is the Sylvester-Hadamard matrix), else X' = X
 *     descale   = max |X'_blk| / 448            (1 if the block is all zero); with
 *                 FA_QUANT_POW2_DESCALE, the smallest power of two >= that quotient
 *     scale     = 448 / max |X'_blk|            (1 / descale with FA_QUANT_POW2_DESCALE)
 *     code      = e4m3(X' * scale)              (round to nearest even, saturate at 448)
 * Apply the same `signs` to Q and K (QK^T is unchanged) and none to V.  Power-of-two value
 * descales let fa_fwd_fp8_blockscaled fold them into P exactly; other value descales add one
 * more e4m3 rounding of relative size up to 2^-4 to each probability.
 *   x        : device pointer, [B, H, N, d] bf16 (16-byte aligned)
 *   codes    : device pointer, [B, H, N, d] e4m3fn output (16-byte aligned)
 *   descales : device pointer, [B, H, ceil(N / 128)] fp32 output (4-byte aligned)
 *   signs    : device pointer to d fp32 values, each +1 or -1 (16-byte aligned), or NULL
 *   d        : 64 or 128; B * H <= 65535
 *   flags    : 0 or FA_QUANT_POW2_DESCALE (other bits: FA_ERR_INVALID_ARG)
 * Arithmetic is fp32 (descale and scale correctly rounded once per block).  Returns an
 * fa_status; asynchronous on `stream` like fa_fwd.
 */
FA_API int fa_quantize_e4m3(const void* x, void* codes, float* descales, int B, int H, int N,
                            int d, const float* signs, int flags, void* stream);

/*
 * Attention backward for bf16 operands ("FlashAttention · InkStack", section 1.2: dV = P^T dO,
 * dP = dO V^T, dS = P * (dP - D) with D_i = rowsum(dO_i * O_i), dQ = scale dS K,
 * dK = scale dS^T Q; P recomputed from the forward's LSE as in section 1.2.2).  Three kernel
 * launches on `stream`: D, then dK/dV, then dQ.
 *   q, k, v, o, dout : device pointers, [B, H, N, d] bf16 (16-byte aligned); o and lse are the
 *                      forward outputs for q, k, v (same scale and mask)
 *   lse              : device pointer, [B, H, N] fp32 (4-byte aligned), natural log
 *   dq, dk, dv       : device pointers, [B, H, N, d] bf16 outputs (16-byte aligned)
 *   workspace        : caller-owned device scratch of fa_bwd_workspace_bytes(B, H, N) bytes
 *                      (16-byte aligned), holds D; contents on entry do not matter
 *   dev_status       : as fa_fwd_opts.dev_status (NULL = the library's status word)
 * Sizes, scale, mask and errors as fa_fwd (d in {64, 128}); too small a workspace is
 * FA_ERR_INVALID_ARG.
 */
FA_API int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  float scale, int causal, void* workspace, size_t workspace_bytes,
                  int* dev_status, void* stream);

/* Workspace bytes fa_bwd needs: B * H * N * 4, rounded up to 256; 0 for invalid arguments. */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int N);

/*
 * Read, and if `clear` is nonzero reset to FA_OK, the library's status word on the current
 * device.  Synchronises the device first.  Writes FA_OK or FA_ERR_DEVICE_TIMEOUT to *out.
 * Returns an fa_status for the call itself.
 */
FA_API int fa_device_status(int clear, int* out);

/* A static, human-readable name for a status code. */
FA_API const char* fa_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
FA_API int fa_version(void);

/*
 * Diagnostic: evaluate the kernel's own 2^x routines on n inputs, for testing them against
 * exact exp2.  mode 0 = hardware approximation (MUFU ex2), mode 1 = the FMA polynomial
 * emulation the softmax uses for part of its columns ("FlashAttention4 精读", section 3.1.3
 * "Emulation of the exponential function").  x, y are device float arrays of n elements.
 */
FA_API int fa_debug_exp2(const float* x, float* y, long long n, int mode, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_H */
