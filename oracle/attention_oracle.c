/*
 * attention_oracle.c -- TEST INFRASTRUCTURE, NOT THE PRODUCT PATH.
 *
 * A plain, slow, fp64 CPU evaluation of the exact attention forward pass.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark load it.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * What it computes, for every batch b, head h and requested query row i (pages cited by title):
 *
 *   1. the row of scores  x_ij = scale * dq * dk * sum_t q_it k_jt  for j in J_i, where J_i is
 *      {0..N-1}, or {0..i} under the causal (lower-triangular, diagonal included) mask.
 *      Three-step definition S = QK^T, P = softmax(S), O = PV: "FlashAttention · InkStack",
 *      section "FlashAttention 1: Data Movement" (opening), and "FlashAttention 优化" (Moore
 *      Threads guide), section "标准实现的三步计算".  The mask sits between QK^T and softmax:
 *      "FlashAttention · InkStack", section 1.1.3 "Kernel Fusion".
 *   2. safe softmax: m_i = max_j x_ij, e_ij = exp(x_ij - m_i), l_i = sum_j e_ij,
 *      p_ij = e_ij / l_i ("FlashAttention 优化", section "online softmax 数值稳定性").
 *   3. O_i = dv * sum_j p_ij v_j, and the stored statistic LSE_i = m_i + log(l_i), natural log
 *      ("FlashAttention · InkStack", section 2.1 "优化 Online Softmax").
 *
 * Operands arrive as the raw bytes the GPU path also receives: bf16 (uint16 bit patterns) or
 * fp8 e4m3fn (uint8), decoded exactly to fp64 here from the formats' bit fields; or fp64 values
 * directly (used by the pin tests).  dq, dk, dv are per-tensor descales (1 for bf16 / fp64).
 *
 * The row of scores is materialised one query row at a time (a full fp64 S for one head at
 * N = 32768 would be 8 GiB); this is still the naive three-step algorithm, with no blocking,
 * no online rescaling and no reordering.  Rows run in parallel over POSIX threads.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no -ffast-math: IEEE semantics).
 * Compiling with -DORACLE_MUTATION=n plants one deliberate mistake; the test suite builds those
 * variants to show that its pins catch each of them.  The default build has none.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

enum { OR_BF16 = 0, OR_E4M3 = 1, OR_F64 = 2 };

/* bf16 is the upper half of an IEEE binary32: widen and reinterpret. */
double oracle_decode_bf16(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
 * exponent 1111 with mantissa 111 is NaN; exponent 0000 encodes subnormals m/8 * 2^-6. */
double oracle_decode_e4m3(uint8_t bits) {
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int m = bits & 0x7;
#if ORACLE_MUTATION == 8
    int bias = 8; /* planted: wrong exponent bias */
#else
    int bias = 7;
#endif
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - bias);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - bias);
    return sign ? -mag : mag;
}

void oracle_decode_bf16_array(const uint16_t* src, double* dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_decode_bf16(src[i]);
}

void oracle_decode_e4m3_array(const uint8_t* src, double* dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_decode_e4m3(src[i]);
}

typedef struct {
    const void *q, *k, *v;
    int dtype;
    int64_t B, H, N, d;
    double scale;
    int causal;
    double dq, dk, dv;
    /* optional per-block descales [B*H, nblk] (values = code * descale of the row's block of
     * blk_rows rows); NULL: the per-tensor dq, dk, dv apply */
    const double *dq_blk, *dk_blk, *dv_blk;
    int64_t blk_rows, nblk;
    const int64_t* rows; /* NULL: every row 0..N-1 */
    int64_t n_rows;
    double* o;   /* [B*H, n_rows, d] */
    double* lse; /* [B*H, n_rows] */
    int64_t chunk;
    int64_t n_items;
    int64_t next; /* work counter, guarded by mu */
    pthread_mutex_t mu;
    int failed;
} job_t;

/* Decode `count` consecutive operand elements starting at element `offset`. */
static void load_elems(const job_t* jb, const void* base, int64_t offset, int64_t count,
                       double* dst) {
    if (jb->dtype == OR_BF16)
        oracle_decode_bf16_array((const uint16_t*)base + offset, dst, count);
    else if (jb->dtype == OR_E4M3)
        oracle_decode_e4m3_array((const uint8_t*)base + offset, dst, count);
    else
        memcpy(dst, (const double*)base + offset, (size_t)count * sizeof(double));
}

static void run_item(job_t* jb, int64_t item, double* Kh, double* Vh, double* qrow, double* x) {
    const int64_t N = jb->N, d = jb->d;
    const int64_t chunks_per_head = (jb->n_rows + jb->chunk - 1) / jb->chunk;
    const int64_t bh = item / chunks_per_head;
    const int64_t r_begin = (item % chunks_per_head) * jb->chunk;
    int64_t r_end = r_begin + jb->chunk;
    if (r_end > jb->n_rows) r_end = jb->n_rows;
    const int64_t head_off = bh * N * d;

    /* this head's keys and values, decoded once per work item */
    load_elems(jb, jb->k, head_off, N * d, Kh);
    load_elems(jb, jb->v, head_off, N * d, Vh);
    if (jb->dk_blk)
        for (int64_t j = 0; j < N; ++j)
            for (int64_t t = 0; t < d; ++t)
                Kh[j * d + t] *= jb->dk_blk[bh * jb->nblk + j / jb->blk_rows];
    if (jb->dv_blk)
        for (int64_t j = 0; j < N; ++j)
            for (int64_t t = 0; t < d; ++t)
#if ORACLE_MUTATION == 11
                Vh[j * d + t] *= jb->dk_blk[bh * jb->nblk + j / jb->blk_rows]; /* planted */
#else
                Vh[j * d + t] *= jb->dv_blk[bh * jb->nblk + j / jb->blk_rows];
#endif

    for (int64_t r = r_begin; r < r_end; ++r) {
        const int64_t i = jb->rows ? jb->rows[r] : r;
        load_elems(jb, jb->q, head_off + i * d, d, qrow);
        if (jb->dq_blk) {
#if ORACLE_MUTATION == 10
            const double sq = jb->dq_blk[i / jb->blk_rows]; /* planted: head offset dropped */
#else
            const double sq = jb->dq_blk[bh * jb->nblk + i / jb->blk_rows];
#endif
            for (int64_t t = 0; t < d; ++t) qrow[t] *= sq;
        }

        /* the keys this row may see */
        int64_t n_keys = N;
        if (jb->causal) {
#if ORACLE_MUTATION == 2
            n_keys = i; /* planted: diagonal excluded */
#else
            n_keys = i + 1;
#endif
        }

        /* step 1: the row of scores */
        for (int64_t j = 0; j < n_keys; ++j) {
            double acc = 0.0;
            for (int64_t t = 0; t < d; ++t) acc += qrow[t] * Kh[j * d + t];
#if ORACLE_MUTATION == 1
            x[j] = acc; /* planted: scale dropped */
#else
            x[j] = jb->scale * jb->dq * jb->dk * acc;
#endif
        }

        /* step 2: safe softmax of the row */
        double m = -INFINITY;
        for (int64_t j = 0; j < n_keys; ++j)
            if (x[j] > m) m = x[j];
        double l = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
            x[j] = exp(x[j] - m);
            l += x[j];
        }
        for (int64_t j = 0; j < n_keys; ++j) {
#if ORACLE_MUTATION == 5
            (void)l; /* planted: normalisation dropped */
#else
            x[j] = x[j] / l;
#endif
        }

        /* step 3: P V and the log-sum-exp */
        double* orow = jb->o + (bh * jb->n_rows + r) * d;
        for (int64_t t = 0; t < d; ++t) orow[t] = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
#if ORACLE_MUTATION == 4
            const double* vj = Kh + j * d; /* planted: wrong operand */
#elif ORACLE_MUTATION == 6
            const double* vj = Vh + ((j + 1) % N) * d; /* planted: index shifted by one */
#else
            const double* vj = Vh + j * d;
#endif
            for (int64_t t = 0; t < d; ++t) orow[t] += x[j] * vj[t];
        }
        for (int64_t t = 0; t < d; ++t) {
#if ORACLE_MUTATION == 7
            (void)0; /* planted: value descale ignored */
#else
            orow[t] *= jb->dv;
#endif
        }
#if ORACLE_MUTATION == 3
        jb->lse[bh * jb->n_rows + r] = log(l); /* planted: max dropped from the LSE */
#elif ORACLE_MUTATION == 9
        jb->lse[bh * jb->n_rows + r] = m + log2(l); /* planted: wrong logarithm base */
#else
        jb->lse[bh * jb->n_rows + r] = m + log(l);
#endif
    }
}

static void* worker(void* arg) {
    job_t* jb = (job_t*)arg;
    const int64_t N = jb->N, d = jb->d;
    double* Kh = (double*)malloc((size_t)(N * d) * sizeof(double));
    double* Vh = (double*)malloc((size_t)(N * d) * sizeof(double));
    double* qrow = (double*)malloc((size_t)d * sizeof(double));
    double* x = (double*)malloc((size_t)N * sizeof(double));
    if (!Kh || !Vh || !qrow || !x) {
        pthread_mutex_lock(&jb->mu);
        jb->failed = 1;
        pthread_mutex_unlock(&jb->mu);
    } else {
        for (;;) {
            pthread_mutex_lock(&jb->mu);
            int64_t item = jb->next++;
            pthread_mutex_unlock(&jb->mu);
            if (item >= jb->n_items) break;
            run_item(jb, item, Kh, Vh, qrow, x);
        }
    }
    free(Kh);
    free(Vh);
    free(qrow);
    free(x);
    return NULL;
}

static int run_job(job_t* jb, int nthreads) {
    jb->chunk = 64;
    jb->n_items = jb->B * jb->H * ((jb->n_rows + jb->chunk - 1) / jb->chunk);
    pthread_mutex_init(&jb->mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > jb->n_items) nthreads = (int)jb->n_items;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -2;
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, jb) != 0) break;
        ++started;
    }
    worker(jb);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&jb->mu);
    return jb->failed ? -2 : 0;
}

static int check_common(const void* q, const void* k, const void* v, int dtype, int64_t B,
                        int64_t H, int64_t N, int64_t d, const int64_t* rows, int64_t* n_rows,
                        const double* o, const double* lse) {
    if (!q || !k || !v || !o || !lse) return -1;
    if (B < 1 || H < 1 || N < 1 || d < 1) return -1;
    if (dtype != OR_BF16 && dtype != OR_E4M3 && dtype != OR_F64) return -1;
    if (!rows) *n_rows = N;
    if (*n_rows < 1) return -1;
    if (rows)
        for (int64_t r = 0; r < *n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= N) return -1;
    return 0;
}

/*
 * Evaluate O [B, H, n_rows, d] and LSE [B, H, n_rows] in fp64.
 *   q, k, v : [B, H, N, d] row-major operands (bf16 bits, e4m3 bits or fp64, per `dtype`)
 *   rows    : the query rows to evaluate (each in [0, N)), or NULL for all N rows
 * Returns 0 on success, -1 on bad arguments, -2 if memory ran out.
 */
int oracle_attention_fwd(const void* q, const void* k, const void* v, int dtype, int64_t B,
                         int64_t H, int64_t N, int64_t d, double scale, int causal,
                         double descale_q, double descale_k, double descale_v,
                         const int64_t* rows, int64_t n_rows, double* o, double* lse,
                         int nthreads) {
    if (check_common(q, k, v, dtype, B, H, N, d, rows, &n_rows, o, lse)) return -1;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q;
    jb.k = k;
    jb.v = v;
    jb.dtype = dtype;
    jb.B = B;
    jb.H = H;
    jb.N = N;
    jb.d = d;
    jb.scale = scale;
    jb.causal = causal;
    jb.dq = descale_q;
    jb.dk = descale_k;
    jb.dv = descale_v;
    jb.rows = rows;
    jb.n_rows = n_rows;
    jb.o = o;
    jb.lse = lse;
    return run_job(&jb, nthreads);
}

/*
 * Same evaluation with per-block descales: element (b, h, i, t) of Q has the value
 * code * dq_blk[(b*H + h) * nblk + i / blk_rows], likewise K and V, nblk = ceil(N / blk_rows)
 * (block quantisation, "FlashAttention · InkStack" section 3.3.1 and "FlashAttention 完全拆解
 * （三）", block quantisation: each tile carries its own scale).
 */
int oracle_attention_fwd_blockscaled(const void* q, const void* k, const void* v, int dtype,
                                     int64_t B, int64_t H, int64_t N, int64_t d, double scale,
                                     int causal, const double* dq_blk, const double* dk_blk,
                                     const double* dv_blk, int64_t blk_rows,
                                     const int64_t* rows, int64_t n_rows, double* o,
                                     double* lse, int nthreads) {
    if (check_common(q, k, v, dtype, B, H, N, d, rows, &n_rows, o, lse)) return -1;
    if (!dq_blk || !dk_blk || !dv_blk || blk_rows < 1) return -1;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q;
    jb.k = k;
    jb.v = v;
    jb.dtype = dtype;
    jb.B = B;
    jb.H = H;
    jb.N = N;
    jb.d = d;
    jb.scale = scale;
    jb.causal = causal;
    jb.dq = jb.dk = jb.dv = 1.0;
    jb.dq_blk = dq_blk;
    jb.dk_blk = dk_blk;
    jb.dv_blk = dv_blk;
    jb.blk_rows = blk_rows;
    jb.nblk = (N + blk_rows - 1) / blk_rows;
    jb.rows = rows;
    jb.n_rows = n_rows;
    jb.o = o;
    jb.lse = lse;
    return run_job(&jb, nthreads);
}

/*
 * Backward pass, in fp64 on the decoded operands ("FlashAttention · InkStack", section 1.2.1,
 * the gradients of ordinary attention).  For every batch b, head h and query row i, with the
 * visible keys J_i of the forward pass and L = sum_i dO_i . O_i as the loss whose gradient is taken
 * (dO given):
 *   P_ij = softmax_j(scale * q_i . k_j)                  (safe softmax, as the forward)
 *   O_i  = sum_j P_ij v_j,   LSE_i = m_i + log l_i
 *   D_i  = dO_i . O_i                                     (equal to sum_j P_ij dP_ij)
 *   dP_ij = dO_i . v_j,      dS_ij = P_ij (dP_ij - D_i)
 *   dV_j += P_ij dO_i,       dQ_i = scale sum_j dS_ij k_j,   dK_j += scale dS_ij q_i
 * One work item is one head; its rows run in order, accumulating dK and dV.
 */
typedef struct {
    const void *q, *k, *v, *dout;
    int dtype;
    int64_t B, H, N, d;
    double scale;
    int causal;
    double *dq, *dk, *dv;     /* [B*H, N, d] */
    double *o, *lse, *delta;  /* [B*H, N, d], [B*H, N], [B*H, N] */
    int64_t next;
    pthread_mutex_t mu;
    int failed;
} bwd_job_t;

static void bwd_head(bwd_job_t* jb, int64_t bh, double* Q, double* K, double* V, double* dO,
                     double* p, double* dp) {
    job_t dec; /* only the decoding fields are used */
    memset(&dec, 0, sizeof dec);
    dec.dtype = jb->dtype;
    const int64_t N = jb->N, d = jb->d, off = bh * N * d;
    load_elems(&dec, jb->q, off, N * d, Q);
    load_elems(&dec, jb->k, off, N * d, K);
    load_elems(&dec, jb->v, off, N * d, V);
    load_elems(&dec, jb->dout, off, N * d, dO);
    double* dq = jb->dq + off;
    double* dk = jb->dk + off;
    double* dv = jb->dv + off;
    for (int64_t t = 0; t < N * d; ++t) dk[t] = dv[t] = 0.0;
    for (int64_t i = 0; i < N; ++i) {
        const double* qi = Q + i * d;
        const double* doi = dO + i * d;
        const int64_t nk = jb->causal ? i + 1 : N;
        /* forward recomputation of row i */
        double m = -INFINITY;
        for (int64_t j = 0; j < nk; ++j) {
            double acc = 0.0;
            for (int64_t t = 0; t < d; ++t) acc += qi[t] * K[j * d + t];
            p[j] = jb->scale * acc;
            if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        for (int64_t j = 0; j < nk; ++j) p[j] /= l;
        double* oi = jb->o + (bh * N + i) * d;
        for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
        for (int64_t j = 0; j < nk; ++j)
            for (int64_t t = 0; t < d; ++t) oi[t] += p[j] * V[j * d + t];
        jb->lse[bh * N + i] = m + log(l);
        double D = 0.0;
#if ORACLE_MUTATION == 13
        (void)oi; /* planted: D_i dropped */
#else
        for (int64_t t = 0; t < d; ++t) D += doi[t] * oi[t];
#endif
        jb->delta[bh * N + i] = D;
        /* dP, dS and the three gradients */
        for (int64_t j = 0; j < nk; ++j) {
            double acc = 0.0;
            for (int64_t t = 0; t < d; ++t) acc += doi[t] * V[j * d + t];
            dp[j] = acc;
        }
        double* dqi = dq + i * d;
        for (int64_t t = 0; t < d; ++t) dqi[t] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
#if ORACLE_MUTATION == 14
            const double ds = dp[j] - D; /* planted: P factor dropped */
#else
            const double ds = p[j] * (dp[j] - D);
#endif
            for (int64_t t = 0; t < d; ++t) {
                dqi[t] += jb->scale * ds * K[j * d + t];
#if ORACLE_MUTATION == 12
                dk[j * d + t] += ds * qi[t]; /* planted: scale dropped from dK */
#else
                dk[j * d + t] += jb->scale * ds * qi[t];
#endif
#if ORACLE_MUTATION == 15
                dv[j * d + t] += ds * doi[t]; /* planted: dS in place of P */
#else
                dv[j * d + t] += p[j] * doi[t];
#endif
            }
        }
    }
}

static void* bwd_worker(void* arg) {
    bwd_job_t* jb = (bwd_job_t*)arg;
    const int64_t N = jb->N, d = jb->d;
    double* buf = (double*)malloc((size_t)(4 * N * d + 2 * N) * sizeof(double));
    if (!buf) {
        pthread_mutex_lock(&jb->mu);
        jb->failed = 1;
        pthread_mutex_unlock(&jb->mu);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&jb->mu);
        int64_t bh = jb->next++;
        pthread_mutex_unlock(&jb->mu);
        if (bh >= jb->B * jb->H) break;
        bwd_head(jb, bh, buf, buf + N * d, buf + 2 * N * d, buf + 3 * N * d, buf + 4 * N * d,
                 buf + 4 * N * d + N);
    }
    free(buf);
    return NULL;
}

/*
 * Gradients dq, dk, dv [B, H, N, d] of L = sum(O * dO) for attention over q, k, v [B, H, N, d]
 * (dtype as oracle_attention_fwd: bf16 bits or fp64; fp8 is not a backward operand type), plus
 * the recomputed o [B, H, N, d], lse [B, H, N] and delta D [B, H, N].  Returns 0, -1 on bad
 * arguments, -2 if memory ran out.
 */
int oracle_attention_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype,
                         int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                         double* dq, double* dk, double* dv, double* o, double* lse,
                         double* delta, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || !o || !lse || !delta) return -1;
    if (B < 1 || H < 1 || N < 1 || d < 1) return -1;
    if (dtype != OR_BF16 && dtype != OR_F64) return -1;
    bwd_job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q;
    jb.k = k;
    jb.v = v;
    jb.dout = dout;
    jb.dtype = dtype;
    jb.B = B;
    jb.H = H;
    jb.N = N;
    jb.d = d;
    jb.scale = scale;
    jb.causal = causal;
    jb.dq = dq;
    jb.dk = dk;
    jb.dv = dv;
    jb.o = o;
    jb.lse = lse;
    jb.delta = delta;
    pthread_mutex_init(&jb.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B * H) nthreads = (int)(B * H);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -2;
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, bwd_worker, &jb) != 0) break;
        ++started;
    }
    bwd_worker(&jb);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&jb.mu);
    return jb.failed ? -2 : 0;
}

int oracle_mutation_id(void) { return ORACLE_MUTATION; }
