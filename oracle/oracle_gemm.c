/*
 * Oracle for the dense GEMM with a pointwise epilogue, D = epi(alpha * A * B).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA path is checked against.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may build, load or call it; the library
 * path never does.  It shares no code, header, table or helper with the CUDA
 * sources.
 *
 * What it computes (for every 0 <= i < M, 0 <= j < N):
 *   1. decode each operand element exactly from its storage format
 *      (bf16 / fp16 / e4m3 / e5m2 / e2m1 bit patterns, or fp32 narrowed to
 *      tf32);
 *   2. s = sum_{k=0}^{K-1} a(i,k) * b(k,j), in double, k ascending
 *      ("Matrix Multiplication", Step 3 "Looping over K": C[i,j] is the sum
 *      over k of A[i,k]*B[k,j]; accumulate wider than the inputs);
 *   3. y = alpha * s  ("Walk through GEMM", section 5 "Apply the epilogue":
 *      alpha is applied first ...);
 *   4. if ReLU: y = max(y, 0) with Julia's max semantics (... then the max
 *      with zero): NaN stays NaN, -0 becomes +0;
 *   5. D_ref[i + j*ldd] = y, as double.
 *   6. (narrow outputs) orc_round_output rounds y to the output format.
 * A batched GEMM is that definition applied to each batch entry on its own;
 * the oracle's callers step the operand pointers.
 *
 * Block-scaled products (orc_gemm_mx; "Matrix Multiplication", "Where to go
 * from here", names block-scaled FP8 and FP4 matmuls; the pages give no
 * format, so the oracle takes the OCP Microscaling one): every run of 32
 * consecutive k of a row of A, and of a column of B, shares one scale
 * X = 2^(e-127) (an 8-bit exponent code e; e = 255 is NaN), and
 *   s = sum over blocks kb of  Xa(i,kb) * Xb(kb,j) * (sum_{k in kb} a(i,k) b(k,j)),
 * each block's inner sum taken first, blocks in ascending order; steps 3-5
 * then apply as above.  Scales are stored one per row and block:
 *   Xa(i,kb) from SA[i*ldsa + kb],  Xb(kb,j) from SB[j*ldsb + kb],
 *   0 <= kb < ceil(K/32).
 * orc_gemm_nvf4 is the same sum for the other published FP4 scaling (NVFP4):
 * packed E2M1 operands, blocks of 16 consecutive k, and each scale an
 * unsigned E4M3 code (4 exponent bits with bias 7, 3 fraction bits; code 0x7F
 * is NaN; codes with the top bit set are not scales and are refused).
 *
 * Storage ("Walk through GEMM", section 2 "Bind runtime global arrays"):
 *   A logical (M,K), K-contiguous:  a(i,k) = A[i*lda + k]
 *   B logical (K,N), K-contiguous:  b(k,j) = B[k + j*ldb]
 * Elements outside k < K, i < M, j < N (stride padding) are never read.
 *
 * The multithreaded entry splits output columns j over threads; every
 * element's summation order is the same whatever the thread count.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread.
 * -ffp-contract=off keeps s += a*b as a rounded product and a rounded add
 * (no fused multiply-add), so the result is the same on every host.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* Operand storage formats understood by the oracle. */
enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_TF32 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4, ORC_E2M1 = 5 };

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double orc_decode_bf16(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int f = h & 0x7F;
    double v;
    if (e == 0xFF) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f, -126 - 7);            /* subnormal: 0.f * 2^-126 */
    } else {
        v = ldexp((double)(128 + f), e - 127 - 7); /* 1.f * 2^(e-127) */
    }
    return s ? -v : v;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_decode_fp16(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0x1F) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f, -14 - 10);
    } else {
        v = ldexp((double)(1024 + f), e - 15 - 10);
    }
    return s ? -v : v;
}

/*
 * fp32 -> tf32 narrowing ("Matrix Multiplication", Step 4 "Using the tensor
 * cores": TFloat32 keeps fp32's sign and 8-bit exponent and a 10-bit
 * fraction).  The conversion rounds the 24-bit significand to 11 bits, to
 * nearest with ties away from zero (the usual fp32->tf32 conversion), keeping
 * the exponent range; a value whose rounded magnitude exceeds the largest
 * finite tf32, (2 - 2^-10) * 2^127, becomes infinity.  Inf and NaN pass
 * through.  Works on the magnitude as an integer significand times a power of
 * two, which covers subnormals with the same rounding position.
 */
double orc_decode_tf32(uint32_t u) {
    int s = (u >> 31) & 1;
    int e = (u >> 23) & 0xFF;
    uint32_t f = u & 0x7FFFFF;
    double v;
    if (e == 0xFF) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        uint32_t sig = (e == 0) ? f : (f | 0x800000u); /* value = sig * 2^(ee-23) */
        int ee = (e == 0) ? -126 : e - 127;
        uint32_t q = sig >> 13;           /* kept: 11 (or fewer) leading bits */
        uint32_t r = sig & 0x1FFFu;       /* dropped: 13 bits */
        if (r >= 0x1000u) q += 1;         /* half or more: away from zero */
        v = ldexp((double)q, ee - 23 + 13);
        if (v > ldexp(2047.0, 127 - 10)) v = INFINITY;
    }
    return s ? -v : v;
}

/*
 * 8-bit floating point operands (the FP8 formats of the tensor core's
 * f8f6f4 kind, the step before the block-scaled matmuls of "Matrix
 * Multiplication", "Where to go from here").
 * E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; no
 *   infinities; exponent 15 with fraction 7 is NaN; largest finite 448.
 * E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits; exponent
 *   31 is infinity (fraction 0) or NaN; largest finite 57344.
 */
double orc_decode_e4m3(uint8_t h) {
    int s = (h >> 7) & 1;
    int e = (h >> 3) & 0xF;
    int f = h & 0x7;
    double v;
    if (e == 0xF && f == 0x7) v = NAN;
    else if (e == 0) v = ldexp((double)f, -6 - 3);
    else v = ldexp((double)(8 + f), e - 7 - 3);
    return s ? -v : v;
}

double orc_decode_e5m2(uint8_t h) {
    int s = (h >> 7) & 1;
    int e = (h >> 2) & 0x1F;
    int f = h & 0x3;
    double v;
    if (e == 0x1F) v = (f == 0) ? INFINITY : NAN;
    else if (e == 0) v = ldexp((double)f, -14 - 2);
    else v = ldexp((double)(4 + f), e - 15 - 2);
    return s ? -v : v;
}

/*
 * 4-bit floating point (E2M1, the FP4 of the block-scaled matmuls): 1 sign
 * bit, 2 exponent bits (bias 1), 1 fraction bit; no infinities or NaN.
 * Magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6.  Stored two per byte:
 * element 2t in the low nibble of byte t, element 2t + 1 in the high nibble.
 */
double orc_decode_e2m1(uint8_t nibble) {
    int s = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 0x3;
    int f = nibble & 0x1;
    double v = (e == 0) ? ldexp((double)f, -1) : ldexp((double)(2 + f), e - 1 - 1);
    return s ? -v : v;
}

static double decode_elem(const void *base, int64_t idx, int dtype) {
    switch (dtype) {
    case ORC_E2M1: {
        uint8_t byte = ((const uint8_t *)base)[idx >> 1];
        return orc_decode_e2m1((idx & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF));
    }
    case ORC_BF16: return orc_decode_bf16(((const uint16_t *)base)[idx]);
    case ORC_FP16: return orc_decode_fp16(((const uint16_t *)base)[idx]);
    case ORC_E4M3: return orc_decode_e4m3(((const uint8_t *)base)[idx]);
    case ORC_E5M2: return orc_decode_e5m2(((const uint8_t *)base)[idx]);
    default: {
        uint32_t u;
        memcpy(&u, (const unsigned char *)base + 4 * idx, 4);
        return orc_decode_tf32(u);
    }
    }
}

/* Julia's max(y, 0): NaN propagates; -0 and negatives give +0. */
static double relu_max(double y) {
    if (isnan(y)) return y;
    return (y > 0.0) ? y : 0.0;
}

static double epilogue(double alpha, double s, int relu) {
    double y = alpha * s;
    return relu ? relu_max(y) : y;
}

int orc_num_host_threads(void) {
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        int c = CPU_COUNT(&set);
        if (c > 0) return c;
    }
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ---------------- full product over decoded operands ---------------- */

typedef struct {
    int64_t M, N, K;
    double alpha;
    int relu;
    const double *Ad; /* decoded A, (M, K) row-major */
    const double *Bd; /* decoded B, (N, K) row-major: Bd[j*K + k] = b(k,j) */
    double *D;
    int64_t ldd;
    double *scale;    /* optional |alpha| * sum_k |a||b| */
    int64_t j0, j1;
} full_job;

static void *full_worker(void *p) {
    full_job *jb = (full_job *)p;
    for (int64_t j = jb->j0; j < jb->j1; ++j) {
        const double *bj = jb->Bd + j * jb->K;
        for (int64_t i = 0; i < jb->M; ++i) {
            const double *ai = jb->Ad + i * jb->K;
            double s = 0.0;
            for (int64_t k = 0; k < jb->K; ++k) s += ai[k] * bj[k];
            jb->D[i + j * jb->ldd] = epilogue(jb->alpha, s, jb->relu);
            if (jb->scale) {
                double t = 0.0;
                for (int64_t k = 0; k < jb->K; ++k) t += fabs(ai[k]) * fabs(bj[k]);
                jb->scale[i + j * jb->ldd] = fabs(jb->alpha) * t;
            }
        }
    }
    return NULL;
}

/*
 * D_ref (double, element (i,j) at D[i + j*ldd]) for the whole M x N output.
 * Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 */
int orc_gemm(int64_t M, int64_t N, int64_t K, double alpha,
             const void *A, int64_t lda, const void *B, int64_t ldb,
             int dtype, int relu, double *D, int64_t ldd, double *scale,
             int nthreads) {
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldd < M) return -1;
    if (dtype < ORC_BF16 || dtype > ORC_E5M2) return -1;
    if (M == 0 || N == 0) return 0;
    double *Ad = (double *)malloc(sizeof(double) * (size_t)(M * (K ? K : 1)));
    double *Bd = (double *)malloc(sizeof(double) * (size_t)(N * (K ? K : 1)));
    if (!Ad || !Bd) { free(Ad); free(Bd); return -2; }
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) Ad[i * K + k] = decode_elem(A, i * lda + k, dtype);
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k) Bd[j * K + k] = decode_elem(B, k + j * ldb, dtype);

    if (nthreads <= 0) nthreads = orc_num_host_threads();
    if (nthreads > N) nthreads = (int)N;
    full_job *jobs = (full_job *)calloc((size_t)nthreads, sizeof(full_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(Ad); free(Bd); free(jobs); free(tids); return -2; }
    for (int t = 0; t < nthreads; ++t) {
        full_job *jb = &jobs[t];
        jb->M = M; jb->N = N; jb->K = K; jb->alpha = alpha; jb->relu = relu;
        jb->Ad = Ad; jb->Bd = Bd; jb->D = D; jb->ldd = ldd; jb->scale = scale;
        jb->j0 = N * t / nthreads;
        jb->j1 = N * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, full_worker, &jobs[t]) != 0) break;
        started = t;
    }
    full_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    /* Columns whose thread could not start are done here. */
    for (int t = started + 1; t < nthreads; ++t) full_worker(&jobs[t]);
    free(jobs); free(tids); free(Ad); free(Bd);
    return 0;
}

/* ---------------- selected entries, decoded on the fly ---------------- */

typedef struct {
    int64_t K;
    double alpha;
    int relu, dtype;
    const void *A, *B;
    int64_t lda, ldb;
    const int64_t *I, *J;
    double *out, *scale;
    int64_t p0, p1;
} entry_job;

static void *entry_worker(void *p) {
    entry_job *jb = (entry_job *)p;
    for (int64_t q = jb->p0; q < jb->p1; ++q) {
        int64_t i = jb->I[q], j = jb->J[q];
        double s = 0.0, t = 0.0;
        for (int64_t k = 0; k < jb->K; ++k) {
            double a = decode_elem(jb->A, i * jb->lda + k, jb->dtype);
            double b = decode_elem(jb->B, k + j * jb->ldb, jb->dtype);
            s += a * b;
            t += fabs(a) * fabs(b);
        }
        jb->out[q] = epilogue(jb->alpha, s, jb->relu);
        if (jb->scale) jb->scale[q] = fabs(jb->alpha) * t;
    }
    return NULL;
}

/*
 * D_ref at the listed coordinates (I[q], J[q]), q < count, into out[q];
 * the same arithmetic as orc_gemm, one element at a time.  Coordinates must
 * satisfy 0 <= I < M and 0 <= J < N (checked).
 */
int orc_gemm_entries(int64_t M, int64_t N, int64_t K, double alpha,
                     const void *A, int64_t lda, const void *B, int64_t ldb,
                     int dtype, int relu, const int64_t *I, const int64_t *J,
                     int64_t count, double *out, double *scale, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || count < 0) return -1;
    if (dtype < ORC_BF16 || dtype > ORC_E5M2) return -1;
    for (int64_t q = 0; q < count; ++q)
        if (I[q] < 0 || I[q] >= M || J[q] < 0 || J[q] >= N) return -1;
    if (count == 0) return 0;
    if (nthreads <= 0) nthreads = orc_num_host_threads();
    if (nthreads > count) nthreads = (int)count;
    entry_job *jobs = (entry_job *)calloc((size_t)nthreads, sizeof(entry_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -2; }
    for (int t = 0; t < nthreads; ++t) {
        entry_job *jb = &jobs[t];
        jb->K = K; jb->alpha = alpha; jb->relu = relu; jb->dtype = dtype;
        jb->A = A; jb->B = B; jb->lda = lda; jb->ldb = ldb;
        jb->I = I; jb->J = J; jb->out = out; jb->scale = scale;
        jb->p0 = count * t / nthreads;
        jb->p1 = count * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, entry_worker, &jobs[t]) != 0) break;
        started = t;
    }
    entry_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) entry_worker(&jobs[t]);
    free(jobs); free(tids);
    return 0;
}

/*
 * Narrow output ("Matrix Multiplication", Step 4: keep the FP32 accumulator
 * and convert on the way out).  Rounds a double to a binary format with
 * `p` significand bits (implicit bit included), minimum normal exponent
 * `emin` and maximum exponent `emax`, to nearest with ties to even; values
 * beyond the largest finite number become infinity; NaN, infinities and
 * signed zeros pass through.  Below 2^emin the quantum stays 2^(emin-p+1)
 * (subnormals).
 *   bf16: p = 8,  emin = -126, emax = 127
 *   fp16: p = 11, emin = -14,  emax = 15
 */
static double round_format(double y, int p, int emin, int emax) {
    if (isnan(y) || isinf(y) || y == 0.0) return y;
    double a = fabs(y);
    int e;
    frexp(a, &e);         /* a in [2^(e-1), 2^e) */
    int ee = e - 1;
    if (ee < emin) ee = emin;
    double quantum = ldexp(1.0, ee - (p - 1));
    double q = a / quantum; /* exact: a power-of-two scaling */
    double fq = floor(q);
    double r = q - fq;
    if (r > 0.5 || (r == 0.5 && fmod(fq, 2.0) == 1.0)) fq += 1.0;
    double out = fq * quantum;
    double maxf = ldexp(2.0 - ldexp(1.0, -(p - 1)), emax);
    if (out > maxf) out = INFINITY;
    return copysign(out, y);
}

/* Output formats: 0 = fp32, 1 = bf16, 2 = fp16.  In place on y[0..n). */
void orc_round_output(double *y, int64_t n, int out_fmt) {
    for (int64_t q = 0; q < n; ++q) {
        switch (out_fmt) {
        case 0: y[q] = round_format(y[q], 24, -126, 127); break;
        case 1: y[q] = round_format(y[q], 8, -126, 127); break;
        case 2: y[q] = round_format(y[q], 11, -14, 15); break;
        default: break;
        }
    }
}

/* ---------------- block-scaled (microscaling) products ---------------- */

#define ORC_MX_BLOCK 32

/* 8-bit power-of-two scale: 2^(e-127); e = 255 is NaN. */
double orc_decode_e8m0(uint8_t e) {
    if (e == 0xFF) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/*
 * Unsigned E4M3 scale (NVFP4): code c = 0eeeemmm; e = 0 is subnormal,
 * m/8 * 2^-6; otherwise (1 + m/8) * 2^(e-7); e = 15 with m = 7 is NaN.  The
 * largest finite scale is 448, the smallest positive 2^-9.
 */
double orc_decode_ue4m3(uint8_t c) {
    const int e = (c >> 3) & 0xF, m = c & 7;
    if (c & 0x80) return NAN;              /* not a scale code (refused by orc_gemm_nvf4) */
    if (e == 15 && m == 7) return NAN;
    if (e == 0) return ldexp((double)m, -9);
    return ldexp((double)(8 + m), e - 10);
}

typedef struct {
    int64_t M, K, KB, block;
    double alpha;
    int relu;
    const double *Ad, *Bd;   /* decoded, unscaled: Ad[i*K + k], Bd[j*K + k] */
    const double *Xa, *Xb;   /* decoded scales: Xa[i*KB + kb], Xb[j*KB + kb] */
    double *D;
    int64_t ldd;
    double *scale;
    int64_t j0, j1;
} mx_job;

static void *mx_worker(void *p) {
    mx_job *jb = (mx_job *)p;
    for (int64_t j = jb->j0; j < jb->j1; ++j) {
        const double *bj = jb->Bd + j * jb->K;
        const double *xb = jb->Xb + j * jb->KB;
        for (int64_t i = 0; i < jb->M; ++i) {
            const double *ai = jb->Ad + i * jb->K;
            const double *xa = jb->Xa + i * jb->KB;
            double s = 0.0, t = 0.0;
            for (int64_t kb = 0; kb < jb->KB; ++kb) {
                int64_t k0 = kb * jb->block;
                int64_t k1 = k0 + jb->block < jb->K ? k0 + jb->block : jb->K;
                double bs = 0.0, bt = 0.0;
                for (int64_t k = k0; k < k1; ++k) {
                    bs += ai[k] * bj[k];
                    bt += fabs(ai[k]) * fabs(bj[k]);
                }
                double x = xa[kb] * xb[kb];
                s += x * bs;
                t += fabs(x) * bt;
            }
            jb->D[i + j * jb->ldd] = epilogue(jb->alpha, s, jb->relu);
            if (jb->scale) jb->scale[i + j * jb->ldd] = t * fabs(jb->alpha);
        }
    }
    return NULL;
}

/*
 * Block-scaled D_ref for the whole M x N output (see the header comment):
 * FP8 (E4M3 / E5M2) or FP4 (E2M1, packed) operands with one 8-bit exponent
 * scale per 32 k.  For E2M1, lda and ldb count elements and must be even.
 * Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 */
/*
 * The block-scaled sum over decoded operands and scales (block = k per
 * scale), output columns split over threads; frees Ad, Bd, Xa, Xb.
 */
static int bs_run(int64_t M, int64_t N, int64_t K, int64_t KB, int64_t block, double alpha,
                  int relu, double *Ad, double *Bd, double *Xa, double *Xb, double *D,
                  int64_t ldd, double *scale, int nthreads);

/* Decoded operands (K-contiguous rows of A, columns of B) and scales. */
static int bs_decode(int64_t M, int64_t N, int64_t K, int64_t KB, const void *A, int64_t lda,
                     const uint8_t *SA, int64_t ldsa, const void *B, int64_t ldb,
                     const uint8_t *SB, int64_t ldsb, int dtype, double (*scale_of)(uint8_t),
                     double **Ad, double **Bd, double **Xa, double **Xb) {
    size_t kk = (size_t)(K ? K : 1), kbb = (size_t)(KB ? KB : 1);
    *Ad = (double *)malloc(sizeof(double) * (size_t)M * kk);
    *Bd = (double *)malloc(sizeof(double) * (size_t)N * kk);
    *Xa = (double *)malloc(sizeof(double) * (size_t)M * kbb);
    *Xb = (double *)malloc(sizeof(double) * (size_t)N * kbb);
    if (!*Ad || !*Bd || !*Xa || !*Xb) {
        free(*Ad); free(*Bd); free(*Xa); free(*Xb);
        return -2;
    }
    for (int64_t i = 0; i < M; ++i) {
        const int64_t row = i * lda;
        for (int64_t k = 0; k < K; ++k) (*Ad)[i * K + k] = decode_elem(A, row + k, dtype);
        for (int64_t kb = 0; kb < KB; ++kb) (*Xa)[i * KB + kb] = scale_of(SA[i * ldsa + kb]);
    }
    for (int64_t j = 0; j < N; ++j) {
        const int64_t col = j * ldb;
        for (int64_t k = 0; k < K; ++k) (*Bd)[j * K + k] = decode_elem(B, col + k, dtype);
        for (int64_t kb = 0; kb < KB; ++kb) (*Xb)[j * KB + kb] = scale_of(SB[j * ldsb + kb]);
    }
    return 0;
}

int orc_gemm_mx(int64_t M, int64_t N, int64_t K, double alpha,
                const void *A, int64_t lda, const uint8_t *SA, int64_t ldsa,
                const void *B, int64_t ldb, const uint8_t *SB, int64_t ldsb,
                int dtype, int relu, double *D, int64_t ldd, double *scale, int nthreads) {
    int64_t KB = (K + ORC_MX_BLOCK - 1) / ORC_MX_BLOCK;
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldd < M) return -1;
    if (ldsa < KB || ldsb < KB) return -1;
    if (dtype != ORC_E4M3 && dtype != ORC_E5M2 && dtype != ORC_E2M1) return -1;
    if (dtype == ORC_E2M1 && ((lda | ldb) & 1)) return -1;  /* rows start on whole bytes */
    if (M == 0 || N == 0) return 0;
    double *Ad, *Bd, *Xa, *Xb;
    int rc = bs_decode(M, N, K, KB, A, lda, SA, ldsa, B, ldb, SB, ldsb, dtype, orc_decode_e8m0,
                       &Ad, &Bd, &Xa, &Xb);
    if (rc) return rc;
    return bs_run(M, N, K, KB, ORC_MX_BLOCK, alpha, relu, Ad, Bd, Xa, Xb, D, ldd, scale,
                  nthreads);
}

#define ORC_NV_BLOCK 16

/*
 * NVFP4 D_ref: packed E2M1 operands (lda, ldb count elements, even), one
 * unsigned E4M3 scale per 16 k.  Returns 0, -1 on bad arguments (including
 * a scale code with the top bit set), -2 on allocation failure.
 */
int orc_gemm_nvf4(int64_t M, int64_t N, int64_t K, double alpha,
                  const void *A, int64_t lda, const uint8_t *SA, int64_t ldsa,
                  const void *B, int64_t ldb, const uint8_t *SB, int64_t ldsb,
                  int relu, double *D, int64_t ldd, double *scale, int nthreads) {
    int64_t KB = (K + ORC_NV_BLOCK - 1) / ORC_NV_BLOCK;
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldd < M) return -1;
    if (ldsa < KB || ldsb < KB || ((lda | ldb) & 1)) return -1;
    if (M == 0 || N == 0) return 0;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t kb = 0; kb < KB; ++kb)
            if (SA[i * ldsa + kb] & 0x80) return -1;
    for (int64_t j = 0; j < N; ++j)
        for (int64_t kb = 0; kb < KB; ++kb)
            if (SB[j * ldsb + kb] & 0x80) return -1;
    double *Ad, *Bd, *Xa, *Xb;
    int rc = bs_decode(M, N, K, KB, A, lda, SA, ldsa, B, ldb, SB, ldsb, ORC_E2M1,
                       orc_decode_ue4m3, &Ad, &Bd, &Xa, &Xb);
    if (rc) return rc;
    return bs_run(M, N, K, KB, ORC_NV_BLOCK, alpha, relu, Ad, Bd, Xa, Xb, D, ldd, scale,
                  nthreads);
}

static int bs_run(int64_t M, int64_t N, int64_t K, int64_t KB, int64_t block, double alpha,
                  int relu, double *Ad, double *Bd, double *Xa, double *Xb, double *D,
                  int64_t ldd, double *scale, int nthreads) {
    if (nthreads <= 0) nthreads = orc_num_host_threads();
    if (nthreads > N) nthreads = (int)N;
    mx_job *jobs = (mx_job *)calloc((size_t)nthreads, sizeof(mx_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(Ad); free(Bd); free(Xa); free(Xb); free(jobs); free(tids);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        mx_job *jb = &jobs[t];
        jb->M = M; jb->K = K; jb->KB = KB; jb->block = block; jb->alpha = alpha; jb->relu = relu;
        jb->Ad = Ad; jb->Bd = Bd; jb->Xa = Xa; jb->Xb = Xb;
        jb->D = D; jb->ldd = ldd; jb->scale = scale;
        jb->j0 = N * t / nthreads;
        jb->j1 = N * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, mx_worker, &jobs[t]) != 0) break;
        started = t;
    }
    mx_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) mx_worker(&jobs[t]);
    free(jobs); free(tids); free(Ad); free(Bd); free(Xa); free(Xb);
    return 0;
}

/* ---------------- composed pointwise epilogues ---------------- */

/*
 * "Walk through GEMM", section 5 applies the epilogue as a pointwise map of
 * the accumulator, and "Tylo README" lists composed epilogues among its
 * worked consumers: elementwise functions keep each value where it is, so a
 * chain of them runs where the accumulator is.  orc_gemm_epi computes
 *   y = alpha * s  (s as in orc_gemm), then y = op_n(... op_1(y)),
 * every op in double, and reports y.  Ops (kind, a, b, bias):
 *   0 SCALE      y = a * y
 *   1 ADD        y = y + a
 *   2 RELU       y = max(y, 0)  (Julia's max: NaN stays, -0 becomes +0)
 *   3 LEAKY      y > 0 ? y : a * y   (NaN stays)
 *   4 CLAMP      min(max(y, a), b)   (NaN stays)
 *   5 SIGMOID    1 / (1 + exp(-y))
 *   6 SILU       y / (1 + exp(-y))
 *   7 GELU_TANH  y/2 * (1 + tanh(sqrt(2/pi) * (y + 0.044715 y^3)))
 *                (the tanh form of the Gaussian error linear unit,
 *                Hendrycks and Gimpel)
 *   8 BIAS_ROW   y = y + bias[i]   (one value per output row)
 *   9 BIAS_COL   y = y + bias[j]   (one value per output column)
 * The scale output is |alpha| * sum_k |a||b| as in orc_gemm (the bound of
 * the product before the ops).
 */
enum { ORC_EPI_SCALE = 0, ORC_EPI_ADD, ORC_EPI_RELU, ORC_EPI_LEAKY, ORC_EPI_CLAMP, ORC_EPI_SIGMOID,
       ORC_EPI_SILU, ORC_EPI_GELU_TANH, ORC_EPI_BIAS_ROW, ORC_EPI_BIAS_COL, ORC_EPI_KINDS };

static double apply_op(int kind, double a, double b, const float *bias, int64_t i, int64_t j,
                       double y) {
    switch (kind) {
    case ORC_EPI_SCALE: return a * y;
    case ORC_EPI_ADD: return y + a;
    case ORC_EPI_RELU: return relu_max(y);
    case ORC_EPI_LEAKY: return (isnan(y) || y > 0.0) ? y : a * y;
    case ORC_EPI_CLAMP:  /* both comparisons are false for NaN, which stays */
        if (y < a) y = a;
        if (y > b) y = b;
        return y;
    case ORC_EPI_SIGMOID: return 1.0 / (1.0 + exp(-y));
    case ORC_EPI_SILU: return y / (1.0 + exp(-y));
    case ORC_EPI_GELU_TANH:
        return 0.5 * y * (1.0 + tanh(sqrt(2.0 / M_PI) * (y + 0.044715 * y * y * y)));
    case ORC_EPI_BIAS_ROW: return y + (double)bias[i];
    case ORC_EPI_BIAS_COL: return y + (double)bias[j];
    default: return NAN;
    }
}

static int check_ops(const int *kinds, const float *const *biases, int n_ops) {
    if (n_ops < 0) return -1;
    for (int q = 0; q < n_ops; ++q) {
        if (kinds[q] < 0 || kinds[q] >= ORC_EPI_KINDS) return -1;
        if ((kinds[q] == ORC_EPI_BIAS_ROW || kinds[q] == ORC_EPI_BIAS_COL) && !biases[q]) return -1;
    }
    return 0;
}

/* The chain alone, in place on an M x N column-major array of products. */
int orc_apply_epi(int64_t M, int64_t N, const int *kinds, const double *as, const double *bs,
                  const float *const *biases, int n_ops, double *D, int64_t ldd) {
    if (check_ops(kinds, biases, n_ops) != 0 || M < 0 || N < 0 || ldd < (M > 1 ? M : 1))
        return -1;
    for (int64_t j = 0; j < N; ++j)
        for (int64_t i = 0; i < M; ++i) {
            double y = D[i + j * ldd];
            for (int q = 0; q < n_ops; ++q) y = apply_op(kinds[q], as[q], bs[q], biases[q], i, j, y);
            D[i + j * ldd] = y;
        }
    return 0;
}

int orc_gemm_epi(int64_t M, int64_t N, int64_t K, double alpha,
                 const void *A, int64_t lda, const void *B, int64_t ldb, int dtype,
                 const int *kinds, const double *as, const double *bs, const float *const *biases,
                 int n_ops, double *D, int64_t ldd, double *scale, int nthreads) {
    if (check_ops(kinds, biases, n_ops) != 0) return -1;
    /* The product alpha * s first (no ReLU), then the chain. */
    int rc = orc_gemm(M, N, K, alpha, A, lda, B, ldb, dtype, 0, D, ldd, scale, nthreads);
    if (rc != 0) return rc;
    return orc_apply_epi(M, N, kinds, as, bs, biases, n_ops, D, ldd);
}

/* Decode an array of scale codes (for the decode pins). */
void orc_decode_e8m0_array(const uint8_t *src, int64_t n, double *dst) {
    for (int64_t q = 0; q < n; ++q) dst[q] = orc_decode_e8m0(src[q]);
}

void orc_decode_ue4m3_array(const uint8_t *src, int64_t n, double *dst) {
    for (int64_t q = 0; q < n; ++q) dst[q] = orc_decode_ue4m3(src[q]);
}

/* Decode a whole array of storage elements (for the decode pins). */
void orc_decode_array(const void *src, int64_t n, int dtype, double *dst) {
    for (int64_t q = 0; q < n; ++q) dst[q] = decode_elem(src, q, dtype);
}
