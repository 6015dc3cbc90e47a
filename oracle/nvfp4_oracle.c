/*
 * nvfp4_oracle.c -- plain, slow CPU definition of the NVFP4 weight path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * What it defines (sources):
 *   - Weight-only quantisation: activations stay 16-bit, weights are encoded
 *     ("RL with NVFP4 + LoRA" post, tggo.me/sberlogasci/42740, section "Метод").
 *   - Each weight is an E2M1 code plus a block scale shared by its block; codes
 *     are about 90% of the file ("Scale-QLoRA", rit.work blog, format
 *     paragraph).  The page does not state the block size, scale type or grid;
 *     the NVFP4 definition used here is: 16-element blocks along a row, E4M3
 *     block scale, FP32 per-tensor scale, E2M1 grid {0,0.5,1,1.5,2,3,4,6},
 *     round-to-nearest-even, two codes per byte.
 *   - Dynamic ("max") scales recomputed from the current tensor, or frozen
 *     scales kept fixed ("Nemotron 3.5 Lightning: NVFP4 via QAD", aikraft.ru,
 *     section 03 "Dynamic vs Frozen").
 *   - Scale-only update: codes frozen, trained block scales rounded onto the
 *     target scale grid, merge writes only scale bytes ("Scale-QLoRA",
 *     paragraphs on the method and on the guarantee).
 *   - Parallel LoRA branch as in QLoRA and noise through the RMSNorm gain
 *     (equivalent to multiplicative weight noise) ("RL with NVFP4 + LoRA",
 *     section "Метод").
 *   - The layer's input gradient with the quantised weight frozen and only
 *     the LoRA factors trained (same section): dX = (dY deq(W) + s (dY B) A)
 *     diag(z), the bf16 rounding of X' taken as the identity; and the LoRA
 *     factors' gradients dB = s dY^T (X' A^T), dA = s (dY B)^T X'.
 *
 * Every encoder is a brute-force nearest search over the enumerated finite
 * grid (ties to the code whose least significant bit is 0); every GEMM is a
 * plain triple loop in double precision.  Rows are spread over threads only
 * because rows are independent; no loop is blocked, fused or reordered.
 *
 * Parity pins live in tests/ (test_oracle_*.py): codec round trips against
 * closed forms and library conversions, the grid round trip, the half-step
 * error bound, the 8/9 code share, the scale-only-update invariants, exact
 * rational brute force on tiny GEMMs and exact dyadic cases; for the input
 * gradient the exact adjoint identity <dY, Y(X)> = <dX, X> against the
 * forward, float64 autograd and exact rationals (test_oracle_dgrad.py); for
 * the LoRA gradients the forward's exact linearity in A and in B, float64
 * autograd and exact rationals (test_oracle_lora_grads.py).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_NONFINITE 1
#define ORC_BAD_SHAPE 2

/* ------------------------------------------------------------------ */
/* Scalar formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern -> float: the bf16 bits are the top half of an fp32. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* float -> bf16, round to nearest, ties to even (NaN kept quiet). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f))
        return (uint16_t)((u >> 16) | 0x40);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1; /* carry may move into the exponent: still correct RNE */
    return (uint16_t)upper;
}

/* E2M1 value of a 4-bit code: bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 * mantissa; exponent 0 is subnormal (0 or 0.5). */
double orc_e2m1_value(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (the "fn" flavour: no infinities, S.1111.111 is NaN) value of a byte:
 * bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa. */
double orc_e4m3_value(int byte)
{
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest entry of an ascending grid of non-negative magnitudes to |x|.
 * Values at or beyond the top saturate to the top (satfinite).  A tie between
 * two neighbours goes to the even code. */
static int nearest_code(double x_abs, const double *grid, int n)
{
    if (!(x_abs < grid[n - 1]))
        return n - 1;
    int best = 0;
    double bd = fabs(x_abs - grid[0]);
    for (int c = 1; c < n; c++) {
        double d = fabs(x_abs - grid[c]);
        if (d < bd || (d == bd && (c & 1) == 0)) {
            best = c;
            bd = d;
        }
    }
    return best;
}

static double g_e2m1_mag[8];
static double g_e4m3_mag[127]; /* non-negative finite codes 0x00..0x7E */
static pthread_once_t g_once = PTHREAD_ONCE_INIT;

static void build_grids(void)
{
    for (int c = 0; c < 8; c++)
        g_e2m1_mag[c] = orc_e2m1_value(c);
    for (int c = 0; c < 127; c++)
        g_e4m3_mag[c] = orc_e4m3_value(c);
}

static void grids(void) { pthread_once(&g_once, build_grids); }

/* E2M1, round to nearest even, saturating; the sign bit follows signbit(x). */
int orc_e2m1_encode(float x)
{
    grids();
    int mag = nearest_code(fabs((double)x), g_e2m1_mag, 8);
    return (signbit(x) ? 8 : 0) | mag;
}

/* E4M3 of a non-negative value, round to nearest even, saturating at 448. */
int orc_e4m3_encode_nonneg(float x)
{
    grids();
    return nearest_code((double)x, g_e4m3_mag, 127);
}

/* ------------------------------------------------------------------ */
/* Threads over rows                                                   */
/* ------------------------------------------------------------------ */

typedef void (*row_fn)(void *ctx, int64_t row);

struct row_job {
    row_fn fn;
    void *ctx;
    int64_t lo, hi;
};

static void *row_worker(void *p)
{
    struct row_job *j = (struct row_job *)p;
    for (int64_t r = j->lo; r < j->hi; r++)
        j->fn(j->ctx, r);
    return NULL;
}

static void for_rows(int64_t n, int nthreads, row_fn fn, void *ctx)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > n)
        nthreads = (int)(n > 0 ? n : 1);
    pthread_t tid[256];
    struct row_job jobs[256];
    int64_t per = (n + nthreads - 1) / nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; t++) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].lo = (int64_t)t * per;
        jobs[t].hi = jobs[t].lo + per < n ? jobs[t].lo + per : n;
        if (jobs[t].lo >= jobs[t].hi)
            break;
        if (t == 0)
            continue; /* run on the calling thread below */
        if (pthread_create(&tid[t], NULL, row_worker, &jobs[t]) != 0) {
            row_worker(&jobs[t]);
            jobs[t].fn = NULL;
        }
        started = t;
    }
    if (n > 0)
        row_worker(&jobs[0]);
    for (int t = 1; t <= started; t++)
        if (jobs[t].fn)
            pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------ */
/* Quantise                                                            */
/* ------------------------------------------------------------------ */

struct quant_ctx {
    const uint16_t *w;
    int64_t K;
    float s_t;
    uint8_t *codes, *scales;
};

static void quant_row(void *p, int64_t n)
{
    struct quant_ctx *c = (struct quant_ctx *)p;
    const uint16_t *row = c->w + n * c->K;
    int64_t nb = c->K / 16;
    for (int64_t b = 0; b < nb; b++) {
        /* block amax */
        float a_b = 0.0f;
        for (int i = 0; i < 16; i++) {
            float v = fabsf(orc_bf16_to_f32(row[b * 16 + i]));
            if (v > a_b)
                a_b = v;
        }
        /* block scale: E4M3 of a_b / (6 s_t) */
        float d = 6.0f * c->s_t;
        float e_f = (c->s_t == 0.0f) ? 0.0f : a_b / d;
        int e_b = orc_e4m3_encode_nonneg(e_f);
        c->scales[n * nb + b] = (uint8_t)e_b;
        /* effective scale S_b = dec(e_b) * s_t, one fp32 rounding */
        float S_b = (float)orc_e4m3_value(e_b) * c->s_t;
        for (int i = 0; i < 16; i++) {
            int q = 0;
            if (S_b != 0.0f) {
                float x = orc_bf16_to_f32(row[b * 16 + i]) / S_b;
                q = orc_e2m1_encode(x);
            }
            /* even element in the low nibble */
            int64_t k = b * 16 + i;
            uint8_t *byte = &c->codes[n * (c->K / 2) + k / 2];
            if ((k & 1) == 0)
                *byte = (uint8_t)((*byte & 0xF0) | q);
            else
                *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
        }
    }
}

/* W: N x K bf16 bits, row-major.  given != 0: *st_io holds the frozen tensor
 * scale; otherwise it receives s_t = amax / (6 * 448).  codes: N x K/2 bytes,
 * scales: N x K/16 bytes. */
int orc_quantize(const uint16_t *w, int64_t N, int64_t K, float *st_io, int given,
                 uint8_t *codes, uint8_t *scales, int nthreads)
{
    if (N < 0 || K < 0 || K % 16 != 0)
        return ORC_BAD_SHAPE;
    float a = 0.0f;
    for (int64_t i = 0; i < N * K; i++) {
        float v = fabsf(orc_bf16_to_f32(w[i]));
        if (!isfinite(v))
            return ORC_NONFINITE;
        if (v > a)
            a = v;
    }
    float s_t;
    if (given) {
        s_t = *st_io;
        if (!isfinite(s_t) || s_t < 0.0f)
            return ORC_NONFINITE;
    } else {
        s_t = a / 2688.0f; /* 2688 = 6 (E2M1 max) * 448 (E4M3 max) */
        *st_io = s_t;
    }
    memset(codes, 0, (size_t)(N * (K / 2)));
    struct quant_ctx c = {w, K, s_t, codes, scales};
    for_rows(N, nthreads, quant_row, &c);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Dequantise                                                          */
/* ------------------------------------------------------------------ */

static int code_at(const uint8_t *codes, int64_t K, int64_t n, int64_t k)
{
    uint8_t byte = codes[n * (K / 2) + k / 2];
    return (k & 1) ? (byte >> 4) : (byte & 0x0F);
}

/* deq = fl32( fl32(v(q) * dec(e_b)) * s_t ); the inner product is exact. */
void orc_dequantize(const uint8_t *codes, const uint8_t *scales, float s_t,
                    int64_t N, int64_t K, float *out_f32, uint16_t *out_bf16)
{
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) {
            float vd = (float)(orc_e2m1_value(code_at(codes, K, n, k)) *
                               orc_e4m3_value(scales[n * (K / 16) + k / 16]));
            float v = vd * s_t;
            if (out_f32)
                out_f32[n * K + k] = v;
            if (out_bf16)
                out_bf16[n * K + k] = orc_f32_to_bf16(v);
        }
}

/* ------------------------------------------------------------------ */
/* Scale-only update                                                   */
/* ------------------------------------------------------------------ */

/* scales[i] = E4M3_RNE(param[i] / s_t); negative parameters carry no
 * magnitude and give 0; s_t == 0 gives 0.  Codes are not an argument: the
 * update cannot touch them. */
int orc_round_scales(const float *param, float s_t, int64_t nblocks, uint8_t *scales)
{
    int st = ORC_OK;
    if (!isfinite(s_t) || s_t < 0.0f)
        return ORC_NONFINITE;
    for (int64_t i = 0; i < nblocks; i++) {
        float p = param[i];
        if (!isfinite(p)) {
            st = ORC_NONFINITE;
            scales[i] = 0;
            continue;
        }
        float e = (s_t == 0.0f || p <= 0.0f) ? 0.0f : p / s_t;
        scales[i] = (uint8_t)orc_e4m3_encode_nonneg(e);
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* W4A16 GEMM with parallel LoRA and input noise, in double            */
/* ------------------------------------------------------------------ */

/* X' = bf16( fl32(X * z) ) when z is given, else X. */
void orc_noisy_input(const uint16_t *x, const float *z, int64_t M, int64_t K, uint16_t *xp)
{
    for (int64_t m = 0; m < M; m++)
        for (int64_t k = 0; k < K; k++) {
            uint16_t b = x[m * K + k];
            if (z) {
                float p = orc_bf16_to_f32(b) * z[k];
                b = orc_f32_to_bf16(p);
            }
            xp[m * K + k] = b;
        }
}

struct gemm_ctx {
    const uint16_t *xp;
    int64_t M, K, r;
    const uint8_t *codes, *scales;
    double s_t, s;
    const double *T; /* M x r */
    const uint16_t *B;
    double *y; /* M x N */
    int64_t N;
};

static void gemm_row(void *p, int64_t n)
{
    struct gemm_ctx *c = (struct gemm_ctx *)p;
    for (int64_t m = 0; m < c->M; m++) {
        double acc = 0.0;
        for (int64_t k = 0; k < c->K; k++) {
            double d = orc_e2m1_value(code_at(c->codes, c->K, n, k)) *
                       orc_e4m3_value(c->scales[n * (c->K / 16) + k / 16]) * c->s_t;
            acc += (double)orc_bf16_to_f32(c->xp[m * c->K + k]) * d;
        }
        double lora = 0.0;
        for (int64_t j = 0; j < c->r; j++)
            lora += c->T[m * c->r + j] * (double)orc_bf16_to_f32(c->B[n * c->r + j]);
        c->y[m * c->N + n] = acc + c->s * lora;
    }
}

/* Y (M x N, double) = X' deq(W)^T + s (X' A^T) B^T.
 * x: M x K bf16; z: K floats or NULL; A: r x K bf16 or NULL; B: N x r bf16 or
 * NULL (either NULL or r == 0 drops the LoRA term). */
int orc_gemm(const uint16_t *x, int64_t M, int64_t N, int64_t K,
             const uint8_t *codes, const uint8_t *scales, float s_t,
             const uint16_t *A, const uint16_t *B, int64_t r, float s,
             const float *z, double *y, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 16 != 0 || r < 0)
        return ORC_BAD_SHAPE;
    if (!A || !B)
        r = 0;
    uint16_t *xp = (uint16_t *)malloc((size_t)(M * K + 1) * 2);
    double *T = (double *)malloc((size_t)(M * r + 1) * sizeof(double));
    if (!xp || !T) {
        free(xp);
        free(T);
        return ORC_BAD_SHAPE;
    }
    orc_noisy_input(x, z, M, K, xp);
    for (int64_t m = 0; m < M; m++)
        for (int64_t j = 0; j < r; j++) {
            double t = 0.0;
            for (int64_t k = 0; k < K; k++)
                t += (double)orc_bf16_to_f32(xp[m * K + k]) * (double)orc_bf16_to_f32(A[j * K + k]);
            T[m * r + j] = t;
        }
    struct gemm_ctx c = {xp, M, K, r, codes, scales, (double)s_t, (double)s, T, B, y, N};
    for_rows(N, nthreads, gemm_row, &c);
    free(xp);
    free(T);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Gradient of the same layer with respect to its input, in double     */
/* ------------------------------------------------------------------ */

/* Only the LoRA factors are trained ("RL with NVFP4 + LoRA", section "Метод":
 * the quantised weight is frozen, gradients flow through it to the layers
 * below).  With Y = X' Wd^T + s (X' A^T) B^T and X' = X z, the chain rule
 * gives dX = (dY Wd + s (dY B) A) diag(z); the bf16 rounding of X' is taken
 * as the identity (its derivative almost everywhere). */
struct dgrad_ctx {
    const uint16_t *dy; /* M x N */
    int64_t N, K, r;
    const uint8_t *codes, *scales;
    double s_t, s;
    const double *U; /* M x r: dY B */
    const uint16_t *A;
    const float *z;
    double *dx; /* M x K */
};

static void dgrad_row(void *p, int64_t m)
{
    struct dgrad_ctx *c = (struct dgrad_ctx *)p;
    for (int64_t k = 0; k < c->K; k++) {
        double acc = 0.0;
        for (int64_t n = 0; n < c->N; n++) {
            double d = orc_e2m1_value(code_at(c->codes, c->K, n, k)) *
                       orc_e4m3_value(c->scales[n * (c->K / 16) + k / 16]) * c->s_t;
            acc += (double)orc_bf16_to_f32(c->dy[m * c->N + n]) * d;
        }
        double lora = 0.0;
        for (int64_t j = 0; j < c->r; j++)
            lora += c->U[m * c->r + j] * (double)orc_bf16_to_f32(c->A[j * c->K + k]);
        double g = acc + c->s * lora;
        c->dx[m * c->K + k] = c->z ? g * (double)c->z[k] : g;
    }
}

/* dX (M x K, double) = (dY deq(W) + s (dY B) A) diag(z).
 * dy: M x N bf16; z: K floats or NULL (then diag(z) = I); A: r x K bf16 or
 * NULL; B: N x r bf16 or NULL (either NULL or r == 0 drops the LoRA term). */
int orc_gemm_dgrad(const uint16_t *dy, int64_t M, int64_t N, int64_t K,
                   const uint8_t *codes, const uint8_t *scales, float s_t,
                   const uint16_t *A, const uint16_t *B, int64_t r, float s,
                   const float *z, double *dx, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 16 != 0 || r < 0)
        return ORC_BAD_SHAPE;
    if (!A || !B)
        r = 0;
    double *U = (double *)malloc((size_t)(M * r + 1) * sizeof(double));
    if (!U)
        return ORC_BAD_SHAPE;
    for (int64_t m = 0; m < M; m++)
        for (int64_t j = 0; j < r; j++) {
            double u = 0.0;
            for (int64_t n = 0; n < N; n++)
                u += (double)orc_bf16_to_f32(dy[m * N + n]) * (double)orc_bf16_to_f32(B[n * r + j]);
            U[m * r + j] = u;
        }
    struct dgrad_ctx c = {dy, N, K, r, codes, scales, (double)s_t, (double)s, U, A, z, dx};
    for_rows(M, nthreads, dgrad_row, &c);
    free(U);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Gradients of the LoRA factors, in double                            */
/* ------------------------------------------------------------------ */

/* The trained parameters are A and B ("RL with NVFP4 + LoRA", section
 * "Метод").  With T = X' A^T and the LoRA term s T B^T of Y:
 *   dB = s dY^T T          (N x r),
 *   dA = s (dY B)^T X'     (r x K),
 * X' = bf16(X z) as in the forward. */
struct lgrad_ctx {
    const uint16_t *xp, *dy;
    int64_t M, N, K, r;
    double s;
    const double *T, *U; /* M x r each */
    double *da, *db;
};

static void lgrad_b_row(void *p, int64_t n)
{
    struct lgrad_ctx *c = (struct lgrad_ctx *)p;
    for (int64_t j = 0; j < c->r; j++) {
        double acc = 0.0;
        for (int64_t m = 0; m < c->M; m++)
            acc += (double)orc_bf16_to_f32(c->dy[m * c->N + n]) * c->T[m * c->r + j];
        c->db[n * c->r + j] = c->s * acc;
    }
}

static void lgrad_a_row(void *p, int64_t j)
{
    struct lgrad_ctx *c = (struct lgrad_ctx *)p;
    for (int64_t k = 0; k < c->K; k++) {
        double acc = 0.0;
        for (int64_t m = 0; m < c->M; m++)
            acc += c->U[m * c->r + j] * (double)orc_bf16_to_f32(c->xp[m * c->K + k]);
        c->da[j * c->K + k] = c->s * acc;
    }
}

/* da: r x K, db: N x r (double).  x: M x K bf16, z: K floats or NULL, dy:
 * M x N bf16, A: r x K bf16, B: N x r bf16. */
int orc_lora_grads(const uint16_t *x, const float *z, const uint16_t *dy, int64_t M, int64_t N, int64_t K,
                   const uint16_t *A, const uint16_t *B, int64_t r, float s, double *da, double *db,
                   int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || r < 1 || !A || !B)
        return ORC_BAD_SHAPE;
    uint16_t *xp = (uint16_t *)malloc((size_t)(M * K + 1) * 2);
    double *T = (double *)malloc((size_t)(M * r + 1) * sizeof(double));
    double *U = (double *)malloc((size_t)(M * r + 1) * sizeof(double));
    if (!xp || !T || !U) {
        free(xp);
        free(T);
        free(U);
        return ORC_BAD_SHAPE;
    }
    orc_noisy_input(x, z, M, K, xp);
    for (int64_t m = 0; m < M; m++)
        for (int64_t j = 0; j < r; j++) {
            double t = 0.0, u = 0.0;
            for (int64_t k = 0; k < K; k++)
                t += (double)orc_bf16_to_f32(xp[m * K + k]) * (double)orc_bf16_to_f32(A[j * K + k]);
            for (int64_t n = 0; n < N; n++)
                u += (double)orc_bf16_to_f32(dy[m * N + n]) * (double)orc_bf16_to_f32(B[n * r + j]);
            T[m * r + j] = t;
            U[m * r + j] = u;
        }
    struct lgrad_ctx c = {xp, dy, M, N, K, r, (double)s, T, U, da, db};
    for_rows(N, nthreads, lgrad_b_row, &c);
    for_rows(r, nthreads, lgrad_a_row, &c);
    free(xp);
    free(T);
    free(U);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Array forms of the scalar encoders (used to sweep the device        */
/* encoders over large input sets)                                     */
/* ------------------------------------------------------------------ */

struct enc_ctx {
    const float *x;
    uint8_t *out;
    int64_t n, per;
    int which;
};

static void enc_row(void *p, int64_t r)
{
    struct enc_ctx *c = (struct enc_ctx *)p;
    int64_t lo = r * c->per, hi = lo + c->per < c->n ? lo + c->per : c->n;
    for (int64_t i = lo; i < hi; i++)
        c->out[i] = (uint8_t)(c->which == 0 ? orc_e2m1_encode(c->x[i]) : orc_e4m3_encode_nonneg(c->x[i]));
}

/* which == 0: E2M1 code of x (sign in bit 3); which == 1: E4M3 byte of x >= 0 */
void orc_encode_array(const float *x, int64_t n, int which, uint8_t *out, int nthreads)
{
    grids();
    struct enc_ctx c = {x, out, n, 1 << 16, which};
    for_rows((n + c.per - 1) / c.per, nthreads, enc_row, &c);
}
