/*
 * oracle.c -- slow, plain fp64 CPU oracle for the fused GEMM + epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link
 * or call this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no source with the CUDA library.
 *
 * What it computes (for every requested output row i and every column j < N):
 *
 *   s[i,j] = sum_{k=0}^{K-1} A[i,k] * B[k,j]           in fp64, k ascending,
 *                                                     s = 0 when K = 0
 *
 *   bias+ReLU  out[i,j] = RNE( max(0, s[i,j] + bias[j]) )
 *       "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", the defining
 *       equation and the note under it: the bias is per column, broadcast over
 *       rows, and added once after the K loop.  "Epilogue concept", "Where the
 *       accumulator is finally correct": the epilogue runs only on the complete
 *       sum.
 *
 *   addmm + gate  X = s[i,j] + bias[j];  out[i,j] = RNE( X + X * Y[i,j] )
 *       "Optimizing GEMM + Activation on CDNA4 with TLX", "The GLU Block".
 *       X is never rounded before the gate: the result is rounded once.
 *
 *   residual  out[i,j] = RNE( max(0, s[i,j] + bias[j] + R[i,j]) )
 *       "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", "Variants": a same-shape residual
 *       tile is loaded after the K loop and added to the accumulator before the activation.
 *       The bias is added first, then R (fp64, so the order only matters at the last bit of a
 *       sum that is rounded once anyway).
 *
 *   quantized  out[i,j] = RNE_e4m3( clamp(scale * max(0, s[i,j] + bias[j]), -448, 448) )
 *       "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", "Variants": matmul + quantized
 *       output -- a scale and a clamp applied to the (biased, activated) accumulator, then the
 *       cast to fp8 before the store.  e4m3 ("fn": no infinities, largest finite 448) is
 *       written here from its definition: 1 sign, 4 exponent (bias 7) and 3 fraction bits.
 *
 *   linear  out[i,j] = RNE( s[i,j] + bias[j] )  (no activation; used only to
 *       pin the reduction against a library matmul and to check the unfused
 *       chain's intermediate).
 *
 * Rounding point: "I3. Fuse a GEMM epilogue and change tile scheduling",
 * "Why the baseline uses FP32": the correctness reference is an fp64
 * GEMM + bias + activation rounded once at the end.  RNE is
 * round-to-nearest-even, written here from the IEEE-754 binary16 definition and
 * the bfloat16 definition (the upper half of binary32), straight from double
 * (no double -> float -> 16-bit double rounding), with subnormals and overflow
 * to infinity.
 *
 * K = 0: "I3 ...", "Implement in stages", stage 2: the zero accumulator still
 * goes through the epilogue, so bias+ReLU gives ReLU(bias) on every row; the
 * gate gives bias + bias * Y (the same reading applied to the gate).
 *
 * ReLU of a NaN is not defined by the pages; inputs are finite.  The clamp is
 * written (v > 0) ? v : +0.
 *
 * Loop order: rows are independent; within a row the sum for every column is
 * accumulated with k ascending, exactly as in the definition above (the loop
 * over k is outside the loop over j only so that B is read row by row; no
 * element's sum is split, blocked or reordered).  Products of two 16-bit
 * floats are exact in fp64, so a fused or unfused multiply-add gives the
 * same value.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F16 = 1, ORC_BF16 = 2, ORC_F32 = 3, ORC_E4M3 = 4 };
enum { ORC_EPI_RELU = 0, ORC_EPI_GATE = 1, ORC_EPI_LINEAR = 2, ORC_EPI_RESIDUAL = 3,
       ORC_EPI_QUANT = 4 };

/*
 * Deliberate mistakes, selectable only to show that the tests' pins catch
 * them (negative controls).  ORC_OK is the oracle proper.  Each one is a
 * pitfall the pages name or a plausible slip:
 *   RELU_FIRST    ReLU(AB) + bias          ("Pitfalls": wrong operation order)
 *   BIAS_ROW      bias[i] instead of bias[j] ("Pitfalls": wrong broadcast)
 *   BIAS_IN_SUM   bias added on every K step ("Epilogue concept", "Things that break")
 *   DROP_GEMM     the sum left out (bias-only output)
 *   TRANSPOSE_B   B read as if it were N x K
 *   DROP_LAST_K   the last k term left out
 *   GATE_SIGN     X - X*Y instead of X + X*Y
 *   RESID_AFTER   ReLU(AB + bias) + R: the residual added after the activation
 *   SCALE_FIRST   quantized output with the scale applied before the bias: ReLU(scale*AB + bias)
 */
enum { ORC_OK = 0, ORC_MUT_RELU_FIRST = 1, ORC_MUT_BIAS_ROW = 2, ORC_MUT_BIAS_IN_SUM = 3,
       ORC_MUT_DROP_GEMM = 4, ORC_MUT_TRANSPOSE_B = 5, ORC_MUT_DROP_LAST_K = 6,
       ORC_MUT_GATE_SIGN = 7, ORC_MUT_RESID_AFTER = 8, ORC_MUT_SCALE_FIRST = 9 };

/* ---- decoding (definitions of the formats) ---------------------------- */

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);                 /* subnormal / zero */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);  /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
static double decode_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -133);                /* subnormal / zero */
    else if (expo == 255)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + frac), expo - 134);  /* (1.f) * 2^(e-127) */
    return sign ? -v : v;
}

/* fp8 e4m3 ("fn"): 1 sign, 4 exponent (bias 7), 3 fraction bits; S.1111.111 is NaN, no inf. */
static double decode_e4m3(uint8_t h)
{
    int sign = (h >> 7) & 1;
    int expo = (h >> 3) & 0xf;
    int frac = h & 0x7;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -9);                  /* subnormal / zero */
    else if (expo == 15 && frac == 7)
        v = NAN;
    else
        v = ldexp((double)(8 + frac), expo - 10);     /* (1.f) * 2^(e-7) */
    return sign ? -v : v;
}

static double decode(const void *p, int64_t idx, int type)
{
    switch (type) {
    case ORC_F16: return decode_f16(((const uint16_t *)p)[idx]);
    case ORC_BF16: return decode_bf16(((const uint16_t *)p)[idx]);
    case ORC_E4M3: return decode_e4m3(((const uint8_t *)p)[idx]);
    default: return (double)((const float *)p)[idx];
    }
}

/* ---- rounding (round to nearest, ties to even) ------------------------ */

/*
 * Round x to the nearest number with `p` significand bits (implicit bit
 * included), smallest normal 2^emin, largest binade 2^emax; ties go to the
 * even significand.  Values that round to 2^(emax+1) or beyond become inf.
 */
static double round_to_format(double x, int p, int emin, int emax)
{
    if (x == 0.0 || isnan(x) || isinf(x))
        return x;
    double ax = fabs(x);
    int e;
    (void)frexp(ax, &e);         /* ax = f * 2^e, f in [0.5, 1) */
    int lead = e - 1;            /* weight of the leading bit: 2^lead */
    if (lead < emin)
        lead = emin;             /* below the normal range the spacing is fixed */
    double q = ldexp(1.0, lead - (p - 1));   /* spacing of the format here */
    double r = nearbyint(ax / q) * q;        /* ax/q is exact; ties-to-even */
    if (r >= ldexp(1.0, emax + 1))
        r = INFINITY;
    return copysign(r, x);
}

static uint16_t encode_f16(double x)
{
    if (isnan(x))
        return 0x7e00;
    double r = round_to_format(x, 11, -14, 15);
    uint16_t s = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isinf(a))
        return s | 0x7c00;
    if (a < ldexp(1.0, -14))                       /* subnormal or zero */
        return s | (uint16_t)(a / ldexp(1.0, -24));
    int e;
    double f = frexp(a, &e);                       /* a = f * 2^e */
    uint16_t biased = (uint16_t)(e - 1 + 15);
    uint16_t frac = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
    return s | (uint16_t)(biased << 10) | frac;
}

static uint16_t encode_bf16(double x)
{
    if (isnan(x))
        return 0x7fc0;
    double r = round_to_format(x, 8, -126, 127);
    uint16_t s = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isinf(a))
        return s | 0x7f80;
    if (a < ldexp(1.0, -126))
        return s | (uint16_t)(a / ldexp(1.0, -133));
    int e;
    double f = frexp(a, &e);
    uint16_t biased = (uint16_t)(e - 1 + 127);
    uint16_t frac = (uint16_t)((f * 2.0 - 1.0) * 128.0);
    return s | (uint16_t)(biased << 7) | frac;
}

/* RNE to e4m3; magnitudes that round beyond 448 saturate to 448 (satfinite). */
static uint8_t encode_e4m3(double x)
{
    if (isnan(x))
        return 0x7f;
    double r = round_to_format(x, 4, -6, 8);
    uint8_t s = signbit(r) ? 0x80 : 0;
    double a = fabs(r);
    if (isinf(a) || a > 448.0)
        return s | 0x7e;
    if (a < ldexp(1.0, -6))                        /* subnormal or zero */
        return s | (uint8_t)(a / ldexp(1.0, -9));
    int e;
    double f = frexp(a, &e);
    uint8_t biased = (uint8_t)(e - 1 + 7);
    uint8_t frac = (uint8_t)((f * 2.0 - 1.0) * 8.0);
    return s | (uint8_t)(biased << 3) | frac;
}

static void store(void *p, int64_t idx, int type, double v)
{
    switch (type) {
    case ORC_F16: ((uint16_t *)p)[idx] = encode_f16(v); break;
    case ORC_BF16: ((uint16_t *)p)[idx] = encode_bf16(v); break;
    case ORC_E4M3: ((uint8_t *)p)[idx] = encode_e4m3(v); break;
    default: ((float *)p)[idx] = (float)v; break;   /* C conversion: RNE */
    }
}

/* Exported so the tests can pin the encoders against library conversions. */
void orc_encode(const double *x, void *out, int64_t n, int type)
{
    for (int64_t i = 0; i < n; ++i)
        store(out, i, type, x[i]);
}

void orc_decode(const void *p, double *out, int64_t n, int type)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = decode(p, i, type);
}

/* ---- the epilogue ------------------------------------------------------ */

static double epilogue(int epi, double s, double bias_j, double y, int mutant, double scale)
{
    if (mutant == ORC_MUT_RELU_FIRST && epi == ORC_EPI_RELU)
        return ((s > 0.0) ? s : 0.0) + bias_j;
    double v = s + bias_j;                        /* bias once, after the sum */
    switch (epi) {
    case ORC_EPI_RELU: return (v > 0.0) ? v : 0.0;   /* max(0, v) */
    case ORC_EPI_GATE:
        if (mutant == ORC_MUT_GATE_SIGN)
            return v - v * y;
        return v + v * y;                            /* X + X * Y */
    case ORC_EPI_RESIDUAL:
        if (mutant == ORC_MUT_RESID_AFTER)
            return ((v > 0.0) ? v : 0.0) + y;
        v = v + y;                                   /* + R[i,j] before the activation */
        return (v > 0.0) ? v : 0.0;
    case ORC_EPI_QUANT:
        if (mutant == ORC_MUT_SCALE_FIRST) {
            v = scale * s + bias_j;
            v = (v > 0.0) ? v : 0.0;
        } else {
            v = (v > 0.0) ? v : 0.0;                 /* activation */
            v = scale * v;                           /* scale */
        }
        if (v > 448.0) v = 448.0;                    /* clamp to the fp8 range */
        if (v < -448.0) v = -448.0;
        return v;                                    /* the cast happens at the store */
    default: return v;                               /* linear */
    }
}

/* ---- the row worker ---------------------------------------------------- */

typedef struct {
    const void *A, *bias, *Y;
    const double *Bd;        /* B decoded to fp64, K x N row-major */
    void *out;               /* nrows x N, out_type */
    double *ref;             /* nrows x N, unrounded epilogue value, or NULL */
    double *absdot;          /* nrows x N, sum_k |A[i,k] B[k,j]|, or NULL */
    const int64_t *rows;     /* row indices into A / Y, or NULL = 0..nrows-1 */
    int64_t N, K;
    int ab_type, bias_type, out_type, y_type, epi, mutant;
    double scale;            /* quantized epilogue only */
    int64_t r_begin, r_end;  /* this worker's slice of the row list */
} work_t;

static void *row_worker(void *arg)
{
    work_t *w = (work_t *)arg;
    const int64_t N = w->N, K = w->K;
    double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *sa = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int64_t r = w->r_begin; r < w->r_end; ++r) {
        const int64_t i = w->rows ? w->rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            s[j] = 0.0;
            sa[j] = 0.0;
        }
        const int mut = w->mutant;
        const int64_t k_end = (mut == ORC_MUT_DROP_LAST_K && K > 0) ? K - 1 : K;
        for (int64_t k = 0; k < k_end && mut != ORC_MUT_DROP_GEMM; ++k) {
            const double a = decode(w->A, i * K + k, w->ab_type);
            for (int64_t j = 0; j < N; ++j) {
                const double bkj = (mut == ORC_MUT_TRANSPOSE_B) ? w->Bd[(j * K + k) % (K * N)]
                                                                : w->Bd[k * N + j];
                double p = a * bkj;                 /* exact for 16-bit inputs */
                if (mut == ORC_MUT_BIAS_IN_SUM)
                    p += decode(w->bias, j, w->bias_type);
                s[j] += p;
                sa[j] += fabs(p);
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            const double b = decode(w->bias, (mut == ORC_MUT_BIAS_ROW) ? i % N : j, w->bias_type);
            const double y = (w->epi == ORC_EPI_GATE || w->epi == ORC_EPI_RESIDUAL)
                                 ? decode(w->Y, i * N + j, w->y_type) : 0.0;
            const double v = epilogue(w->epi, (mut == ORC_MUT_BIAS_IN_SUM) ? s[j] - b : s[j], b, y,
                                      mut, w->scale);
            store(w->out, r * N + j, w->out_type, v);
            if (w->ref)
                w->ref[r * N + j] = v;
            if (w->absdot)
                w->absdot[r * N + j] = sa[j];
        }
    }
    free(s);
    free(sa);
    return NULL;
}

/*
 * orc_gemm_epilogue: compute `nrows` output rows.
 *   A      M x K row-major (ab_type), may be NULL when K == 0
 *   B      K x N row-major (ab_type), may be NULL when K == 0
 *   bias   N (bias_type)
 *   Y      M x N row-major (y_type): the gate's Y, or the residual R
 *   rows   nrows row indices, or NULL for rows 0..nrows-1
 *   out    nrows x N (out_type): the rounded result for each listed row
 *   ref    nrows x N fp64: the value before the final rounding (may be NULL)
 *   absdot nrows x N fp64: sum_k |A[i,k] B[k,j]| (may be NULL)
 *   mutant ORC_OK for the oracle; any other value selects a negative control
 *   scale  the quantized epilogue's scale (ignored otherwise)
 * Returns the number of threads used, or -1 on a bad argument.
 */
int orc_gemm_epilogue(const void *A, const void *B, const void *bias, const void *Y,
                      void *out, double *ref, double *absdot,
                      int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                      int ab_type, int bias_type, int out_type, int y_type, int epi,
                      int mutant, double scale, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || nthreads < 1)
        return -1;
    if (nrows == 0 || N == 0)
        return 1;
    double *Bd = (double *)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    if (!Bd)
        return -1;
    for (int64_t t = 0; t < K * N; ++t)
        Bd[t] = decode(B, t, ab_type);

    if (nthreads > nrows)
        nthreads = (int)nrows;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    work_t *w = (work_t *)malloc(sizeof(work_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        w[t] = (work_t){A, bias, Y, Bd, out, ref, absdot, rows, N, K,
                        ab_type, bias_type, out_type, y_type, epi, mutant, scale,
                        nrows * t / nthreads, nrows * (t + 1) / nthreads};
        pthread_create(&th[t], NULL, row_worker, &w[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    free(th);
    free(w);
    free(Bd);
    return nthreads;
}
