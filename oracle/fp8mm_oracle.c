/*
 * fp8mm_oracle.c -- plain CPU oracle for the FP8 scaled matrix multiply.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header, table or constant with the CUDA
 * library (fp8_scaled_gemm_gb300/csrc).
 *
 * What it computes (one output element, i < M, j < N):
 *
 *   dot_ij = sum_k dec(A[i,k]) * dec(Bt[j,k])                      exact in fp64
 *   S_ij   = s_a * s_b           (per-tensor)   or s_a[i] * s_b[j]  (row-wise)
 *   ref_ij = dot_ij * S_ij + bias[j]            (bias optional)     in fp64
 *   out_ij = bf16_rne(ref_ij)                   one rounding, fp64 -> bf16
 *            (or fp16 / fp32 RNE, or e4m3 RNE with saturation, for the other
 *            output types)
 *
 * Sources:
 *  - the product with scales applied after an fp32-or-better accumulation and
 *    then a cast to the output type: gist "matmul_fp8.py" (FP8 Matmul),
 *    `matmul_fp8_kernel`, the block that multiplies the accumulator by
 *    `scale = scale_a[:, None] * scale_b[None, :]` (row-wise) or
 *    `scale_a * scale_b` (per-tensor) and casts to `out_ptr`'s dtype;
 *  - row-wise scale shapes (x's scale has length M, y's has length N, TN only):
 *    PyTorch PR #125204 "fp8 row-scaling kernel for scaled_mm", Summary;
 *  - B passed column-major (TN): gist "matmul_fp8.py", `benchmark()`, the
 *    `b.to(dtype).t().contiguous().t()` step, so the oracle reads B as the
 *    row-major matrix Bt[N,K];
 *  - the bias epilogue: PyTorch PR #142045, Summary ("Limitations": scaled_mm
 *    with bias values);
 *  - the element type: torch.float8_e4m3fn / tl.float8e4nv, largest finite
 *    value 448 (`torch.finfo(dtype).max`): gist "matmul_fp8.py", the dtype
 *    map and `benchmark()`.
 *
 * Why fp64 is exact for the dot product: every e4m3fn value is an integer
 * multiple of 2^-9 with magnitude <= 448, so each product is a multiple of
 * 2^-18 with magnitude < 2^17.62; for K <= 2^14 every partial sum stays below
 * 2^31.7 on the 2^-18 grid, i.e. needs at most 50 significand bits (< 53).
 * The same holds for the sum of |products| used by the parity tolerance.
 *
 * e4m3fn encoding (OCP FP8 E4M3, "fn" = finite + NaN): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * m * 2^-9; exponent 15 with mantissa 7 is NaN (codes 0x7F and 0xFF); there is
 * no infinity.
 *
 * bf16: IEEE-754 binary32 truncated to its top 16 bits (8 exponent bits,
 * 7 stored mantissa bits). The conversion here goes from fp64 to bf16 in a
 * single round-to-nearest-even step, never through fp32 (which could round
 * twice).
 *
 * Build: gcc -O2 -fopenmp -fPIC -shared (no -ffast-math: the rounding code
 * relies on IEEE semantics and on nearbyint() in round-to-nearest-even mode).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* e4m3fn code -> value, from the bit-field definition above. */
double oracle_e4m3_to_f64(uint8_t code)
{
    const int sign = (code >> 7) & 1;
    const int expo = (code >> 3) & 0xF;
    const int mant = code & 0x7;
    double mag;
    if (expo == 15 && mant == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant, -9);            /* subnormal: m * 2^-9 */
    else
        mag = ldexp(8.0 + (double)mant, expo - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

void oracle_e4m3_table(double table[256])
{
    for (int c = 0; c < 256; ++c)
        table[c] = oracle_e4m3_to_f64((uint8_t)c);
}

/* e5m2 code -> value (OCP FP8 E5M2: 1 sign bit, 5 exponent bits with bias
 * 15, 2 mantissa bits, IEEE-style: exponent 0 encodes subnormals m * 2^-16,
 * exponent 31 encodes infinity (m = 0) and NaN (m != 0)). The gist
 * "matmul_fp8.py", `benchmark()`, names torch.float8_e5m2 beside e4m3fn. */
double oracle_e5m2_to_f64(uint8_t code)
{
    const int sign = (code >> 7) & 1;
    const int expo = (code >> 2) & 0x1F;
    const int mant = code & 0x3;
    double mag;
    if (expo == 31)
        mag = mant ? NAN : INFINITY;
    else if (expo == 0)
        mag = ldexp((double)mant, -16);              /* subnormal: m * 2^-16 */
    else
        mag = ldexp(4.0 + (double)mant, expo - 17);  /* (1 + m/4) * 2^(e-15) */
    return sign ? -mag : mag;
}

void oracle_e5m2_table(double table[256])
{
    for (int c = 0; c < 256; ++c)
        table[c] = oracle_e5m2_to_f64((uint8_t)c);
}

/*
 * fp64 -> IEEE binary16 bit pattern, round to nearest, ties to even, in one
 * step: quantum 2^(e-10) for 2^e <= |x| < 2^(e+1), e clamped at -14 below
 * (subnormal quantum 2^-24); results of 65520 (= 2^16 - 2^4, the tie above
 * the largest finite 65504) or more overflow to infinity.
 */
uint16_t oracle_f64_to_f16_rne(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a, quantum, q;
    int e;
    if (isnan(x))
        return (uint16_t)(sign | 0x7E00u);
    a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e);
    e -= 1;
    if (e < -14)
        e = -14;
    quantum = ldexp(1.0, e - 10);
    q = nearbyint(a / quantum);          /* integer significand count */
    if (q * quantum >= 65520.0)
        return (uint16_t)(sign | 0x7C00u);
    /* encode: subnormal (e == -14 and q < 1024) or normal */
    if (q < 1024.0)
        return (uint16_t)(sign | (uint16_t)q);           /* exponent field 0 */
    if (q >= 2048.0) {                    /* rounding carried into the next binade */
        q /= 2.0;
        e += 1;
    }
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)q - 1024));
}

void oracle_f64_to_f16_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f64_to_f16_rne(x[i]);
}

/* binary16 bit pattern -> value (exact). */
double oracle_f16_to_f64(uint16_t bits)
{
    const int sign = (bits >> 15) & 1;
    const int expo = (bits >> 10) & 0x1F;
    const int mant = bits & 0x3FF;
    double mag;
    if (expo == 31)
        mag = mant ? NAN : INFINITY;
    else if (expo == 0)
        mag = ldexp((double)mant, -24);
    else
        mag = ldexp(1024.0 + (double)mant, expo - 25);
    return sign ? -mag : mag;
}

/* bf16 bit pattern -> value (exact: bf16 is a subset of fp64). */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/*
 * fp64 -> bf16, round to nearest, ties to even, in one step.
 * The value's quantum is 2^(e-7) for 2^e <= |x| < 2^(e+1), with e clamped at
 * -126 below (bf16 subnormals share fp32's exponent range, quantum 2^-133).
 * |x| / quantum is exact in fp64 (division by a power of two), nearbyint()
 * rounds it half-to-even, and the result times the quantum is exact again.
 * Results of 2^128 or more overflow to infinity. NaN maps to a quiet NaN
 * with the input's sign.
 */
uint16_t oracle_f64_to_bf16_rne(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a, quantum, q, v;
    int e;
    float f;
    uint32_t w;
    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0u);
    a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e);       /* a = f * 2^e with 0.5 <= f < 1 */
    e -= 1;                   /* 2^e <= a < 2^(e+1) */
    if (e < -126)
        e = -126;
    quantum = ldexp(1.0, e - 7);
    q = nearbyint(a / quantum);
    v = q * quantum;
    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    f = (float)v;             /* exact: v is a bf16 value */
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(sign | (uint16_t)(w >> 16));
}

/* Element-wise fp64 -> bf16 over an array (same rounding as above). */
void oracle_f64_to_bf16_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f64_to_bf16_rne(x[i]);
}

/*
 * fp64 -> IEEE binary32 bit pattern, round to nearest, ties to even, in one
 * step, by the same quantum method: quantum 2^(e-23) for 2^e <= |x| <
 * 2^(e+1), e clamped at -126 below (subnormal quantum 2^-149); results of
 * 2^128 or more (from 2^128 - 2^103, the tie above the largest finite
 * value) overflow to infinity. NaN maps to a quiet NaN with the input's
 * sign. The fp32 output of the scaled matmul (gist "matmul_fp8.py",
 * `benchmark()`, which takes the output dtype as an argument).
 */
uint32_t oracle_f64_to_f32_rne(double x)
{
    const uint32_t sign = signbit(x) ? 0x80000000u : 0u;
    double a, quantum, q, v;
    int e;
    float f;
    uint32_t w;
    if (isnan(x))
        return sign | 0x7FC00000u;
    a = fabs(x);
    if (isinf(a))
        return sign | 0x7F800000u;
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e);
    e -= 1;
    if (e < -126)
        e = -126;
    quantum = ldexp(1.0, e - 23);
    q = nearbyint(a / quantum);
    v = q * quantum;
    if (v >= ldexp(1.0, 128))
        return sign | 0x7F800000u;
    f = (float)v;             /* exact: v is an fp32 value */
    memcpy(&w, &f, sizeof w);
    return sign | w;
}

/* binary32 bit pattern -> value (exact). */
double oracle_f32_to_f64(uint32_t bits)
{
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * fp64 -> e4m3fn code for an e4m3 OUTPUT, one round-to-nearest-even step
 * with saturation: the cast of the fp32 accumulator to an fp8 output dtype
 * (gist "matmul_fp8.py", `matmul_fp8_kernel`, "Cast the accumulator to
 * output dtype (fp8)"). The pages do not say what happens beyond the
 * format's range; this reading saturates, as the hardware conversion such a
 * cast lowers to does: every |x| that rounds above 448 (and +-inf) gives
 * +-448 (0x7E / 0xFE). NaN gives 0x7F. Quantum 2^(e-3) for 2^e <= |x| <
 * 2^(e+1), e clamped at -6 below (subnormal quantum 2^-9).
 */
uint8_t oracle_f64_to_e4m3_sat(double x)
{
    const uint8_t sign = signbit(x) ? 0x80u : 0u;
    double a, q;
    int e;
    if (isnan(x))
        return 0x7Fu;
    a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a) || a >= 448.0)
        return (uint8_t)(sign | 0x7Eu);
    (void)frexp(a, &e);
    e -= 1;
    if (e < -6)
        e = -6;
    q = nearbyint(a / ldexp(1.0, e - 3));   /* significand in eighths */
    if (q == 0.0)
        return sign;                          /* below half the smallest subnormal */
    if (q < 8.0)
        return (uint8_t)(sign | (uint8_t)q);  /* subnormal (e == -6): m * 2^-9 */
    if (q >= 16.0) {                          /* rounding carried into the next binade */
        q /= 2.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && q > 14.0))        /* rounded above 448: saturate */
        return (uint8_t)(sign | 0x7Eu);
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)((int)q - 8));
}

/*
 * The scaled matrix multiply on a grid of selected outputs.
 *
 *   A        fp8 codes, [M, K] row-major; a_type 0 = e4m3fn, 1 = e5m2
 *   Bt       fp8 codes, [N, K] row-major (B[K, N] column-major); b_type likewise
 *   scale_a  1 value (scale_mode 0) or M values (scale_mode 1)
 *   scale_b  1 value (scale_mode 0) or N values (scale_mode 1)
 *   bias     [N] values, or NULL: bf16 bit patterns (out_type 0 and 3),
 *            binary16 (1) or binary32 (2)
 *   out_type 0 = bf16, 1 = fp16 (IEEE binary16), 2 = fp32 (IEEE binary32),
 *            3 = e4m3fn (saturating, see oracle_f64_to_e4m3_sat)
 *   rows     n_rows row indices into [0, M), or NULL for all rows (n_rows = M)
 *   cols     n_cols column indices into [0, N), or NULL for all (n_cols = N)
 *   out      [n_rows, n_cols] bit patterns of the output type (2, 2, 4 or
 *            1 bytes each)
 *   ref64    [n_rows, n_cols] unrounded fp64 result, or NULL
 *   absum    [n_rows, n_cols] S_ij * sum_k |a_ik * b_kj| (fp64), or NULL
 *
 * The fp64 dot product is exact when both operands are e4m3fn (see the file
 * header). With e5m2 operands (values are multiples of 2^-16 up to 57344)
 * a sum can need more than 53 bits; it is then rounded in fp64, an error
 * below K * 2^-53 * absum, far inside any fp32-accumulation tolerance.
 *
 * Returns 0, or -1 on a bad argument, -2 when out of memory.
 */
/* One output element's bias value and rounding, by output type. */
static double bias_value(const void *bias, int64_t j, int out_type)
{
    if (out_type == 1)
        return oracle_f16_to_f64(((const uint16_t *)bias)[j]);
    if (out_type == 2)
        return oracle_f32_to_f64(((const uint32_t *)bias)[j]);
    return oracle_bf16_to_f64(((const uint16_t *)bias)[j]);   /* bf16 and e4m3 outputs */
}

static void store_rounded(void *out, int64_t idx, double ref, int out_type)
{
    if (out_type == 0)
        ((uint16_t *)out)[idx] = oracle_f64_to_bf16_rne(ref);
    else if (out_type == 1)
        ((uint16_t *)out)[idx] = oracle_f64_to_f16_rne(ref);
    else if (out_type == 2)
        ((uint32_t *)out)[idx] = oracle_f64_to_f32_rne(ref);
    else
        ((uint8_t *)out)[idx] = oracle_f64_to_e4m3_sat(ref);
}

int oracle_scaled_mm_typed(const uint8_t *A, int a_type, const uint8_t *Bt, int b_type,
                           int64_t M, int64_t N, int64_t K,
                           const float *scale_a, const float *scale_b, int scale_mode,
                           const void *bias, int out_type,
                           const int64_t *rows, int64_t n_rows,
                           const int64_t *cols, int64_t n_cols,
                           void *out, double *ref64, double *absum,
                           int n_threads)
{
    double table_a[256], table_b[256];
    double *bdec;
    int64_t r, c;
    int bad = 0;

    if (!A || !Bt || !scale_a || !scale_b || !out || M < 0 || N < 0 || K < 0)
        return -1;
    if (scale_mode != 0 && scale_mode != 1)
        return -1;
    if ((a_type != 0 && a_type != 1) || (b_type != 0 && b_type != 1) || out_type < 0 || out_type > 3)
        return -1;
    if (!rows)
        n_rows = M;
    if (!cols)
        n_cols = N;
    for (r = 0; r < n_rows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= M))
            return -1;
    for (c = 0; c < n_cols; ++c)
        if (cols && (cols[c] < 0 || cols[c] >= N))
            return -1;
    if (n_rows == 0 || n_cols == 0)
        return 0;

    if (a_type == 0)
        oracle_e4m3_table(table_a);
    else
        oracle_e5m2_table(table_a);
    if (b_type == 0)
        oracle_e4m3_table(table_b);
    else
        oracle_e5m2_table(table_b);

    /* Decode the selected rows of Bt once. */
    bdec = (double *)malloc((size_t)n_cols * (size_t)(K > 0 ? K : 1) * sizeof(double));
    if (!bdec)
        return -2;
    for (c = 0; c < n_cols; ++c) {
        const int64_t j = cols ? cols[c] : c;
        for (int64_t k = 0; k < K; ++k)
            bdec[c * K + k] = table_b[Bt[j * K + k]];
    }

#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (r = 0; r < n_rows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *adec = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        if (!adec) {
            bad |= 1;
            continue;
        }
        for (int64_t k = 0; k < K; ++k)
            adec[k] = table_a[A[i * K + k]];
        for (int64_t cc = 0; cc < n_cols; ++cc) {
            const int64_t j = cols ? cols[cc] : cc;
            const double *b = bdec + cc * K;
            double dot = 0.0, mag = 0.0;
            double S, ref;
            for (int64_t k = 0; k < K; ++k) {
                const double p = adec[k] * b[k];
                dot += p;
                mag += fabs(p);
            }
            if (scale_mode == 0)
                S = (double)scale_a[0] * (double)scale_b[0];
            else
                S = (double)scale_a[i] * (double)scale_b[j];
            ref = dot * S;
            if (bias)
                ref += bias_value(bias, j, out_type);
            store_rounded(out, r * n_cols + cc, ref, out_type);
            if (ref64)
                ref64[r * n_cols + cc] = ref;
            if (absum)
                absum[r * n_cols + cc] = fabs(S) * mag;
        }
        free(adec);
    }
    free(bdec);
    return bad ? -2 : 0;
}

/* The e4m3fn x e4m3fn -> bf16 case (the benchmark path). */
int oracle_scaled_mm(const uint8_t *A, const uint8_t *Bt,
                     int64_t M, int64_t N, int64_t K,
                     const float *scale_a, const float *scale_b, int scale_mode,
                     const uint16_t *bias,
                     const int64_t *rows, int64_t n_rows,
                     const int64_t *cols, int64_t n_cols,
                     uint16_t *out, double *ref64, double *absum,
                     int n_threads)
{
    return oracle_scaled_mm_typed(A, 0, Bt, 0, M, N, K, scale_a, scale_b, scale_mode, bias, 0, rows, n_rows,
                                  cols, n_cols, out, ref64, absum, n_threads);
}

/*
 * Quantisation of bf16 data to fp8 codes, the step before the matmul in the
 * gist "matmul_fp8.py", `get_scale` and `benchmark()`:
 *
 *   amax  = max |x|                 over the tensor (mode 0) or each row (mode 1)
 *   scale = fp32(amax) / qmax       fp32 division; qmax = 448 (e4m3fn), 57344 (e5m2)
 *   v     = fp32(x) / scale         fp32 division, one correctly rounded step
 *   v     = clamp(v, -qmax, qmax)   NaN stays NaN
 *   q     = encode(v)               round to nearest, ties to even mantissa
 *
 * Two cases the recipe leaves open, read this way: a zero scale (every
 * element of the tensor or row is +-0) gives the codes of +-0 rather than
 * the NaN of 0/0, and every NaN becomes the code 0x7F.
 *
 * The divisions are IEEE binary32 operations (C float arithmetic compiled
 * without contraction or fast-math), the precision the pages compute in
 * (a bf16 tensor divided by an fp32 scale promotes to fp32).
 */
uint8_t oracle_encode_e4m3(float v)
{
    const uint8_t sign = signbit(v) ? 0x80u : 0u;
    double a, q;
    int e;
    if (isnan(v))
        return 0x7Fu;                     /* one NaN code for every NaN */
    a = fabs((double)v);
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e);
    e -= 1;                               /* 2^e <= a < 2^(e+1) */
    if (e < -6) {                         /* subnormal range: quantum 2^-9 */
        q = nearbyint(a / ldexp(1.0, -9));
        if (q >= 8.0)                     /* rounded up to the smallest normal */
            return (uint8_t)(sign | 0x08u);
        return (uint8_t)(sign | (uint8_t)q);
    }
    q = nearbyint(a / ldexp(1.0, e - 3)); /* significand in eighths: 8..16 */
    if (q >= 16.0) {
        q /= 2.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && q > 14.0))    /* beyond 448: not reached after the clamp */
        return (uint8_t)(sign | 0x7Eu);
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)((int)q - 8));
}

uint8_t oracle_encode_e5m2(float v)
{
    const uint8_t sign = signbit(v) ? 0x80u : 0u;
    double a, q;
    int e;
    if (isnan(v))
        return 0x7Fu;
    a = fabs((double)v);
    if (isinf(a))
        return (uint8_t)(sign | 0x7Cu);
    if (a == 0.0)
        return sign;
    (void)frexp(a, &e);
    e -= 1;
    if (e < -14) {                        /* subnormal range: quantum 2^-16 */
        q = nearbyint(a / ldexp(1.0, -16));
        if (q >= 4.0)
            return (uint8_t)(sign | 0x04u);
        return (uint8_t)(sign | (uint8_t)q);
    }
    q = nearbyint(a / ldexp(1.0, e - 2)); /* significand in quarters: 4..8 */
    if (q >= 8.0) {
        q /= 2.0;
        e += 1;
    }
    if (e > 15)                           /* beyond 57344: not reached after the clamp */
        return (uint8_t)(sign | 0x7Bu);
    return (uint8_t)(sign | (uint8_t)((e + 15) << 2) | (uint8_t)((int)q - 4));
}

/*
 * x: bf16 bit patterns [R, C] row-major; mode 0 per-tensor, 1 per-row;
 * q_type 0 e4m3fn, 1 e5m2; q: [R, C] codes; scale: 1 (mode 0) or R values.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_quantize(const uint16_t *x, int64_t R, int64_t C, int mode, int q_type, uint8_t *q, float *scale,
                    int n_threads)
{
    const float qmax = q_type == 0 ? 448.0f : 57344.0f;
    int64_t r;
    if (!x || !q || !scale || R < 0 || C < 0 || (mode != 0 && mode != 1) || (q_type != 0 && q_type != 1))
        return -1;
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    if (mode == 0) {
        float amax = 0.0f;
        for (int64_t i = 0; i < R * C; ++i) {
            const float a = fabsf((float)oracle_bf16_to_f64(x[i]));
            if (a > amax || isnan(a))
                amax = isnan(amax) ? amax : a;
        }
        scale[0] = amax / qmax;
    }
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; ++r) {
        float s;
        if (mode == 1) {
            float amax = 0.0f;
            for (int64_t c = 0; c < C; ++c) {
                const float a = fabsf((float)oracle_bf16_to_f64(x[r * C + c]));
                if (a > amax || isnan(a))
                    amax = isnan(amax) ? amax : a;
            }
            scale[r] = amax / qmax;
            s = scale[r];
        } else {
            s = scale[0];
        }
        for (int64_t c = 0; c < C; ++c) {
            const float xv = (float)oracle_bf16_to_f64(x[r * C + c]);
            float v = s == 0.0f ? xv : xv / s;
            if (v < -qmax)
                v = -qmax;
            else if (v > qmax)
                v = qmax;
            q[r * C + c] = q_type == 0 ? oracle_encode_e4m3(v) : oracle_encode_e5m2(v);
        }
    }
    return 0;
}

/* Threads an OpenMP parallel region would use by default (for reports). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
