/*
 * CPU oracle for FP8 W8A8 block-scaled linear layers.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file: only the tests, the package smoke check and the benchmark's CPU
 * baseline do. It shares no code, header, table or constant generator with the
 * CUDA library; the two are compared, never combined.
 *
 * Plain, slow and written to be checked by eye against the pages:
 *
 *  - "FP8 Formats for Deep Learning" summary on "[vLLM] FP8: 8비트 부동소수점
 *    양자화" (section "논문 핵심 내용" and its format table): E4M3 has 4 exponent
 *    bits and 3 mantissa bits, has no infinity, and spans +-448. The same range
 *    is repeated on "FP8 serving slower than BF16" (section "하드웨어 세대가
 *    전제를 바꾼다").
 *  - The scaling strategies listed on the vLLM page (section "스케일링 전략
 *    체계"): symmetric ("Sym") scales per tensor, per token and per 128 block,
 *    static or dynamic; the 128x128 weight blocks of section "블록 양자화".
 *  - The "good case" of "FP8 and FP4: Throughput Needs Scaling" (section
 *    "Kernel caveat가 마지막 관문이다"): FP8 operands, high-precision
 *    accumulation. The oracle computes the exact-as-possible reference of that:
 *    dequantize both operands and multiply in FP64.
 *
 * Where the pages are silent the readings are fixed here and listed in the
 * design notes: E4M3 bias 7 with S.1111.111 as NaN, round-to-nearest-even with
 * saturation to +-448, scale = fl32(max(amax, 1e-10) / 448), quantized value =
 * e4m3(fl32(x / scale)), scales in FP32.
 *
 * Parity status: every function below is pinned by a test that does not reuse
 * its arithmetic (library casts, exhaustive enumeration, exact rational brute
 * force, closed forms, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

/* Smallest amax used to form a scale, so that an all-zero block gets a finite
 * scale (reading: the pages do not say what an all-zero block does). */
#define ORA_AMAX_FLOOR 1e-10f
/* Largest finite E4M3 magnitude: 1.75 * 2^8 (format table, +-448). */
#define ORA_E4M3_MAX 448.0

/* ---------------------------------------------------------------- E4M3 --- */

/* Exact value of an E4M3 code. Field layout s.eeee.mmm, bias 7:
 *   e > 0 : (-1)^s * 2^(e-7) * (1 + m/8)
 *   e = 0 : (-1)^s * 2^(-6) * (m/8)          (subnormal)
 *   e = 15, m = 7 : NaN (no infinity in E4M3) */
double ora_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Code of a representable non-negative magnitude r (0 <= r <= 448). */
static uint8_t e4m3_code_of_exact(double r)
{
    int e2;
    double f;
    if (r == 0.0)
        return 0;
    if (r < ldexp(1.0, -6)) {
        /* subnormal: r = m * 2^-9 */
        return (uint8_t)(r / ldexp(1.0, -9));
    }
    f = frexp(r, &e2);            /* r = f * 2^e2, f in [0.5, 1) */
    /* r = (1 + m/8) * 2^(e2-1)  ->  biased exponent e2 - 1 + 7 */
    return (uint8_t)(((e2 - 1 + 7) << 3) | (int)((2.0 * f - 1.0) * 8.0));
}

/* Round an FP32 value to E4M3: nearest representable value, ties to the even
 * code, saturating to +-448 (reading of "saturating to +-448"). The sign of
 * zero is kept. NaN -> 0x7F; +-Inf saturate like any other out-of-range value. */
uint8_t ora_e4m3_encode(float v)
{
    uint8_t sign;
    double a, quantum, n, r;
    int e2, exponent;
    if (isnan(v))
        return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs((double)v);
    if (a >= ORA_E4M3_MAX)
        return sign | 0x7E;
    if (a == 0.0)
        return sign;
    /* binade of a: 2^exponent <= a < 2^(exponent+1); below the smallest
     * normal binade (2^-6) the spacing stays that of the subnormals. */
    frexp(a, &e2);
    exponent = e2 - 1;
    if (exponent < -6)
        exponent = -6;
    /* 3 mantissa bits: representable values in this binade are multiples
     * of 2^(exponent-3). a / quantum is exact (power-of-two divisor). */
    quantum = ldexp(1.0, exponent - 3);
    n = nearbyint(a / quantum);   /* default rounding mode: nearest, ties to even */
    r = n * quantum;
    if (r > ORA_E4M3_MAX)
        r = ORA_E4M3_MAX;
    return sign | e4m3_code_of_exact(r);
}

/* Codes of the n FP32 values whose bit patterns are first, first+1, ...:
 * the encoder above applied to each (for sweeps over the whole FP32 range). */
void ora_e4m3_encode_bits(uint32_t first, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; i++) {
        union { uint32_t u; float f; } cv;
        cv.u = first + (uint32_t)i;
        out[i] = ora_e4m3_encode(cv.f);
    }
}

/* -------------------------------------------------------------- inputs --- */

/* BF16 bit pattern -> FP32 value (exact: BF16 is the top half of FP32). */
static float bf16_bits_to_float(uint16_t b)
{
    union { uint32_t u; float f; } cv;
    cv.u = (uint32_t)b << 16;
    return cv.f;
}

/* ---------------------------------------------------------- quantizers --- */

/* Scale of one block: fl32(max(amax, floor) / 448). The FP64 quotient of two
 * FP32 values rounded once to FP32 is the correctly rounded FP32 quotient. */
static float block_scale(float amax)
{
    float a = amax > ORA_AMAX_FLOOR ? amax : ORA_AMAX_FLOOR;
    return (float)((double)a / ORA_E4M3_MAX);
}

/* One E4M3 code for x under scale s: e4m3(fl32(x / s)). */
static uint8_t quant_value(float x, float s)
{
    return ora_e4m3_encode((float)((double)x / (double)s));
}

/*
 * Symmetric block quantization of a BF16 matrix x [rows][cols] (row-major):
 * the matrix is cut into blocks of br x bc (the last block in each direction
 * may be short), and each block gets one FP32 scale from its own amax and its
 * own E4M3 codes. Scale of block (rb, cb) goes to s[rb * s_stride_r + cb * s_stride_c].
 *
 *   per-token 1x128 groups (activations): br = 1,    bc = 128, s[g][m]  -> strides (1, rows)
 *   128x128 blocks (weights):             br = 128,  bc = 128, s[nb][kb] -> strides (ceil(cols/128), 1)
 *   per-tensor:                           br = rows, bc = cols
 *   per-token:                            br = 1,    bc = cols
 */
void ora_quant_blocks(const uint16_t *x, int64_t rows, int64_t cols,
                      int64_t br, int64_t bc, uint8_t *q, float *s,
                      int64_t s_stride_r, int64_t s_stride_c)
{
    int64_t rb, cb, r, c;
    for (rb = 0; rb * br < rows; rb++) {
        for (cb = 0; cb * bc < cols; cb++) {
            int64_t r0 = rb * br, r1 = r0 + br < rows ? r0 + br : rows;
            int64_t c0 = cb * bc, c1 = c0 + bc < cols ? c0 + bc : cols;
            float amax = 0.0f, scale;
            for (r = r0; r < r1; r++)
                for (c = c0; c < c1; c++) {
                    float a = fabsf(bf16_bits_to_float(x[r * cols + c]));
                    if (a > amax)
                        amax = a;
                }
            scale = block_scale(amax);
            s[rb * s_stride_r + cb * s_stride_c] = scale;
            for (r = r0; r < r1; r++)
                for (c = c0; c < c1; c++)
                    q[r * cols + c] = quant_value(bf16_bits_to_float(x[r * cols + c]), scale);
        }
    }
}

/* Quantization of a BF16 matrix with one given (static) FP32 scale. */
void ora_quant_static(const uint16_t *x, int64_t n, float scale, uint8_t *q)
{
    int64_t i;
    for (i = 0; i < n; i++)
        q[i] = quant_value(bf16_bits_to_float(x[i]), scale);
}

/* Scale a dynamic per-tensor quantization would pick for x (n values). */
float ora_tensor_scale(const uint16_t *x, int64_t n)
{
    int64_t i;
    float amax = 0.0f;
    for (i = 0; i < n; i++) {
        float a = fabsf(bf16_bits_to_float(x[i]));
        if (a > amax)
            amax = a;
    }
    return block_scale(amax);
}

/* ---------------------------------------------------------------- GEMM --- */

/*
 * Dequantize-then-GEMM in FP64 for one output element:
 *   a[m,k] = Sa(m, k) * dec(Qa[m,k]),   b[n,k] = Sw(n, k) * dec(Qw[n,k])
 *   Y[m,n] = sum_k a[m,k] * b[n,k]
 * and the magnitude sum_k |a[m,k] * b[n,k]| that the tolerance scales with.
 *
 * With activation groups of gk along K (scale sa[k/gk][m], i.e. [K/gk][lda_s])
 * and weight blocks of bn x bk (scale sw[n/bn][k/bk], i.e. [ceil(N/bn)][K/bk])
 * this equals sum_g Sa*Sw * sum_{k in g} dec*dec when gk == bk, up to the
 * order of rounding in FP64.
 */
static void gemm_point(const uint8_t *qa, const float *sa, int64_t lda_s,
                       const uint8_t *qw, const float *sw,
                       int64_t K, int64_t gk, int64_t bn, int64_t bk,
                       int64_t m, int64_t n, double *y, double *absdot)
{
    int64_t k, kb_count = (K + bk - 1) / bk;
    double acc = 0.0, mag = 0.0;
    for (k = 0; k < K; k++) {
        double a = (double)sa[(k / gk) * lda_s + m] * ora_e4m3_decode(qa[m * K + k]);
        double b = (double)sw[(n / bn) * kb_count + k / bk] * ora_e4m3_decode(qw[n * K + k]);
        acc += a * b;
        mag += fabs(a * b);
    }
    *y = acc;
    if (absdot)
        *absdot = mag;
}

/* Block-scaled GEMM for rows [m0, m1) of the output (all N columns).
 * y and absdot (nullable) are [m1-m0][N]; lda_s is the row count of the full
 * activation-scale matrix (its M). */
void ora_gemm_block_rows(const uint8_t *qa, const float *sa, int64_t lda_s,
                         const uint8_t *qw, const float *sw,
                         int64_t m0, int64_t m1, int64_t N, int64_t K,
                         int64_t gk, int64_t bn, int64_t bk,
                         double *y, double *absdot)
{
    int64_t m, n;
    for (m = m0; m < m1; m++)
        for (n = 0; n < N; n++)
            gemm_point(qa, sa, lda_s, qw, sw, K, gk, bn, bk, m, n,
                       &y[(m - m0) * N + n], absdot ? &absdot[(m - m0) * N + n] : NULL);
}

/* Block-scaled GEMM at a list of output points (m_i, n_i). */
void ora_gemm_block_points(const uint8_t *qa, const float *sa, int64_t lda_s,
                           const uint8_t *qw, const float *sw,
                           int64_t K, int64_t gk, int64_t bn, int64_t bk,
                           const int64_t *ms, const int64_t *ns, int64_t npts,
                           double *y, double *absdot)
{
    int64_t i;
    for (i = 0; i < npts; i++)
        gemm_point(qa, sa, lda_s, qw, sw, K, gk, bn, bk, ms[i], ns[i],
                   &y[i], absdot ? &absdot[i] : NULL);
}

/*
 * Grouped (mixture-of-experts) block-scaled GEMM at output points: rows
 * [offsets[e], offsets[e+1]) of Qa belong to expert e, whose weights are
 * Qw + e*N*K with scales Sw + e*ceil(N/bn)*(K/bk). Points whose row lies in
 * no expert's range get y = 0 (no expert writes them).
 */
void ora_gemm_grouped_points(const uint8_t *qa, const float *sa, int64_t lda_s,
                             const uint8_t *qw, const float *sw,
                             const int32_t *offsets, int64_t num_groups,
                             int64_t N, int64_t K, int64_t gk, int64_t bn, int64_t bk,
                             const int64_t *ms, const int64_t *ns, int64_t npts,
                             double *y, double *absdot)
{
    int64_t i, e, nb_count = (N + bn - 1) / bn, kb_count = (K + bk - 1) / bk;
    for (i = 0; i < npts; i++) {
        int64_t expert = -1;
        for (e = 0; e < num_groups; e++)
            if (ms[i] >= offsets[e] && ms[i] < offsets[e + 1])
                expert = e;
        if (expert < 0) {
            y[i] = 0.0;
            if (absdot)
                absdot[i] = 0.0;
            continue;
        }
        gemm_point(qa, sa, lda_s, qw + expert * N * K, sw + expert * nb_count * kb_count,
                   K, gk, bn, bk, ms[i], ns[i], &y[i], absdot ? &absdot[i] : NULL);
    }
}

/* Per-tensor GEMM for rows [m0, m1): Y = sa * sw * sum_k dec(Qa) dec(Qw),
 * written as the dequantize-then-GEMM above with one scale per operand. */
void ora_gemm_tensor_rows(const uint8_t *qa, float sa, const uint8_t *qw, float sw,
                          int64_t m0, int64_t m1, int64_t N, int64_t K,
                          double *y, double *absdot)
{
    int64_t m, n, k;
    for (m = m0; m < m1; m++)
        for (n = 0; n < N; n++) {
            double acc = 0.0, mag = 0.0;
            for (k = 0; k < K; k++) {
                double a = (double)sa * ora_e4m3_decode(qa[m * K + k]);
                double b = (double)sw * ora_e4m3_decode(qw[n * K + k]);
                acc += a * b;
                mag += fabs(a * b);
            }
            y[(m - m0) * N + n] = acc;
            if (absdot)
                absdot[(m - m0) * N + n] = mag;
        }
}

/* Per-tensor GEMM at output points. */
void ora_gemm_tensor_points(const uint8_t *qa, float sa, const uint8_t *qw, float sw,
                            int64_t K, const int64_t *ms, const int64_t *ns, int64_t npts,
                            double *y, double *absdot)
{
    int64_t i;
    for (i = 0; i < npts; i++)
        ora_gemm_tensor_rows(qa + ms[i] * K, sa, qw + ns[i] * K, sw, 0, 1, 1, K,
                             &y[i], absdot ? &absdot[i] : NULL);
}

/* ------------------------------------------------------------ KV cache --- */

/* BF16 bit pattern of an FP32 value: the nearest BF16 value (8 significant
 * bits, the FP32 exponent range), ties to the even pattern; overflow rounds
 * to infinity as in any IEEE binary format; NaN stays NaN (quiet, sign kept). */
static uint16_t float_to_bf16_bits(float f)
{
    union { uint32_t u; float f; } cv;
    double a, quantum, r;
    int e2, exponent;
    uint16_t sign;
    cv.f = f;
    sign = (uint16_t)((cv.u >> 16) & 0x8000u);
    if (isnan(f))
        return (uint16_t)(sign | 0x7FC0u);
    a = fabs((double)f);
    if (isinf(f) || a == 0.0) {
        cv.f = f;
        return (uint16_t)(cv.u >> 16);  /* +-Inf and +-0 are BF16 values */
    }
    /* binade 2^exponent <= a < 2^(exponent+1); below 2^-126 the spacing is
     * that of the subnormals, 2^-133. 8 significant bits: quantum 2^(exponent-7). */
    frexp(a, &e2);
    exponent = e2 - 1;
    if (exponent < -126)
        exponent = -126;
    quantum = ldexp(1.0, exponent - 7);
    r = nearbyint(a / quantum) * quantum;  /* a / quantum is exact */
    cv.f = (float)r;                       /* r is a BF16 value, or 2^128 -> Inf */
    return (uint16_t)(sign | (uint16_t)((cv.u >> 16) & 0x7FFFu));
}

/*
 * FP8 KV cache store ("[vLLM] FP8", section "KV 캐시 양자화": keys and values
 * kept in FP8 with one scale per tensor). Row t of x [tokens][elems] goes to
 * cache row slots[t] as e4m3(fl32(x / scale)); negative slots are padding and
 * slots >= num_slots are skipped.
 */
void ora_kv_store(const uint16_t *x, int64_t tokens, int64_t elems, const int64_t *slots,
                  int64_t num_slots, float scale, uint8_t *cache)
{
    int64_t t, e;
    for (t = 0; t < tokens; t++) {
        if (slots[t] < 0 || slots[t] >= num_slots)
            continue;
        for (e = 0; e < elems; e++)
            cache[slots[t] * elems + e] = quant_value(bf16_bits_to_float(x[t * elems + e]), scale);
    }
}

/* FP8 KV cache load: row t of out [tokens][elems] (BF16 bit patterns) is
 * cache row slots[t] dequantized, bf16(fl32(dec(q) * scale)); the product of
 * a code (4 significant bits) and an FP32 scale is exact in FP64, so the cast
 * to float is the correctly rounded FP32 product. Skipped rows are untouched. */
void ora_kv_load(const uint8_t *cache, int64_t tokens, int64_t elems, const int64_t *slots,
                 int64_t num_slots, float scale, uint16_t *out)
{
    int64_t t, e;
    for (t = 0; t < tokens; t++) {
        if (slots[t] < 0 || slots[t] >= num_slots)
            continue;
        for (e = 0; e < elems; e++)
            out[t * elems + e] = float_to_bf16_bits((float)(ora_e4m3_decode(cache[slots[t] * elems + e]) *
                                                            (double)scale));
    }
}

/* The BF16 rounding above, exposed for its pin against an independent cast. */
void ora_bf16_from_f32(const float *x, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; i++)
        out[i] = float_to_bf16_bits(x[i]);
}
