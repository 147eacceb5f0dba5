/*
 * mx_oracle.c -- plain, slow, CPU reference for the MX block-scaled and the
 * FP16/BF16 matrix multiply.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, table or helper with the
 * CUDA library.
 *
 * What it follows:
 *  - RIGEL technical summary ("RIGEL - Engenharia Reversa do Caminho de
 *    Computacao de Tensores Metal 4.1 no Apple M4 Max"), section
 *    "Metodologia: O Harness RIGEL", checksum gate: the reference is a float64
 *    computation over exactly the quantized bytes the GPU consumes.
 *  - WWDC26 session 330 ("Metal tensors ... / Optimize custom ML ops with
 *    Metal tensors"), "Multi-plane tensors" and the 4:48 listing: a quantized
 *    tensor is an E4M3 data plane plus a UE8M0 ("FP8 E8M0") scale plane with
 *    block factors {32, 1}: one scale per 32 consecutive elements of the
 *    innermost (K) dimension.
 *  - WWDC26 session 330, "Quantized data types" and the custom-format
 *    passage of "Quantized matrix multiplication": 8-, 4- and 2-bit integer
 *    element types with the same E8M0 block scales, and a matmul that
 *    dequantizes one operand to f16 before multiplying.
 *  - The OCP Microscaling (MX) v1.0 definitions of E4M3, E5M2, E2M1 and UE8M0
 *    and of the conversion rule: X = 2^(floor(log2(amax)) - emax_elem),
 *    elements rounded to nearest-even and saturated (E5M2 included: an MX
 *    block never encodes an infinity, only its scale can say NaN).
 *
 * Every arithmetic step is done in double, where all code values, all scales
 * and all products of two scaled codes are exact.  Formats are decoded from
 * their bit fields in closed form; encoding is done by searching the list of
 * representable values (no bit tricks), so that it shares no method with a
 * hardware conversion instruction.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC mx_oracle.c -o liboracle.so -lm
 */
#define _DEFAULT_SOURCE
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>

#define MXO_E4M3 1
#define MXO_E2M1 2
#define MXO_E5M2 3
#define MXO_INT8 4
#define MXO_INT4 5
#define MXO_INT2 6
#define MXO_F16 2
#define MXO_BF16 1
#define MXO_ACT_NONE 0
#define MXO_ACT_GELU 1
#define MXO_ACT_GELU_TANH 2

/* ------------------------------------------------------------------------ */
/* Decoding (closed form from the bit fields).                               */
/* ------------------------------------------------------------------------ */

/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  No infinity;
 * S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448
 * (RIGEL summary, Main findings §3: E4M3 saturates at +-448, no Inf code). */
double mxo_decode_e4m3(uint8_t b)
{
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);                 /* m/8 * 2^(1-7) */
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 mantissa bits; exponent 31
 * holds infinity (mantissa 0) and NaN; the largest finite magnitude is
 * 1.75 * 2^15 = 57344. */
double mxo_decode_e5m2(uint8_t b)
{
    int s = (b >> 7) & 1, e = (b >> 2) & 31, m = b & 3;
    double mag;
    if (e == 31) return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0)
        mag = ldexp((double)m, -16);                /* m/4 * 2^(1-15) */
    else
        mag = ldexp(1.0 + m / 4.0, e - 15);
    return s ? -mag : mag;
}

/* E2M1 (low 4 bits of b): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit.
 * No infinity and no NaN; the largest magnitude is 1.5 * 2^2 = 6. */
double mxo_decode_e2m1(uint8_t b)
{
    int s = (b >> 3) & 1, e = (b >> 1) & 3, m = b & 1;
    double mag;
    if (e == 0)
        mag = 0.5 * m;                              /* m/2 * 2^(1-1) */
    else
        mag = ldexp(1.0 + m / 2.0, e - 1);
    return s ? -mag : mag;
}

/* Integer element formats: the low `bits` bits of c as a two's-complement
 * integer (int8 -128..127, int4 -8..7, int2 -2..1). */
static int int_bits(int fmt) { return fmt == MXO_INT8 ? 8 : fmt == MXO_INT4 ? 4 : 2; }

double mxo_decode_int(uint8_t c, int bits)
{
    int v = c & ((1 << bits) - 1);
    if (v >= (1 << (bits - 1))) v -= (1 << bits);
    return (double)v;
}

/* UE8M0: an unsigned 8-bit exponent; value 2^(c-127); 0xFF is NaN. */
double mxo_decode_ue8m0(uint8_t c)
{
    if (c == 0xFF) return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* IEEE binary16: 1 / 5 (bias 15) / 10. */
double mxo_decode_f16(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double mag;
    if (e == 31) return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0)
        mag = ldexp((double)m, -24);
    else
        mag = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -mag : mag;
}

/* bfloat16: 1 / 8 (bias 127) / 7. */
double mxo_decode_bf16(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 7) & 255, m = h & 127;
    double mag;
    if (e == 255) return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0)
        mag = ldexp((double)m, -133);
    else
        mag = ldexp(1.0 + m / 128.0, e - 127);
    return s ? -mag : mag;
}

/* ------------------------------------------------------------------------ */
/* Encoding: round to nearest, ties to even, saturate; by search.            */
/* ------------------------------------------------------------------------ */

/* Non-negative codes of a format in increasing order of value, finite only.
 * For E4M3 these are 0x00..0x7E, for E5M2 0x00..0x7B, for E2M1 0x0..0x7.
 * Value is increasing in the code for all three, so the code list is its own
 * sorted order. */
static double e4m3_pos[127];
static double e5m2_pos[124];
static double e2m1_pos[8];
static int tables_ready = 0;

static void build_tables(void)
{
    if (tables_ready) return;
    for (int c = 0; c < 127; ++c) e4m3_pos[c] = mxo_decode_e4m3((uint8_t)c);
    for (int c = 0; c < 124; ++c) e5m2_pos[c] = mxo_decode_e5m2((uint8_t)c);
    for (int c = 0; c < 8; ++c) e2m1_pos[c] = mxo_decode_e2m1((uint8_t)c);
    tables_ready = 1;
}

/* Nearest entry of vals[0..n) to a >= 0; ties go to the even index (whose
 * mantissa LSB is 0); a above the largest value saturates to it. */
static int nearest_code(const double* vals, int n, double a)
{
    if (a >= vals[n - 1]) return n - 1;
    int lo = 0, hi = n - 1;                 /* vals[lo] <= a < vals[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (vals[mid] <= a) lo = mid; else hi = mid;
    }
    double dlo = a - vals[lo], dhi = vals[hi] - a;
    if (dlo < dhi) return lo;
    if (dhi < dlo) return hi;
    return (lo % 2 == 0) ? lo : hi;
}

uint8_t mxo_encode_e4m3(double v)
{
    build_tables();
    if (isnan(v)) return 0x7F;
    int neg = signbit(v) ? 1 : 0;
    int c = nearest_code(e4m3_pos, 127, fabs(v));
    return (uint8_t)(c | (neg << 7));
}

/* Finite codes only: values beyond 57344 saturate to it, as the scaled
 * elements of an MX block are converted with saturation. */
uint8_t mxo_encode_e5m2(double v)
{
    build_tables();
    if (isnan(v)) return 0x7F;
    int neg = signbit(v) ? 1 : 0;
    int c = nearest_code(e5m2_pos, 124, fabs(v));
    return (uint8_t)(c | (neg << 7));
}

uint8_t mxo_encode_e2m1(double v)
{
    build_tables();
    if (isnan(v)) return 0x7;      /* E2M1 has no NaN; only the scale says NaN */
    int neg = signbit(v) ? 1 : 0;
    int c = nearest_code(e2m1_pos, 8, fabs(v));
    return (uint8_t)(c | (neg << 3));
}

/* Encode n values into codes of an element format (one code per byte). */
void mxo_encode_array(const double* v, int64_t n, int fmt, uint8_t* out)
{
    build_tables();
    for (int64_t i = 0; i < n; ++i)
        out[i] = (fmt == MXO_E4M3) ? mxo_encode_e4m3(v[i])
                 : (fmt == MXO_E5M2) ? mxo_encode_e5m2(v[i]) : mxo_encode_e2m1(v[i]);
}

/* Round v to the nearest integer, ties to the even one (written out from the
 * definition: the two integers around v and their distances), then saturate
 * to the two's-complement range of `bits` bits; returns the code's low bits. */
uint8_t mxo_encode_int(double v, int bits)
{
    const double lo = -(double)(1 << (bits - 1)), hi = (double)((1 << (bits - 1)) - 1);
    double q;
    if (isnan(v)) return 0;
    if (v <= lo) q = lo;
    else if (v >= hi) q = hi;
    else {
        double f = floor(v), d = v - f;
        if (d < 0.5) q = f;
        else if (d > 0.5) q = f + 1.0;
        else q = (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
        if (q > hi) q = hi;
    }
    return (uint8_t)((int)q & ((1 << bits) - 1));
}

/* ------------------------------------------------------------------------ */
/* MX quantizer (OCP MX rule), one 32-element block at a time.               */
/* ------------------------------------------------------------------------ */

/* floor(log2(a)) for a finite a > 0, taken from frexp of the exact double
 * value (a float widens to double exactly, subnormals included). */
static int floor_log2(double a)
{
    int p;
    (void)frexp(a, &p);             /* a = f * 2^p, f in [0.5, 1) */
    return p - 1;
}

int mxo_floor_log2_f32(float a) { return floor_log2((double)a); }

/* Quantize one block of 32 values.  emax is the exponent of the element
 * format's largest power of two (8 for E4M3, 15 for E5M2, 2 for E2M1, and
 * bits - 2 for the integer formats: 64, 4 and 1 are the largest powers of two
 * that int8, int4 and int2 hold, which for int8 is the OCP MXINT8 rule with
 * its implicit 2^-6 folded into the scale).
 * Writes 32 codes (one per byte, unpacked) and returns the UE8M0 scale code.
 *   amax = 0          -> scale code 0 (2^-127), all elements +-0
 *   NaN/Inf in block  -> scale code 0xFF (NaN); element codes are then
 *                        meaningless and are written as the encoding of 0. */
static uint8_t quantize_block(const double x[32], int fmt, uint8_t codes[32])
{
    const int is_int = (fmt == MXO_INT8 || fmt == MXO_INT4 || fmt == MXO_INT2);
    int emax = (fmt == MXO_E4M3) ? 8 : (fmt == MXO_E5M2) ? 15 : is_int ? int_bits(fmt) - 2 : 2;
    double amax = 0.0;
    int nonfinite = 0;
    for (int i = 0; i < 32; ++i) {
        if (!isfinite(x[i])) nonfinite = 1;
        else if (fabs(x[i]) > amax) amax = fabs(x[i]);
    }
    if (nonfinite) {
        for (int i = 0; i < 32; ++i) codes[i] = 0;
        return 0xFF;
    }
    int es;
    if (amax == 0.0) {
        es = -127;
    } else {
        es = floor_log2(amax) - emax;
        if (es < -127) es = -127;
        if (es > 127) es = 127;
    }
    for (int i = 0; i < 32; ++i) {
        double q = ldexp(x[i], -es);            /* exact in double */
        codes[i] = is_int ? mxo_encode_int(q, int_bits(fmt))
                   : (fmt == MXO_E4M3) ? mxo_encode_e4m3(q)
                   : (fmt == MXO_E5M2) ? mxo_encode_e5m2(q) : mxo_encode_e2m1(q);
    }
    return (uint8_t)(es + 127);
}

/* Quantize a rows x K matrix whose element (r, k) is src[r*s_row + k*s_k]
 * (so both a K-contiguous A and a row-major K x N B, read as N x K, are
 * covered).  K must be a multiple of 32.
 *   codes  : rows x K, one code per byte (unpacked), row-major
 *   scales : rows x (K/32) UE8M0 codes, row-major */
void mxo_quantize(const float* src, int64_t rows, int64_t K, int64_t s_row,
                  int64_t s_k, int fmt, uint8_t* codes, uint8_t* scales)
{
    build_tables();
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double x[32];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 32; ++i)
                x[i] = (double)src[r * s_row + (b * 32 + i) * s_k];
            scales[r * nb + b] =
                quantize_block(x, fmt, codes + r * K + b * 32);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* GEMMs in float64.                                                          */
/* ------------------------------------------------------------------------ */

/* Value of code c of an element format (E2M1 codes in the low nibble). */
static double decode_fmt(int fmt, int c)
{
    if (fmt == MXO_INT8 || fmt == MXO_INT4 || fmt == MXO_INT2)
        return mxo_decode_int((uint8_t)c, int_bits(fmt));
    return (fmt == MXO_E4M3) ? mxo_decode_e4m3((uint8_t)c)
           : (fmt == MXO_E5M2) ? mxo_decode_e5m2((uint8_t)c)
                               : mxo_decode_e2m1((uint8_t)(c & 15));
}

/* C[i][j] = sum_k (qa_ik * Xa_i,k/32) * (qb_jk * Xb_j,k/32), k ascending,
 * S[i][j] = sum_k |same product|.
 *   codesA  M x K (one code per byte, format fmt_a), scalesA M x K/32
 *   codesB  N x K (format fmt_b; B stored K-major, i.e. the transpose of the
 *           K x N operand)
 *   rows    optional list of nrows row indices of A to evaluate (NULL: all M,
 *           nrows must equal M); C and S are nrows x N. */

void mxo_gemm_mx(const uint8_t* codesA, const uint8_t* scalesA,
                 const uint8_t* codesB, const uint8_t* scalesB,
                 int64_t M, int64_t N, int64_t K, int fmt_a, int fmt_b,
                 const int64_t* rows, int64_t nrows, double* C, double* S)
{
    (void)M;
    double tab[256], tabb[256];
    for (int c = 0; c < 256; ++c) {
        tab[c] = decode_fmt(fmt_a, c);
        tabb[c] = decode_fmt(fmt_b, c);
    }
    int64_t nb = K / 32;
#pragma omp parallel
    {
        double* a = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t ii = 0; ii < nrows; ++ii) {
            int64_t i = rows ? rows[ii] : ii;
            for (int64_t k = 0; k < K; ++k)
                a[k] = tab[codesA[i * K + k]] *
                       mxo_decode_ue8m0(scalesA[i * nb + k / 32]);
            for (int64_t j = 0; j < N; ++j) {
                double c = 0.0, s = 0.0;
                for (int64_t b = 0; b < nb; ++b) {
                    double xb = mxo_decode_ue8m0(scalesB[j * nb + b]);
                    for (int64_t k = b * 32; k < b * 32 + 32; ++k) {
                        double p = a[k] * (tabb[codesB[j * K + k]] * xb);
                        c += p;
                        s += fabs(p);
                    }
                }
                C[ii * N + j] = c;
                S[ii * N + j] = s;
            }
        }
        free(a);
    }
}

/* C = A * B_mx^T for a row-major fp16 / bf16 A (M x K, bit patterns) and an MX
 * tensor B (codes N x K of format fmt_b, scales N x K/32): the matmul with one
 * operand in a custom quantized format, dequantized before the multiply
 * (WWDC26 session 330, "Quantized matrix multiplication", custom formats).
 * float64, ascending k; rows / nrows as in mxo_gemm_mx. */
void mxo_gemm_a16_bmx(const uint16_t* A, int dtype, const uint8_t* codesB,
                      const uint8_t* scalesB, int fmt_b, int64_t M, int64_t N,
                      int64_t K, const int64_t* rows, int64_t nrows, double* C,
                      double* S)
{
    (void)M;
    double tab[256];
    for (int c = 0; c < 256; ++c) tab[c] = decode_fmt(fmt_b, c);
    int64_t nb = K / 32;
#pragma omp parallel
    {
        double* a = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t ii = 0; ii < nrows; ++ii) {
            int64_t i = rows ? rows[ii] : ii;
            for (int64_t k = 0; k < K; ++k)
                a[k] = (dtype == MXO_BF16) ? mxo_decode_bf16(A[i * K + k])
                                           : mxo_decode_f16(A[i * K + k]);
            for (int64_t j = 0; j < N; ++j) {
                double c = 0.0, s = 0.0;
                for (int64_t b = 0; b < nb; ++b) {
                    double xb = mxo_decode_ue8m0(scalesB[j * nb + b]);
                    for (int64_t k = b * 32; k < b * 32 + 32; ++k) {
                        double p = a[k] * (tab[codesB[j * K + k]] * xb);
                        c += p;
                        s += fabs(p);
                    }
                }
                C[ii * N + j] = c;
                S[ii * N + j] = s;
            }
        }
        free(a);
    }
}

/* C = A * B for row-major A (M x K) and B (K x N) given as fp16 or bf16 bit
 * patterns; float64 accumulation in ascending k (the triple loop of the
 * dicastech tutorial "Treinar LLM em Swift", Passo 1, in i-k-j order).
 * rows / nrows as in mxo_gemm_mx. */
void mxo_gemm_f16(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N,
                  int64_t K, int dtype, const int64_t* rows, int64_t nrows,
                  double* C, double* S)
{
    (void)M;
    double* tab = (double*)malloc(sizeof(double) * 65536);
    for (int h = 0; h < 65536; ++h)
        tab[h] = (dtype == MXO_BF16) ? mxo_decode_bf16((uint16_t)h)
                                     : mxo_decode_f16((uint16_t)h);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ii = 0; ii < nrows; ++ii) {
        int64_t i = rows ? rows[ii] : ii;
        double* c = C + ii * N;
        double* s = S + ii * N;
        for (int64_t j = 0; j < N; ++j) { c[j] = 0.0; s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            double a = tab[A[i * K + k]];
            const uint16_t* brow = B + k * N;
            for (int64_t j = 0; j < N; ++j) {
                double p = a * tab[brow[j]];
                c[j] += p;
                s[j] += fabs(p);
            }
        }
    }
    free(tab);
}

/* ------------------------------------------------------------------------ */
/* Fused epilogue: bias and activation on the product.                       */
/* ------------------------------------------------------------------------ */

/* GELU(x) = x * Phi(x), Phi the standard normal CDF, written through erfc so
 * that the negative tail keeps its relative accuracy:
 * Phi(x) = erfc(-x / sqrt(2)) / 2. */
double mxo_gelu(double x)
{
    return 0.5 * x * erfc(-x / sqrt(2.0));
}

/* The tanh approximation of GELU (Hendrycks and Gimpel, "Gaussian Error
 * Linear Units"): 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))). */
double mxo_gelu_tanh(double x)
{
    const double k = sqrt(2.0 / M_PI);
    return 0.5 * x * (1.0 + tanh(k * (x + 0.044715 * x * x * x)));
}

/* The epilogue of the fused GEMM + bias + GELU kernel (RIGEL summary, Main
 * findings section 4): Y[i][j] = act(C[i][j] + bias[j]) for an rows x N
 * matrix C; bias may be NULL (no bias).  In place. */
void mxo_epilogue(double* C, int64_t rows, int64_t N, const double* bias, int act)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double x = C[i * N + j] + (bias ? bias[j] : 0.0);
            if (act == MXO_ACT_GELU) x = mxo_gelu(x);
            else if (act == MXO_ACT_GELU_TANH) x = mxo_gelu_tanh(x);
            C[i * N + j] = x;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Attention: O = softmax(Q K^T * scale) V, one head at a time.              */
/* ------------------------------------------------------------------------ */

/* The computation the FlashAttention kernel of WWDC26 session 330
 * ("Building advanced ops", 10:27-12:33: Q x K, a row-max reduction, exp,
 * then the product with V) fuses into one pass, written out as its
 * definition in float64: for head h and query i,
 *   s_j = scale * sum_c q_ic k_jc            (j < Lk)
 *   w_j = exp(s_j - max_j s_j) / sum_j exp(s_j - max_j s_j)
 *   O_ic = sum_j w_j v_jc,   Sv_ic = sum_j w_j |v_jc|
 * Q is BH x Lq x d, K and V are BH x Lk x d, fp16 or bf16 bit patterns,
 * row-major; rows (optional, nrows of them) selects query rows of every head;
 * O and Sv are BH x nrows x d. */
void mxo_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int dtype,
                   int64_t BH, int64_t Lq, int64_t Lk, int64_t d, double scale,
                   const int64_t* rows, int64_t nrows, double* O, double* Sv)
{
    double* tab = (double*)malloc(sizeof(double) * 65536);
    for (int h = 0; h < 65536; ++h)
        tab[h] = (dtype == MXO_BF16) ? mxo_decode_bf16((uint16_t)h)
                                     : mxo_decode_f16((uint16_t)h);
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int64_t b = 0; b < BH; ++b) {
            for (int64_t ii = 0; ii < nrows; ++ii) {
                int64_t i = rows ? rows[ii] : ii;
                const uint16_t* q = Q + (b * Lq + i) * d;
                double mx = -INFINITY;
                for (int64_t j = 0; j < Lk; ++j) {
                    const uint16_t* k = K + (b * Lk + j) * d;
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; ++c) acc += tab[q[c]] * tab[k[c]];
                    s[j] = scale * acc;
                    if (s[j] > mx) mx = s[j];
                }
                double den = 0.0;
                for (int64_t j = 0; j < Lk; ++j) {
                    s[j] = exp(s[j] - mx);
                    den += s[j];
                }
                double* o = O + (b * nrows + ii) * d;
                double* sv = Sv + (b * nrows + ii) * d;
                for (int64_t c = 0; c < d; ++c) { o[c] = 0.0; sv[c] = 0.0; }
                for (int64_t j = 0; j < Lk; ++j) {
                    const double w = s[j] / den;
                    const uint16_t* v = V + (b * Lk + j) * d;
                    for (int64_t c = 0; c < d; ++c) {
                        o[c] += w * tab[v[c]];
                        sv[c] += w * fabs(tab[v[c]]);
                    }
                }
            }
        }
        free(s);
    }
    free(tab);
}

int mxo_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}

/* Threads for the following parallel regions (n <= 0: the OpenMP default,
 * one per host core).  Timing control only: results do not depend on it. */
void mxo_set_num_threads(int n)
{
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    extern int omp_get_num_procs(void);
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}
