/*
 * oracle.c -- plain CPU oracle for the block-scaled FP8 linear-layer GEMMs.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
 * baseline leg of bench.py load this library.  The CUDA library never includes,
 * links or calls it, and it includes nothing from the CUDA side.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math), so
 * every float operation written below is one IEEE-754 binary32 or binary64
 * operation rounded to nearest even.
 *
 * Sources (web pages, by title):
 *  [P1] "Replaced cublasLt calls with rocblas gemm + 6 manually crafted
 *       epilogues" -- linear layer Y = X.W^T + b, its backward (dX, dW, db),
 *       bias length per epilogue, fp32 reductions, bias-then-GELU order.
 *  [P3] "Weight gradient kernels for dense and MoE models" -- fp8 x fp8 -> fp32
 *       "nt" weight-gradient GEMM with out += a.b^T semantics, the k-grouped
 *       MoE variant, the per-token (1x128) cast of both operands, and the
 *       worked ones/rand example.
 *  [P4] "FP8 GEMM for the fprop should use fast accumulation" -- e4m3 for the
 *       forward GEMM, e5m2 on the gradient side, fast vs full accumulation,
 *       per-tensor scales.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - fp8 bit layouts are the OCP FP8 definitions (the pages only name e4m3 and
 *    e5m2); encoding is round-to-nearest-even with saturation to +-max.
 *  - the per-token cast is not defined on [P3]; it is read as: per row and per
 *    128-element block, amax = max|x|, inv = fl32(FMAX/amax),
 *    scale = fl32(amax/FMAX), q = enc(fl32(x*inv)).  A block whose amax is 0,
 *    or whose FMAX/amax overflows binary32, gets scale = 1, inv = 1.
 *  - GELU is the tanh form 0.5 z (1 + tanh(sqrt(2/pi)(z + 0.044715 z^3))),
 *    evaluated through the identity 0.5 (1 + tanh u) = 1 / (1 + exp(-2u)).
 */
#include "oracle.h"

#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* fp8 codec: decode by table built from the bit fields                      */
/* ------------------------------------------------------------------------ */

/* Value of one code from its sign / exponent / mantissa fields.
 *   e4m3 ("fn" variant): 1-4-3, bias 7, no infinity, S.1111.111 is NaN.
 *   e5m2:                1-5-2, bias 15, exponent 11111 is Inf (m=0) / NaN.
 * Exponent field 0 is subnormal: m / 2^mbits * 2^(1 - bias). */
static double decode_fields(int fmt, unsigned code)
{
    const int ebits = (fmt == ORACLE_E4M3) ? 4 : 5;
    const int mbits = 7 - ebits;
    const int bias = (fmt == ORACLE_E4M3) ? 7 : 15;
    const unsigned sign = (code >> 7) & 1u;
    const unsigned e = (code >> mbits) & ((1u << ebits) - 1u);
    const unsigned m = code & ((1u << mbits) - 1u);
    double v;
    if (fmt == ORACLE_E4M3 && e == 15u && m == 7u) return NAN;
    if (fmt == ORACLE_E5M2 && e == 31u) {
        if (m != 0u) return NAN;
        return sign ? -INFINITY : INFINITY;
    }
    if (e == 0u)
        v = ldexp((double)m, 1 - bias - mbits);
    else
        v = ldexp((double)((1u << mbits) + m), (int)e - bias - mbits);
    return sign ? -v : v;
}

static double g_table[2][256];
static int g_table_ready = 0;

static void build_tables(void)
{
    if (g_table_ready) return;
    for (int f = 0; f < 2; ++f)
        for (unsigned c = 0; c < 256u; ++c) g_table[f][c] = decode_fields(f, c);
    g_table_ready = 1;
}

void oracle_fp8_decode_table(int fmt, double out[256])
{
    build_tables();
    memcpy(out, g_table[fmt ? 1 : 0], sizeof(double) * 256);
}

/* largest finite positive code and its value */
static int max_code(int fmt) { return (fmt == ORACLE_E4M3) ? 0x7E : 0x7B; }

double oracle_fp8_max(int fmt)
{
    build_tables();
    return g_table[fmt ? 1 : 0][max_code(fmt)];
}

/* Exact round-to-nearest-even onto the fp8 grid with saturation.
 * Codes 0..max_code are the non-negative finite values in increasing order,
 * so a bisection finds the two neighbours of |x|; the distances are exact in
 * binary64 (both operands are short dyadic rationals).  Ties go to the code
 * whose mantissa LSB is 0.  |x| at or above the largest finite value gives
 * that value (saturating, "satfinite").  Zero keeps its sign. */
uint8_t oracle_fp8_encode(int fmt, float x)
{
    build_tables();
    const double* t = g_table[fmt ? 1 : 0];
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    const int top = max_code(fmt);
    int code;
    if (a >= t[top]) {
        code = top;
    } else {
        int lo = 0, hi = top; /* t[lo] <= a < t[hi] */
        while (hi - lo > 1) {
            const int mid = (lo + hi) / 2;
            if (t[mid] <= a) lo = mid; else hi = mid;
        }
        const double dlo = a - t[lo];
        const double dhi = t[hi] - a;
        if (dlo < dhi) code = lo;
        else if (dhi < dlo) code = hi;
        else code = (lo & 1) ? hi : lo;
    }
    return (uint8_t)(sign | (uint8_t)code);
}

void oracle_fp8_encode_array(int fmt, const float* x, int64_t n, uint8_t* q)
{
    build_tables();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) q[i] = oracle_fp8_encode(fmt, x[i]);
}

/* ------------------------------------------------------------------------ */
/* bf16                                                                      */
/* ------------------------------------------------------------------------ */

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* bf16 = 1-8-7, bias 127.  Round |v| to a multiple of the bf16 spacing of its
 * binade (2^(e-7), with e clamped at -126 for subnormals) using nearbyint in
 * the default round-to-nearest-even mode; v / spacing is exact. */
uint16_t oracle_f64_to_bf16(double v)
{
    if (isnan(v)) return 0x7FC0;
    const uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    const double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e2;
    frexp(a, &e2);
    int ue = e2 - 1;
    if (ue < -126) ue = -126;
    const double spacing = ldexp(1.0, ue - 7);
    const double r = nearbyint(a / spacing) * spacing;
    if (r > ldexp(255.0, 120)) return (uint16_t)(sign | 0x7F80);
    const float rf = (float)r; /* exact: r is on the bf16 grid */
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

void oracle_f64_to_bf16_array(const double* v, int64_t n, uint16_t* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(v[i]);
}

/* ------------------------------------------------------------------------ */
/* per-128-block quantization ([P3] per-token cast; e4m3/e5m2 from [P4])      */
/* ------------------------------------------------------------------------ */

/* One block of 128 values v[0..127] (already widened from bf16, exact).
 * Output code k goes to out[k * ostride]. */
static void quantize_block(int fmt, const float* v, uint8_t* out, int64_t ostride, float* scale_out)
{
    const float fmax = (float)oracle_fp8_max(fmt);
    float amax = 0.0f;
    for (int k = 0; k < 128; ++k) {
        const float a = fabsf(v[k]);
        if (a > amax) amax = a;
    }
    float inv = 1.0f, scale = 1.0f;
    if (amax > 0.0f) {
        const float t = fmax / amax; /* binary32 division */
        if (t <= FLT_MAX) {
            inv = t;
            scale = amax / fmax; /* binary32 division */
        }
    }
    *scale_out = scale;
    for (int k = 0; k < 128; ++k) {
        const float y = v[k] * inv; /* binary32 product */
        out[(int64_t)k * ostride] = oracle_fp8_encode(fmt, y);
    }
}

/* transpose == 0: blocks run along a row.  x is [rows][cols] (row stride ldx),
 *   cols % 128 == 0; q is [rows][cols]; scale[b * sld + r] for block b of row r.
 * transpose == 1: blocks run down a column.  rows % 128 == 0; q is [cols][rows]
 *   (the transposed matrix, so the 128 values of a block are contiguous);
 *   scale[b * sld + c] for block b (rows 128b..128b+127) of column c. */
void oracle_quantize(int fmt, const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                     int transpose, uint8_t* q, float* scale, int64_t sld)
{
    build_tables();
    if (!transpose) {
        const int64_t nb = cols / 128;
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            float v[128];
            for (int64_t b = 0; b < nb; ++b) {
                for (int k = 0; k < 128; ++k) v[k] = oracle_bf16_to_f32(x[r * ldx + b * 128 + k]);
                quantize_block(fmt, v, q + r * cols + b * 128, 1, &scale[b * sld + r]);
            }
        }
    } else {
        const int64_t nb = rows / 128;
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; ++c) {
            float v[128];
            for (int64_t b = 0; b < nb; ++b) {
                for (int k = 0; k < 128; ++k) v[k] = oracle_bf16_to_f32(x[(b * 128 + k) * ldx + c]);
                quantize_block(fmt, v, q + c * rows + b * 128, 1, &scale[b * sld + c]);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* block-scaled GEMM ([P3] "nt": both operands K-major)                       */
/* ------------------------------------------------------------------------ */

/* acc[ii][jj] = sum over 128-blocks kb of K (starting at column k0 of both
 *               operands) of  sa[kb][i] * sb[kb][j] * sum_{k in kb} dec(qa[i][k]) * dec(qb[j][k])
 * S[ii][jj]   = sum_k |dec(qa[i][k]) sa[kb][i] * dec(qb[j][k]) sb[kb][j]|
 * with i = rows[ii] (or ii when rows is NULL) and j = cols[jj] likewise.
 * Scales are indexed at block (k0/128 + kb).  All sums in binary64.  K = 0
 * gives zeros.  acc and S are [nrows][ncols]; S may be NULL. */
void oracle_gemm(int64_t K, int64_t k0,
                 const uint8_t* qa, int64_t lda, const float* sa, int64_t sa_ld, int fmt_a,
                 const uint8_t* qb, int64_t ldb, const float* sb, int64_t sb_ld, int fmt_b,
                 const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                 double* acc, double* S)
{
    build_tables();
    const double* ta = g_table[fmt_a ? 1 : 0];
    const double* tb = g_table[fmt_b ? 1 : 0];
    const int64_t nkb = K / 128;
    const int64_t kb0 = k0 / 128;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ii = 0; ii < nrows; ++ii) {
        const int64_t i = rows ? rows[ii] : ii;
        for (int64_t jj = 0; jj < ncols; ++jj) {
            const int64_t j = cols ? cols[jj] : jj;
            double total = 0.0, total_abs = 0.0;
            for (int64_t kb = 0; kb < nkb; ++kb) {
                const double s_a = (double)sa[(kb0 + kb) * sa_ld + i];
                const double s_b = (double)sb[(kb0 + kb) * sb_ld + j];
                const uint8_t* pa = qa + i * lda + k0 + kb * 128;
                const uint8_t* pb = qb + j * ldb + k0 + kb * 128;
                double part = 0.0, part_abs = 0.0;
                for (int k = 0; k < 128; ++k) {
                    const double p = ta[pa[k]] * tb[pb[k]];
                    part += p;
                    part_abs += fabs(p);
                }
                total += s_a * s_b * part;
                total_abs += fabs(s_a * s_b) * part_abs;
            }
            acc[ii * ncols + jj] = total;
            if (S) S[ii * ncols + jj] = total_abs;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP8: power-of-two scales per 32 elements (the MX block format named among */
/* the fp8 recipes on "How can we use te.Linear with weight parallel?")       */
/* ------------------------------------------------------------------------ */

/* Smallest integer e in [-127, 127] with amax <= FMAX * 2^e (so that no element
 * of the block saturates); 0 for an all-zero block.  Found by stepping e one
 * power of two at a time with exact binary64 comparisons. */
static int mx_exponent(int fmt, double amax)
{
    const double fmax = oracle_fp8_max(fmt);
    if (amax == 0.0) return 0;
    int e = 0;
    while (e < 127 && amax > ldexp(fmax, e)) ++e;
    while (e > -127 && amax <= ldexp(fmax, e - 1)) --e;
    return e;
}

/* One 32-element block: exponent, then q_k = enc(x_k * 2^-e) (the scaling by a
 * power of two is exact, so this is a single rounding of x_k * 2^-e). */
static void mx_block(int fmt, const float* v, uint8_t* q, int64_t qstride, int8_t* e_out)
{
    double amax = 0.0;
    for (int k = 0; k < 32; ++k) {
        const double a = fabs((double)v[k]);
        if (a > amax) amax = a;
    }
    const int e = mx_exponent(fmt, amax);
    for (int k = 0; k < 32; ++k) q[k * qstride] = oracle_fp8_encode(fmt, (float)ldexp((double)v[k], -e));
    *e_out = (int8_t)e;
}

void oracle_mx_quantize(int fmt, const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                        int transpose, uint8_t* q, int8_t* e, int64_t eld)
{
    build_tables();
    if (!transpose) {
        const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            float v[32];
            for (int64_t b = 0; b < nb; ++b) {
                for (int k = 0; k < 32; ++k) v[k] = oracle_bf16_to_f32(x[r * ldx + b * 32 + k]);
                mx_block(fmt, v, q + r * cols + b * 32, 1, &e[b * eld + r]);
            }
        }
    } else {
        const int64_t nb = rows / 32;
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; ++c) {
            float v[32];
            for (int64_t b = 0; b < nb; ++b) {
                for (int k = 0; k < 32; ++k) v[k] = oracle_bf16_to_f32(x[(b * 32 + k) * ldx + c]);
                mx_block(fmt, v, q + c * rows + b * 32, 1, &e[b * eld + c]);
            }
        }
    }
}

/* acc[ii][jj] = sum_k dec(qa[i][k]) 2^ea[k/32][i] * dec(qb[j][k]) 2^eb[k/32][j],
 * S[ii][jj] = the same sum of absolute values, binary64, i = rows[ii] (or ii),
 * j = cols[jj] (or jj); K a multiple of 32. */
void oracle_mx_gemm(int64_t K,
                    const uint8_t* qa, int64_t lda, const int8_t* ea, int64_t ea_ld, int fmt_a,
                    const uint8_t* qb, int64_t ldb, const int8_t* eb, int64_t eb_ld, int fmt_b,
                    const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                    double* acc, double* S)
{
    build_tables();
    const double* ta = g_table[fmt_a ? 1 : 0];
    const double* tb = g_table[fmt_b ? 1 : 0];
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ii = 0; ii < nrows; ++ii) {
        const int64_t i = rows ? rows[ii] : ii;
        for (int64_t jj = 0; jj < ncols; ++jj) {
            const int64_t j = cols ? cols[jj] : jj;
            double total = 0.0, total_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = ldexp(ta[qa[i * lda + k]], ea[(k / 32) * ea_ld + i]);
                const double b = ldexp(tb[qb[j * ldb + k]], eb[(k / 32) * eb_ld + j]);
                total += a * b;
                total_abs += fabs(a * b);
            }
            acc[ii * ncols + jj] = total;
            if (S) S[ii * ncols + jj] = total_abs;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* per-tensor scaling ([P4]: one scale per operand tensor, taken from an amax  */
/* history -- "delayed scaling" -- or from the tensor itself; with it the      */
/* fast-accumulation GEMM needs no promotion inside the K loop)              */
/* ------------------------------------------------------------------------ */

/* One scale for the whole tensor from a given amax A (the tensor's own amax, or
 * the largest amax of earlier steps): inv = fl32(FMAX/A), scale = fl32(A/FMAX),
 * q = enc(fl32(x*inv)) -- the same reading as the per-block cast, with the
 * block widened to the tensor.  A = 0, or FMAX/A overflowing binary32, gives
 * inv = scale = 1.  Values above A saturate to +-FMAX (a delayed amax may be
 * smaller than the tensor's own).  amax_out = max|x| of this tensor, exact.
 * transpose == 0: q [rows][cols]; transpose == 1: q [cols][rows]. */
void oracle_tensor_quantize(int fmt, const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                            int transpose, float amax_in, uint8_t* q, float* scale_out, float* amax_out)
{
    build_tables();
    const float fmax = (float)oracle_fp8_max(fmt);
    float inv = 1.0f, scale = 1.0f;
    if (amax_in > 0.0f) {
        const float t = fmax / amax_in; /* binary32 division */
        if (t <= FLT_MAX) {
            inv = t;
            scale = amax_in / fmax; /* binary32 division */
        }
    }
    *scale_out = scale;
    float amax = 0.0f;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            const float v = oracle_bf16_to_f32(x[r * ldx + c]);
            const float a = fabsf(v);
            if (a > amax) amax = a;
            const uint8_t code = oracle_fp8_encode(fmt, v * inv); /* binary32 product */
            if (transpose)
                q[c * rows + r] = code;
            else
                q[r * cols + c] = code;
        }
    }
    *amax_out = amax;
}

/* Amax history of delayed scaling: the new amax enters at position 0, every
 * older entry moves one place back (the oldest drops out), and the amax to
 * scale the next cast with is the largest entry of the updated history. */
void oracle_amax_history(float* hist, int64_t len, float amax_new, float* amax_use)
{
    for (int64_t i = len - 1; i > 0; --i) hist[i] = hist[i - 1];
    hist[0] = amax_new;
    float m = 0.0f;
    for (int64_t i = 0; i < len; ++i)
        if (hist[i] > m) m = hist[i];
    *amax_use = m;
}

/* acc[i][j] = sa * sb * sum_k dec(qa[i][k]) dec(qb[j][k]) and S the same sum of
 * absolute values, binary64, for all rows x cols; both operands K-major. */
void oracle_tensor_gemm(int64_t M, int64_t N, int64_t K,
                        const uint8_t* qa, int64_t lda, float sa, int fmt_a,
                        const uint8_t* qb, int64_t ldb, float sb, int fmt_b,
                        double* acc, double* S)
{
    build_tables();
    const double* ta = g_table[fmt_a ? 1 : 0];
    const double* tb = g_table[fmt_b ? 1 : 0];
    const double s = (double)sa * (double)sb;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double total = 0.0, total_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = ta[qa[i * lda + k]] * tb[qb[j * ldb + k]];
                total += p;
                total_abs += fabs(p);
            }
            acc[i * N + j] = s * total;
            if (S) S[i * N + j] = fabs(s) * total_abs;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* epilogue math ([P1]: bias, GELU, dGELU, db = column sum)                  */
/* ------------------------------------------------------------------------ */

/* gelu(z) = 0.5 z (1 + tanh(u)), u = c (z + 0.044715 z^3), c = sqrt(2/pi).
 * Evaluated through 0.5 (1 + tanh u) = 1 / (1 + exp(-2u)): the same number,
 * without the cancellation of 1 + tanh(u) in binary64 when u < -18. */
double oracle_gelu(double z)
{
    const double c = sqrt(2.0 / acos(-1.0));
    const double u = c * (z + 0.044715 * z * z * z);
    return z / (1.0 + exp(-2.0 * u));
}

/* d/dz of the above: 0.5 (1 + t) + 0.5 z (1 - t^2) c (1 + 3 * 0.044715 z^2),
 * t = tanh(u), with 0.5 (1 + t) = s(2u) and 1 - t^2 = 4 s(2u) s(-2u),
 * s(x) = 1 / (1 + exp(-x)). */
double oracle_dgelu(double z)
{
    const double c = sqrt(2.0 / acos(-1.0));
    const double u = c * (z + 0.044715 * z * z * z);
    const double sp = 1.0 / (1.0 + exp(-2.0 * u));
    const double sm = 1.0 / (1.0 + exp(2.0 * u));
    return sp + 2.0 * z * c * (1.0 + 3.0 * 0.044715 * z * z) * sp * sm;
}

void oracle_gelu_array(const double* z, double* y, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_gelu(z[i]);
}

void oracle_dgelu_array(const double* z, double* y, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_dgelu(z[i]);
}

/* db[j] = sum over all M rows of dz[i][j] ([P1] backward, db = sum(dY, axis 0),
 * taken at the pre-activation: the GELU derivative is applied first). */
void oracle_colsum(const double* dz, int64_t M, int64_t N, double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < M; ++i) s += dz[i * N + j];
        out[j] = s;
    }
}

/* BGRADB ([P1] backward): db is taken together with dW by reducing the
 * gradient operand of the weight-gradient GEMM over that GEMM's k (the
 * tokens).  With the operand cast to fp8 by 1x128 blocks, this is
 *   db[r] = sum_k scale[k/128][r] * dec(q[r][k]),
 * summed element by element in binary64.  S[r] = sum_k |scale * dec| (the
 * magnitude sum the error bound is taken against), or skipped when S is NULL. */
void oracle_operand_rowsum(int fmt, const uint8_t* q, int64_t ldq, const float* scale, int64_t scale_ld,
                           int64_t rows, int64_t K, double* out, double* S)
{
    build_tables();
    const double* t = g_table[fmt ? 1 : 0];
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double total = 0.0, total_abs = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double v = (double)scale[(k / 128) * scale_ld + r] * t[q[r * ldq + k]];
            total += v;
            total_abs += fabs(v);
        }
        out[r] = total;
        if (S) S[r] = total_abs;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
