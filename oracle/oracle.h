/*
 * oracle.h -- plain CPU oracle for the block-scaled FP8 linear-layer GEMMs.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path includes, links or
 * calls this file: only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Everything is computed in double precision (fp64) with plain loops, in the
 * order the method states it.  See oracle.c for the passage each function
 * follows.
 */
#ifndef FP8LL_ORACLE_H
#define FP8LL_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* fp8 formats named on "FP8 GEMM for the fprop should use fast accumulation"
 * (e4m3 for fprop, e5m2 on the gradient side).  Bit layouts: OCP FP8. */
enum { ORACLE_E4M3 = 0, ORACLE_E5M2 = 1 };

/* codec */
void    oracle_fp8_decode_table(int fmt, double out[256]);
double  oracle_fp8_max(int fmt);
uint8_t oracle_fp8_encode(int fmt, float x);
void    oracle_fp8_encode_array(int fmt, const float* x, int64_t n, uint8_t* q);

/* bf16 helpers (bit patterns stored as uint16) */
float    oracle_bf16_to_f32(uint16_t h);
uint16_t oracle_f64_to_bf16(double v); /* round to nearest even, via exact comparison */
void     oracle_f64_to_bf16_array(const double* v, int64_t n, uint16_t* out);

/* per-128-block quantization (the page's per-token cast) */
void oracle_quantize(int fmt, const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                     int transpose, uint8_t* q, float* scale, int64_t sld);

/* block-scaled GEMM: acc[i][j] = sum_kb sa*sb * sum_{k in kb} dec(qa)*dec(qb) */
void oracle_gemm(int64_t K, int64_t k0,
                 const uint8_t* qa, int64_t lda, const float* sa, int64_t sa_ld, int fmt_a,
                 const uint8_t* qb, int64_t ldb, const float* sb, int64_t sb_ld, int fmt_b,
                 const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                 double* acc, double* S);

/* epilogue math */
/* MXFP8 (power-of-two scale per 32 elements, stored as the exponent e):
 * quantize rows (transpose = 0: blocks along each row, q [rows][cols], e
 * [cols/32][eld]) or columns (transpose = 1: blocks down each column, q
 * [cols][rows], e [rows/32][eld]); GEMM over K (a multiple of 32). */
void oracle_mx_quantize(int fmt, const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                        int transpose, uint8_t* q, int8_t* e, int64_t eld);
void oracle_mx_gemm(int64_t K,
                    const uint8_t* qa, int64_t lda, const int8_t* ea, int64_t ea_ld, int fmt_a,
                    const uint8_t* qb, int64_t ldb, const int8_t* eb, int64_t eb_ld, int fmt_b,
                    const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                    double* acc, double* S);

/* per-tensor scaling: cast from a given amax, amax history, GEMM */
void oracle_tensor_quantize(int fmt, const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                            int transpose, float amax_in, uint8_t* q, float* scale_out, float* amax_out);
void oracle_amax_history(float* hist, int64_t len, float amax_new, float* amax_use);
void oracle_tensor_gemm(int64_t M, int64_t N, int64_t K,
                        const uint8_t* qa, int64_t lda, float sa, int fmt_a,
                        const uint8_t* qb, int64_t ldb, float sb, int fmt_b,
                        double* acc, double* S);

double oracle_gelu(double z);
double oracle_dgelu(double z);
void   oracle_gelu_array(const double* z, double* y, int64_t n);
void   oracle_dgelu_array(const double* z, double* y, int64_t n);

/* column sums over all rows of a dense [M][N] double matrix: bgrad[j] = sum_i dz[i][j] */
void oracle_colsum(const double* dz, int64_t M, int64_t N, double* out);

/* bias gradient reduced from the weight-gradient GEMM's 1x128-scaled fp8
 * operand: out[r] = sum_k scale[k/128][r] dec(q[r][k]); S (or NULL) the sum of
 * the magnitudes */
void oracle_operand_rowsum(int fmt, const uint8_t* q, int64_t ldq, const float* scale, int64_t scale_ld,
                           int64_t rows, int64_t K, double* out, double* S);

int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
