/*
 * fp8ll.h -- C ABI of the block-scaled FP8 linear-layer GEMM library (sm_103a).
 *
 * The library computes the GEMMs of a training linear layer Y = X W^T + b with
 * fp8 operands that carry one fp32 scale per row per 128-element block of the
 * contraction dimension:
 *
 *   fp8_quantize        bf16 -> e4m3 / e5m2 codes + block scales
 *   fp8_quantize_dual   both orientations of that cast from one read
 *   fp8_quantize_dbias  the transposed cast of a gradient with its bias gradient
 *   fp8_mx_*            the MXFP8 variant (power-of-two scales per 32 values)
 *   fp8_tensor_*        per-tensor scaling (current or delayed amax)
 *   fp8_gemm_fprop      C = A B^T with bias / tanh-GELU epilogues, bf16 out
 *   fp8_gemm_dgrad      C = A B^T times gelu'(Z), optional bias-gradient sums
 *   fp8_gemm_dgrad_quant  the same, also casting its bf16 output (e5m2 rows)
 *   fp8_gemm_wgrad      fp32 out (+)= A B^T
 *   fp8_grouped_wgrad   per-group fp32 out_g (+)= A_g B_g^T, groups along K
 *   fp8_bgrad_from_operand  bias gradient as row sums of a 1x128-scaled operand
 *
 * Conventions shared by every entry point
 *   - One row-major "NT" convention: C[M][N] = A[M][K] . B[N][K]^T; both
 *     operands are K-contiguous ("nt" on "Weight gradient kernels for dense
 *     and MoE models").  Output features are N, so a bias has length N.
 *   - Scales are fp32, laid out [K/128][scale_ld]: scale[kb * scale_ld + r] is
 *     the scale of block kb of row r; scale_ld >= rows and scale_ld % 4 == 0
 *     (fp8_scale_ld(rows) gives the smallest legal value).
 *   - All pointers except k_sizes are DEVICE pointers owned by the caller.  The
 *     library never allocates, frees or synchronizes, except that
 *     fp8_get_device_status synchronizes the given stream.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).
 *   - Return value: FP8LL_OK (0) or a negative FP8LL_ERR_* code.  Arguments are
 *     validated on the host before anything is launched; an invalid call
 *     launches nothing and leaves every buffer untouched.
 *   - Kernels never trap.  A pipeline wait that runs past its time budget
 *     records FP8LL_ERR_TIMEOUT in a device status word, which
 *     fp8_get_device_status reports.
 */
#ifndef FP8LL_H
#define FP8LL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp8ll_stream_t; /* same type as cudaStream_t */

/* fp8 formats: e4m3 for the forward GEMM, e5m2 for gradients ("FP8 GEMM for
 * the fprop should use fast accumulation").  OCP FP8 bit layouts; e4m3 has no
 * infinity (max 448), e5m2 max 57344. */
enum { FP8LL_E4M3 = 0, FP8LL_E5M2 = 1 };

/* Epilogues ("Replaced cublasLt calls with rocblas gemm + 6 manually crafted
 * epilogues": BIAS, GELU and bias-gradient epilogues; bias length is the
 * output-feature count).
 *   NONE        fprop: Y = C
 *   BIAS        fprop: Y = C + bias[j]
 *   BIAS_GELU   fprop: Z = C + bias[j]; Y = gelu(Z); aux = Z (pre-activation)
 *   DGELU       dgrad: dZ = C * gelu'(aux)
 *   DGELU_BGRAD dgrad: dZ as DGELU, and bgrad[j] = sum_i dZ[i][j] (fp32)
 * gelu is the tanh form 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))). */
enum {
    FP8LL_EPI_NONE = 0,
    FP8LL_EPI_BIAS = 1,
    FP8LL_EPI_BIAS_GELU = 2,
    FP8LL_EPI_DGELU = 3,
    FP8LL_EPI_DGELU_BGRAD = 4
};

/* Accumulation precision, an explicit per-call flag ("FP8 GEMM for the fprop
 * should use fast accumulation": DEFAULT = fast, HIGHEST = full).
 *   FULL: each 128-deep K block's fp32 partial product is promoted into the
 *         fp32 accumulator with its own scale pair as soon as it is ready.
 *   FAST: accepted on every GEMM and runs the FULL promotion: results are
 *         bit-identical to FULL, inside the FAST bound.  With one fp32 scale
 *         per row per 128-element block, every block's partial product must
 *         meet its own scale pair (applying one block's pair to a window of
 *         blocks is off by the ratio of their scales), and promoting several
 *         blocks in one batch needs more tensor-memory accumulators than the
 *         512 columns hold at 256-column output tiles. */
enum { FP8LL_ACC_FULL = 0, FP8LL_ACC_FAST = 1 };

enum {
    FP8LL_OK = 0,
    FP8LL_ERR_INVALID_ARG = -1,      /* null / misaligned pointer, bad size, bad enum */
    FP8LL_ERR_UNSUPPORTED_DEVICE = -2, /* current device is not sm_103 */
    FP8LL_ERR_LAUNCH = -3,           /* a CUDA launch or driver call failed */
    FP8LL_ERR_TIMEOUT = -4,          /* a kernel pipeline wait ran out of time */
    FP8LL_ERR_WORKSPACE = -5,        /* workspace missing or too small */
    FP8LL_ERR_SCRATCH = -6           /* fp8_gemm_dgrad_noalloc: the built-in scratch array could not be set up */
};

/* One fp8 operand: codes q[rows][ld_q] (row stride ld_q bytes, K contiguous)
 * and scales scale[K/128][scale_ld].  q and scale must be 16-byte aligned,
 * ld_q % 16 == 0.  fmt is FP8LL_E4M3 or FP8LL_E5M2. */
typedef struct {
    const uint8_t* q;
    const float* scale;
    int64_t ld_q;
    int64_t scale_ld;
    int32_t fmt;
    int32_t reserved;
} fp8ll_operand_t;

/* Smallest legal scale leading dimension for `rows` rows: rows rounded up to
 * a multiple of 4 (16-byte rows for the TMA engine). */
int64_t fp8_scale_ld(int64_t rows);

/* Per-128-block cast of a bf16 matrix ("Weight gradient kernels for dense and
 * MoE models": the per-token cast applied to both operands before the
 * weight-gradient GEMM).  For each block of 128 values:
 *   amax = max|x|; inv = fl32(FMAX / amax); scale = fl32(amax / FMAX);
 *   q = round-to-nearest-even, saturating fp8 encode of fl32(x * inv)
 * with FMAX = 448 (e4m3) or 57344 (e5m2); a block whose amax is 0, or whose
 * FMAX / amax overflows fp32, gets inv = scale = 1.
 *   x:        bf16 [rows][ldx], 16-byte aligned, ldx % 8 == 0, ldx >= cols.
 *   transpose = 0: blocks run along each row (cols % 128 == 0).
 *             q [rows][cols] (row stride cols), scale [cols/128][scale_ld],
 *             scale_ld >= rows.
 *   transpose = 1: blocks run down each column (rows % 128 == 0,
 *             cols % 8 == 0).  q is the transposed matrix [cols][rows] (row
 *             stride rows), scale [rows/128][scale_ld], scale_ld >= cols.
 *             This produces the K-major operands of the weight-gradient
 *             GEMM, whose contraction runs over tokens.
 * rows == 0 or cols == 0 is a no-op. */
int fp8_quantize(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, int transpose,
                 uint8_t* q, float* scale, int64_t scale_ld, fp8ll_stream_t stream);

/* Both casts of fp8_quantize from one read of x: the row-blocked codes
 * (transpose = 0) for the GEMMs that contract over the columns of x and the
 * column-blocked, transposed codes (transpose = 1) for the weight-gradient
 * GEMM that contracts over its rows.  "Weight gradient kernels for dense and
 * MoE models" notes that separate cast launches around the GEMMs cost
 * end-to-end time; here the activations that feed both GEMMs are read once
 * instead of twice.  The outputs are bit-identical to the two separate
 * fp8_quantize calls with the same fmt.
 *   x:          bf16 [rows][ldx], 16-byte aligned, ldx % 8 == 0, ldx >= cols,
 *               rows % 128 == 0, cols % 128 == 0, rows / 128 <= 65535.
 *   q_rows:     [rows][cols];  scale_rows: [cols/128][scale_ld_rows],
 *               scale_ld_rows >= rows.
 *   q_cols:     [cols][rows];  scale_cols: [rows/128][scale_ld_cols],
 *               scale_ld_cols >= cols.
 * All outputs 16-byte aligned, scale leading dimensions % 4 == 0; the four
 * output buffers must not overlap each other or x.  rows == 0 or cols == 0
 * is a no-op. */
int fp8_quantize_dual(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q_rows,
                      float* scale_rows, int64_t scale_ld_rows, uint8_t* q_cols, float* scale_cols,
                      int64_t scale_ld_cols, fp8ll_stream_t stream);

/* Element-wise fp32 -> fp8 code conversion with the same round-to-nearest-
 * even, saturating conversion the quantize kernel applies after scaling (no
 * scaling here).  x, q: device, n elements.  For conformance tests of the
 * device encoder; NaN inputs give a NaN code. */
int fp8_cast_f32(const float* x, int64_t n, int fmt, uint8_t* q, fp8ll_stream_t stream);

/* Forward GEMM ("Replaced cublasLt calls ...": Y = X W^T + b with X (m,k),
 * W (n,k), bias of length n; e4m3 operands per "FP8 GEMM for the fprop should
 * use fast accumulation").
 *   C[i][j] = sum_kb sA[kb][i] sB[kb][j] sum_{k in kb} qA[i][k] qB[j][k]
 *   A: M x K operand (X), B: N x K operand (W); K % 128 == 0, K >= 128.
 *   epi: FP8LL_EPI_NONE, _BIAS or _BIAS_GELU.  bias_bf16: [N] (required for
 *   BIAS / BIAS_GELU, ignored for NONE).  out_bf16: [M][N] contiguous.
 *   aux_bf16: [M][N] receives Z = C + bias for BIAS_GELU (may be NULL; not the
 *   out_bf16 buffer), unused otherwise.  acc_mode: FP8LL_ACC_FULL or _FAST.
 *   M, N >= 1, any value. */
int fp8_gemm_fprop(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                   const void* bias_bf16, int epi, int acc_mode, void* out_bf16, void* aux_bf16,
                   fp8ll_stream_t stream);

/* Bytes of workspace fp8_gemm_dgrad needs for FP8LL_EPI_DGELU_BGRAD: one fp32
 * partial column sum per 32-row band of C (each promotion warp of a 128-row
 * tile writes its own band), 4 * ceil(M/128) * N * 4 bytes. */
size_t fp8_workspace_size(int64_t M, int64_t N);

/* Data-gradient GEMM with the GELU-derivative epilogue ("Replaced cublasLt
 * calls ...": backward of bias + GELU, derivative first, then the bias
 * gradient as a column sum in fp32).
 *   C = A B^T as in fp8_gemm_fprop (A: the incoming gradient, e5m2 typically;
 *   B: the weight operand).  aux_bf16: Z [M][N], the stored pre-activation.
 *   out_bf16: dZ = C * gelu'(Z), bf16 [M][N].
 *   epi = FP8LL_EPI_DGELU_BGRAD also writes bgrad [N] (fp32, length N, the
 *   sum over all M rows of the fp32 dZ before rounding) using `workspace`
 *   (device, >= fp8_workspace_size(M, N) bytes, 16-byte aligned); the sum is
 *   deterministic (fixed order).  epi = FP8LL_EPI_DGELU ignores bgrad and the
 *   workspace. */
int fp8_gemm_dgrad(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                   const void* aux_bf16, int epi, int acc_mode, void* out_bf16, float* bgrad, void* workspace,
                   size_t workspace_bytes, fp8ll_stream_t stream);

/* The data-gradient GEMM that also casts its own output for the next GEMM:
 * fp8_gemm_dgrad with FP8LL_EPI_DGELU (dZ = C * gelu'(Z), bf16 [M][N] in
 * out_bf16) plus the e5m2 codes and 1x128 scales of that stored bf16 dZ,
 * blocked along N -- exactly fp8_quantize(dZ, M, N, N, FP8LL_E5M2, 0, q,
 * scale, scale_ld), which the input-gradient GEMM dX = dZ W consumes.
 * "Weight gradient kernels for dense and MoE models" notes that separate cast
 * launches around the GEMMs cost end-to-end time; here the cast rides on the
 * epilogue that already holds dZ.
 *   N % 128 == 0 (each 128-column block of a row lies in one output tile).
 *   q: [M][N] codes, 16-byte aligned; scale: [N/128][scale_ld] fp32, 16-byte
 *   aligned, scale_ld >= M, scale_ld % 4 == 0.  q and scale may overlap
 *   neither each other nor dZ or Z.  Other arguments as fp8_gemm_dgrad. */
int fp8_gemm_dgrad_quant(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                         const void* aux_bf16, int acc_mode, void* out_bf16, uint8_t* q, float* scale,
                         int64_t scale_ld, fp8ll_stream_t stream);

/* fp8_gemm_dgrad for callers that cannot allocate device memory -- a runtime
 * whose allocator owns all device memory and forbids allocations after
 * start-up, a step replayed from a fixed memory plan, or a C caller with no
 * device allocator.  (The pages have no counterpart: this is a convenience of
 * this library.)  Same arguments and results as fp8_gemm_dgrad, minus the
 * workspace: the bias-gradient partials go to a fixed 16 MiB array inside the
 * library, held by every GPU that loads the library until the process exits.
 *   - Arguments are checked exactly as fp8_gemm_dgrad checks them, and a bad
 *     call gets the same code from both.  Sizes with fp8_workspace_size(M, N)
 *     > 16 MiB (4 * ceil(M/128) * N > 4 Mi partial sums) are then refused
 *     with FP8LL_ERR_WORKSPACE before any launch.
 *   - The first call on each device looks up the array's device address with
 *     that device current and keeps it.  Under lazy module loading (the CUDA
 *     default) this first call is when the CUDA runtime loads the library
 *     part that holds the array and reserves its 16 MiB: make it at start-up,
 *     before the caller's own allocator takes the device's memory, and before
 *     any stream capture.  If the runtime cannot provide the array, the call
 *     returns FP8LL_ERR_SCRATCH.  The kept address does not survive
 *     cudaDeviceReset (reload the library after a reset).
 *   - All calls share the one array: calls that overlap on the GPU (for
 *     example on two streams) race on it.  No clearing is needed between
 *     calls; every partial read is written by the same call first.
 *   - The call itself allocates nothing and calls no allocating routine. */
int fp8_gemm_dgrad_noalloc(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                           const void* aux_bf16, int epi, int acc_mode, void* out_bf16, float* bgrad,
                           fp8ll_stream_t stream);

/* Weight-gradient GEMM ("Weight gradient kernels for dense and MoE models":
 * fp8 x fp8 -> fp32, out += a b^T).
 *   out: fp32 [M][N] contiguous, 16-byte aligned.
 *   accumulate = 1: out[i][j] += C[i][j]  (the page's semantics; calling twice
 *                   adds twice -- the call is not idempotent)
 *   accumulate = 0: out[i][j]  = C[i][j]
 *   K % 128 == 0; K == 0 leaves out unchanged (accumulate = 1) or zeroes it. */
int fp8_gemm_wgrad(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                   float* out, int accumulate, int acc_mode, fp8ll_stream_t stream);

/* k-grouped weight gradient for MoE experts ("Weight gradient kernels for
 * dense and MoE models", grouped table): group g owns K columns
 * [off_g, off_g + k_sizes[g]) of both operands, off_g = sum of earlier sizes,
 * and out_g = out + g * M * N:
 *   out_g (+)= A[:, off_g : off_g + K_g] . B[:, off_g : off_g + K_g]^T
 *   k_sizes: HOST array of G values, each >= 0 and % 128 == 0.  A zero-size
 *   group leaves out_g unchanged (accumulate = 1) or zeroes it.
 *   1 <= G <= 256.  A.ld_q, B.ld_q >= sum of k_sizes. */
int fp8_grouped_wgrad(int G, int64_t M, int64_t N, const int64_t* k_sizes, const fp8ll_operand_t* A,
                      const fp8ll_operand_t* B, float* out, int accumulate, int acc_mode, fp8ll_stream_t stream);

/* The transposed cast of a gradient together with its bias gradient (db =
 * sum(dY, axis=0) of "Replaced cublasLt calls with rocblas gemm + 6 manually
 * crafted epilogues", taken from the bf16 values while they are cast for the
 * weight-gradient GEMM, so the data-gradient GEMM needs no column sums):
 *   q_cols / scale_cols: exactly fp8_quantize(x, ..., transpose = 1) -- codes
 *     [cols][rows], scales [rows/128][scale_ld_cols];
 *   q_rows / scale_rows: NULL, or exactly the row cast (fp8_quantize_dual's
 *     row outputs; needs cols % 128 == 0);
 *   dbias: fp32 [cols], dbias[c] = sum over all rows of x[r][c].
 * rows % 128 == 0, cols % 8 == 0, ldx >= cols, ldx % 8 == 0.  rows == 0 sets
 * dbias to zero.  workspace: >= (rows/128) * cols * 4 bytes, 16-byte aligned
 * (fp8_workspace_size(rows, cols) is enough), else FP8LL_ERR_WORKSPACE; it
 * holds per-128-row partial sums and may overlap none of x, the codes, the
 * scales or dbias (FP8LL_ERR_INVALID_ARG).  The sums run in
 * fp32 in a fixed order (each 128-row block, then the blocks): deterministic. */
int fp8_quantize_dbias(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q_cols,
                       float* scale_cols, int64_t scale_ld_cols, uint8_t* q_rows, float* scale_rows,
                       int64_t scale_ld_rows, float* dbias, void* workspace, size_t workspace_bytes,
                       fp8ll_stream_t stream);

/* Bias gradient reduced from the weight-gradient GEMM's gradient operand
 * (the BGRADB epilogue on "Replaced cublasLt calls with rocblas gemm + 6
 * manually crafted epilogues": db is taken together with dW by reducing the
 * gradient operand over that GEMM's k, the tokens).  For A the [rows][K]
 * operand dZ^T (features x tokens, from the transposed cast of dZ):
 *   db[r] (+)= sum_kb A.scale[kb][r] * sum_{k in block kb} dec(A.q[r][k])
 *   db: fp32 [rows], 4-byte aligned; it may overlap neither A's codes nor its
 *       scales (FP8LL_ERR_INVALID_ARG).
 *   accumulate = 1: db[r] += the sum; 0: db[r] = the sum.
 *   K % 128 == 0; K == 0 gives a sum of 0.  rows == 0 is a no-op.
 * The sums run in fp32 in a fixed order: results are deterministic.  This is
 * the alternative to the bias-gradient sums of fp8_gemm_dgrad's
 * FP8LL_EPI_DGELU_BGRAD, which add up the fp32 dZ before any fp8 rounding;
 * this one adds up the fp8 values the weight gradient consumes. */
int fp8_bgrad_from_operand(int64_t rows, int64_t K, const fp8ll_operand_t* A, float* db, int accumulate,
                           fp8ll_stream_t stream);

/* ------------------------------------------------------------------ MXFP8
 * The MX block format, named among the fp8 recipes on "How can we use
 * te.Linear with weight parallel?": one power-of-two scale per 32 consecutive
 * K-elements of every operand row, applied by the tensor core itself
 * (block-scaled MMA), so the fp32 accumulation runs over the whole K range
 * with no software promotion.  Scale of a block: 2^e with e the smallest
 * integer in [-127, 127] such that amax <= FMAX * 2^e (no element saturates;
 * e = 0 for an all-zero block); codes: round-to-nearest-even, saturating fp8
 * of x * 2^-e.
 *
 * Scale storage (UE8M0 bytes, e + 127), the layout the GEMM copies into
 * tensor memory unchanged: for an operand with `rows` rows and K columns,
 * G = 2 * ceil(rows / 256) groups of 128 rows; K block kb (128 elements),
 * row r = 128 * g + rr, 32-element group k in 0..3 of the block:
 *   sf[(kb * G + g) * 512 + (rr % 32) * 16 + (rr / 32) * 4 + k]
 * Bytes of rows beyond the operand hold 127 (scale 1). */
typedef struct {
    const uint8_t* q;  /* codes [rows][ld_q], K contiguous; 16-byte aligned */
    const uint8_t* sf; /* scale bytes, fp8_mx_sf_bytes(rows, K) of them; 16-byte aligned */
    int64_t ld_q;      /* >= K, multiple of 16 */
    int32_t fmt;
    int32_t reserved;
} fp8ll_mx_operand_t;

/* Bytes of scale storage for an operand of `rows` rows and `k` columns
 * (k % 128 == 0); 0 for invalid sizes. */
size_t fp8_mx_sf_bytes(int64_t rows, int64_t k);

/* MXFP8 cast of a bf16 matrix x [rows][cols] (row stride ldx elements,
 * ldx % 8 == 0).  transpose = 0: blocks along each row, q [rows][cols],
 * cols % 128 == 0, sf for (rows, cols).  transpose = 1: blocks down each
 * column, q [cols][rows] (the transpose), rows % 128 == 0, cols % 8 == 0, sf
 * for (cols, rows).  Codes and scales are bit-exact against the definition
 * above.  Caller-owned device buffers; asynchronous on `stream`. */
int fp8_mx_quantize(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, int transpose, uint8_t* q,
                    uint8_t* sf, fp8ll_stream_t stream);

/* MXFP8 GEMMs: the three GEMMs above with MX operands, the same epilogues,
 * shapes, layouts and error codes (no accumulation mode: the tensor core
 * applies every block's scales):
 *   fp8_mx_gemm_fprop: out = epi(A . B^T + bias), epi NONE / BIAS / BIAS_GELU
 *   fp8_mx_gemm_dgrad: out = (A . B^T) * gelu'(aux), bias gradient as in
 *                      fp8_gemm_dgrad (same workspace size)
 *   fp8_mx_gemm_wgrad: out (+)= A . B^T, fp32
 * K % 128 == 0; M, N >= 1. */
int fp8_mx_gemm_fprop(int64_t M, int64_t N, int64_t K, const fp8ll_mx_operand_t* A, const fp8ll_mx_operand_t* B,
                      const void* bias_bf16, int epi, void* out_bf16, void* aux_bf16, fp8ll_stream_t stream);
int fp8_mx_gemm_dgrad(int64_t M, int64_t N, int64_t K, const fp8ll_mx_operand_t* A, const fp8ll_mx_operand_t* B,
                      const void* aux_bf16, int epi, void* out_bf16, float* bgrad, void* workspace,
                      size_t workspace_bytes, fp8ll_stream_t stream);
int fp8_mx_gemm_wgrad(int64_t M, int64_t N, int64_t K, const fp8ll_mx_operand_t* A, const fp8ll_mx_operand_t* B,
                      float* out, int accumulate, fp8ll_stream_t stream);

/* fp8_mx_quantize(x, ..., transpose = 1) together with the bias gradient of
 * x's columns, dbias[c] = sum over all rows of x[r][c] (as fp8_quantize_dbias,
 * for the MXFP8 recipe's transposed cast of the gradient).  Codes and scale
 * bytes are exactly fp8_mx_quantize's; rows % 128 == 0, cols % 8 == 0;
 * rows == 0 sets dbias to zero.  workspace: >= (rows/128) * cols * 4 bytes,
 * 16-byte aligned, overlapping none of x, q, sf or dbias.  The sums run in the same fixed order
 * as fp8_quantize_dbias's, so the two give the same bits for the same x. */
int fp8_mx_quantize_dbias(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q,
                          uint8_t* sf, float* dbias, void* workspace, size_t workspace_bytes, fp8ll_stream_t stream);

/* ---- per-tensor scaling ----------------------------------------------------
 * "FP8 GEMM for the fprop should use fast accumulation" casts whole tensors
 * with one scale each.  The cast takes the amax to scale with from the caller:
 * the tensor's own (fp8_tensor_amax first: "current scaling") or the largest
 * amax of earlier steps (fp8_amax_history_update: "delayed scaling", where
 * values above it saturate).  For a given amax A:
 *   inv = fl32(FMAX / A); scale = fl32(A / FMAX); q = RNE-saturating fp8
 *   encode of fl32(x * inv)
 * (A = 0, or FMAX / A overflowing fp32: inv = scale = 1).  With one scale per
 * operand, the GEMM accumulates the raw fp8 products over all of K in the
 * tensor core's fp32 accumulator and multiplies once by fl32(sA * sB): no
 * promotion inside the K loop.
 *   q:     codes [rows][ld_q], K-contiguous, 16-byte aligned, ld_q % 16 == 0.
 *   scale: DEVICE pointer to the operand's one fp32 scale (4-byte aligned). */
typedef struct {
    const uint8_t* q;
    const float* scale;
    int64_t ld_q;
    int32_t fmt;
    int32_t reserved;
} fp8ll_tensor_operand_t;

/* *amax = max|x| over a bf16 [rows][ldx] matrix (x 16-byte aligned, cols % 8
 * == 0, ldx % 8 == 0, ldx >= cols); 0 for an empty matrix. */
int fp8_tensor_amax(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, float* amax,
                    fp8ll_stream_t stream);

/* Per-tensor cast with the amax in *amax_in (device).  Outputs (at least one):
 *   q_rows [rows][cols] (cols % 16 == 0), q_cols the transposed codes
 *   [cols][rows] (rows % 128 == 0, rows / 128 <= 65535, cols % 8 == 0); both
 *   together need cols % 128 == 0 and read x once.
 * *scale receives the dequantization scale (a word of its own: not amax_in or
 * amax_out).  amax_out (may be NULL, must not be amax_in): receives max|x| of
 * this x, for the history of the next step.
 * x as in fp8_tensor_amax.  rows == 0 or cols == 0 is a no-op. */
int fp8_tensor_quantize(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, const float* amax_in,
                        uint8_t* q_rows, uint8_t* q_cols, float* scale, float* amax_out, fp8ll_stream_t stream);

/* Delayed scaling, for `count` tensors at once (device pointers): history
 * [count][len] row h <- (amax_new[h], history[h][0 .. len-2]), then
 * amax_use[h] = the largest entry of row h.  count >= 1, len >= 1. */
int fp8_amax_history_update(float* history, int64_t count, int64_t len, const float* amax_new, float* amax_use,
                            fp8ll_stream_t stream);

/* The three GEMMs of fp8_gemm_fprop / fp8_gemm_dgrad / fp8_gemm_wgrad (same
 * shapes, epilogues, layouts and errors) on per-tensor scaled operands:
 *   C[i][j] = fl32(sA * sB) * sum_k qA[i][k] qB[j][k]. */
int fp8_tensor_gemm_fprop(int64_t M, int64_t N, int64_t K, const fp8ll_tensor_operand_t* A,
                          const fp8ll_tensor_operand_t* B, const void* bias_bf16, int epi, void* out_bf16,
                          void* aux_bf16, fp8ll_stream_t stream);
int fp8_tensor_gemm_dgrad(int64_t M, int64_t N, int64_t K, const fp8ll_tensor_operand_t* A,
                          const fp8ll_tensor_operand_t* B, const void* aux_bf16, int epi, void* out_bf16, float* bgrad,
                          void* workspace, size_t workspace_bytes, fp8ll_stream_t stream);
int fp8_tensor_gemm_wgrad(int64_t M, int64_t N, int64_t K, const fp8ll_tensor_operand_t* A,
                          const fp8ll_tensor_operand_t* B, float* out, int accumulate, fp8ll_stream_t stream);

/* Synchronizes `stream`, then returns and clears the device status word of
 * the current device: FP8LL_OK, or the first FP8LL_ERR_TIMEOUT recorded by a
 * kernel since the last call; FP8LL_ERR_LAUNCH if CUDA reports an error. */
int fp8_get_device_status(fp8ll_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* fp8_status_string(int code);

/* Test hook: for the next launch only, the GEMM producer issues no loads, so
 * the pipeline waits run out after `budget_ms` milliseconds and the kernel
 * returns early with FP8LL_ERR_TIMEOUT recorded.  Nothing is written to the
 * GEMM outputs in that launch.  Returns FP8LL_OK. */
int fp8_debug_starve_next_gemm(int budget_ms);

#ifdef __cplusplus
}
#endif
#endif /* FP8LL_H */
