// quantize.cu -- bf16 -> fp8 (e4m3 / e5m2) per-128-block cast kernels.
//
// "Weight gradient kernels for dense and MoE models" casts both GEMM operands
// per token with one fp32 scale per 128 elements before the fp8 GEMM; the
// per-block rule implemented here (and in the oracle, independently) is
//   amax = max|x|, inv = fl32(FMAX/amax), scale = fl32(amax/FMAX),
//   q = RNE-saturating fp8(fl32(x * inv)),
// with inv = scale = 1 for a block whose amax is 0 or whose FMAX/amax
// overflows fp32.  Division and multiplication are IEEE round-to-nearest
// (__fdiv_rn / __fmul_rn, no flush-to-zero), so codes and scales are
// bit-reproducible.
//
// Both kernels are HBM-bound: 2 bytes read + 1 byte + 4/128 bytes written per
// element.
#include <cfloat>
#include <cstdint>
#include <cuda_runtime.h>

#include "cast_rule.cuh"
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8ll {

// 8 values -> 8 codes packed little-endian in a uint2
template <int FMT>
__device__ __forceinline__ uint2 encode8(const float (&f)[8], float inv) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = encode2<FMT>(f[2 * i], f[2 * i + 1], inv);
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// ------------------------------------------------------------------ row-wise
// A half-warp owns one (row, 128-block) task: 16 lanes x 16 bytes of bf16.
// Consecutive tasks are consecutive blocks of a row, so a warp reads 512
// contiguous bytes.  Each warp keeps U task pairs in flight.  When the rows
// are packed (ldx == cols) the flat task index addresses input and output
// directly; the (row, block) split -- a division -- is needed only for the
// scale, by one lane per task, in 32-bit arithmetic when the task count fits.
template <int FMT, int U, bool PACKED>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ldx, uint8_t* __restrict__ q,
                                                            float* __restrict__ scale, int64_t sld) {
    const int64_t nb = cols / 128;
    const int64_t total = rows * nb;
    const bool small = total <= 0xFFFFFFFFll;
    const int lane = threadIdx.x & 31;
    const int hl = lane & 15;
    const int hw = lane >> 4;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

    for (int64_t base = warp * 2 * U; base < total; base += nwarps * 2 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t task = base + 2 * u + hw;
            v[u] = make_uint4(0, 0, 0, 0);
            if (task < total) {
                const uint16_t* src;
                if (PACKED) {
                    src = x + task * 128 + hl * 8;
                } else {
                    const int64_t r = task / nb;
                    src = x + r * ldx + (task - r * nb) * 128 + hl * 8;
                }
                v[u] = __ldcs(reinterpret_cast<const uint4*>(src));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t task = base + 2 * u + hw;
            float f[8];
            f[0] = bf16_lo(v[u].x); f[1] = bf16_hi(v[u].x);
            f[2] = bf16_lo(v[u].y); f[3] = bf16_hi(v[u].y);
            f[4] = bf16_lo(v[u].z); f[5] = bf16_hi(v[u].z);
            f[6] = bf16_lo(v[u].w); f[7] = bf16_hi(v[u].w);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            float inv, s;
            block_scale<FMT>(amax, inv, s);
            const uint2 codes = encode8<FMT>(f, inv);
            if (task < total) {
                // q is always packed: row r, block b starts at (r * nb + b) * 128 = task * 128
                *reinterpret_cast<uint2*>(q + task * 128 + hl * 8) = codes;
                if (hl == 0) {
                    int64_t r, b;
                    if (small) {
                        const uint32_t t32 = static_cast<uint32_t>(task), nb32 = static_cast<uint32_t>(nb);
                        const uint32_t r32 = t32 / nb32;
                        r = r32;
                        b = t32 - r32 * nb32;
                    } else {
                        r = task / nb;
                        b = task - r * nb;
                    }
                    scale[b * sld + r] = s;
                }
            }
        }
    }
}

// --------------------------------------------------------------- transposed
// Blocks run down columns: output row c of q (= input column c) gets 128
// contiguous codes per 128-row block.  A CTA casts 128-row x 128-column tiles
// of x staged in shared memory as 64 words per row (bf16 pairs), each 32-row
// band rotated by 8 words so that the column-wise reads of the four 32-row
// parts hit 32 distinct banks.  Two kernels stage the tiles:
//   quantize_cols_kernel       one tile per CTA, four CTAs per SM (three when
//                              it writes column codes only): each thread
//                              loads its eight 16-byte pieces into registers,
//                              so the row-blocked cast (ROWS) and the tensor's
//                              amax (TENSOR) are taken from the loaded values.
//   quantize_cols_pipe_kernel  persistent, three CTAs per SM, two staged
//                              tiles: while a CTA casts one tile the next one
//                              streams in by cp.async; for the casts that only
//                              write the column-blocked codes (plain and with
//                              the bias-gradient sums), where it measured
//                              faster (5608 -> 5750 and 4579 -> 5515 GB/s at
//                              32768 x 8192).  Reading the staged tile back for
//                              the row codes made the two-way cast slower
//                              (5078 -> 4561), hence the first kernel there.
//
// With ROWS the CTA also writes the row-blocked cast of its tile (128 columns
// = one block per row; codes qr [rows][cols], scales sr [cols/128][sldr]):
// after the loads each half-warp holds one row's 128 values in registers, so
// the row amax (a half-warp butterfly), scale and codes need no second read
// of x.  The arithmetic is the row kernel's, so the codes are the same.
//
// With TENSOR the tile is cast with the one per-tensor scale instead (from the
// given amax: inv = fl32(FMAX/amax), scale = fl32(amax/FMAX); "FP8 GEMM for
// the fprop should use fast accumulation" scales whole tensors): no block amax,
// `scale` receives the single scale (written by the first CTA), sr is unused,
// and when amax_out is given the CTA folds max|x| of its tile into it.
// With DBIAS the cast also takes the bias gradient of x's columns (the
// gradient at the layer's pre-activation, cast down its columns for the
// weight gradient): db = sum over rows of x ("Replaced cublasLt calls with
// rocblas gemm + 6 manually crafted epilogues", db = sum(dY, axis=0), taken
// from the high-precision values before the fp8 rounding).  The amax pass adds
// each thread's 32 values of a column in row order, the quad combines its four
// parts with the amax pass's shuffles, and one lane writes the tile's partial
// sum to dpart[row block][c]; a finalize adds the row blocks in a fixed order.

// The column-blocked cast of one staged tile (rows r0.., columns c0.., row
// block rb) for the persistent kernel: thread t handles column pair t / 4 and
// 32-row part t % 4.  Two passes over the staged tile (amax, then encode)
// instead of holding 64 values in registers.  quantize_cols_kernel below does
// the same arithmetic inline (as a shared function it measured 2-6% slower
// there).
template <int FMT, bool DBIAS>
__device__ __forceinline__ void cast_tile_cols(const uint32_t (*tile)[64], int64_t rows, int64_t cols, int64_t r0,
                                               int64_t c0, int64_t rb, uint8_t* __restrict__ q,
                                               float* __restrict__ scale, int64_t sld, float* __restrict__ dpart) {
    const int cp = threadIdx.x >> 2;  // column pair 0..63
    const int p = threadIdx.x & 3;    // 32-row part
    const int64_t c = c0 + 2 * cp;
    float amax_lo = 0.0f, amax_hi = 0.0f;
    float sum_lo = 0.0f, sum_hi = 0.0f;  // DBIAS
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t w = tile[32 * p + i][(cp + 8 * p) & 63];
        amax_lo = fmaxf(amax_lo, fabsf(bf16_lo(w)));
        amax_hi = fmaxf(amax_hi, fabsf(bf16_hi(w)));
        if (DBIAS) {
            sum_lo = __fadd_rn(sum_lo, bf16_lo(w));
            sum_hi = __fadd_rn(sum_hi, bf16_hi(w));
        }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        amax_lo = fmaxf(amax_lo, __shfl_xor_sync(0xffffffffu, amax_lo, off));
        amax_hi = fmaxf(amax_hi, __shfl_xor_sync(0xffffffffu, amax_hi, off));
        if (DBIAS) {
            // a + b on one lane, b + a on its partner: the same bits on all four
            sum_lo = __fadd_rn(sum_lo, __shfl_xor_sync(0xffffffffu, sum_lo, off));
            sum_hi = __fadd_rn(sum_hi, __shfl_xor_sync(0xffffffffu, sum_hi, off));
        }
    }
    float inv_lo, s_lo, inv_hi, s_hi;
    block_scale<FMT>(amax_lo, inv_lo, s_lo);
    block_scale<FMT>(amax_hi, inv_hi, s_hi);
    if (DBIAS && p == 0 && c < cols) {
        // cols is even: c + 1 < cols too
        dpart[rb * cols + c] = sum_lo;
        dpart[rb * cols + c + 1] = sum_hi;
    }
    if (c < cols) {
        uint32_t wl[8], wh[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t lo16[2], hi16[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t w0 = tile[32 * p + 4 * i + 2 * j][(cp + 8 * p) & 63];
                const uint32_t w1 = tile[32 * p + 4 * i + 2 * j + 1][(cp + 8 * p) & 63];
                lo16[j] = Fp8Fmt<FMT>::cvt2(__fmul_rn(bf16_lo(w0), inv_lo), __fmul_rn(bf16_lo(w1), inv_lo));
                hi16[j] = Fp8Fmt<FMT>::cvt2(__fmul_rn(bf16_hi(w0), inv_hi), __fmul_rn(bf16_hi(w1), inv_hi));
            }
            wl[i] = lo16[0] | (lo16[1] << 16);
            wh[i] = hi16[0] | (hi16[1] << 16);
        }
        uint4* dl = reinterpret_cast<uint4*>(q + c * rows + r0 + 32 * p);
        uint4* dh = reinterpret_cast<uint4*>(q + (c + 1) * rows + r0 + 32 * p);
        dl[0] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        dl[1] = make_uint4(wl[4], wl[5], wl[6], wl[7]);
        dh[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        dh[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
        if (p == 0) {
            scale[rb * sld + c] = s_lo;
            scale[rb * sld + c + 1] = s_hi;
        }
    }
}

// place of word 4 ch (16-byte piece ch, 0..15) of tile row rr in the stage
__device__ __forceinline__ int staged_word(int rr, int ch) { return (ch * 4 + 8 * (rr >> 5)) & 63; }

template <int FMT, bool ROWS, bool TENSOR, bool DBIAS = false>
__global__ void __launch_bounds__(256, ROWS ? 4 : 3) quantize_cols_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ldx, uint8_t* __restrict__ q,
                                                            float* __restrict__ scale, int64_t sld,
                                                            uint8_t* __restrict__ qr, float* __restrict__ sr,
                                                            int64_t sldr, const float* __restrict__ amax_in,
                                                            unsigned* __restrict__ amax_out,
                                                            float* __restrict__ dpart = nullptr) {
    static_assert(!(DBIAS && TENSOR), "the bias-gradient sums ride on the block-amax pass");
    __shared__ __align__(16) uint32_t tile[128][64];
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
    float inv_t = 1.0f, s_t = 1.0f;
    if (TENSOR) {
        block_scale<FMT>(*amax_in, inv_t, s_t);
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *scale = s_t;
    }

    // thread t, iteration it: row (t + 256 it) / 16 of the tile, columns
    // 8 ((t + 256 it) % 16) .. +7; all eight loads are issued first
    uint4 v[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int i = threadIdx.x + it * 256;
        const int64_t c = c0 + (i & 15) * 8;
        v[it] = make_uint4(0, 0, 0, 0);
        if (c < cols) v[it] = __ldcs(reinterpret_cast<const uint4*>(x + (r0 + (i >> 4)) * ldx + c));
    }
    float tmax = 0.0f;  // TENSOR: max|x| over this thread's loads
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int i = threadIdx.x + it * 256;
        const int rr = i >> 4;
        const int ch = i & 15;
        const int w = (ch * 4 + 8 * (rr >> 5)) & 63;
        *reinterpret_cast<uint4*>(&tile[rr][w]) = v[it];
        if (ROWS || (TENSOR && amax_out)) {
            const float f[8] = {bf16_lo(v[it].x), bf16_hi(v[it].x), bf16_lo(v[it].y), bf16_hi(v[it].y),
                                bf16_lo(v[it].z), bf16_hi(v[it].z), bf16_lo(v[it].w), bf16_hi(v[it].w)};
            float amax = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
            if (TENSOR) {
                tmax = fmaxf(tmax, amax);
                if (ROWS) *reinterpret_cast<uint2*>(qr + (r0 + rr) * cols + c0 + ch * 8) = encode8<FMT>(f, inv_t);
            } else {
#pragma unroll
                for (int off = 1; off <= 8; off <<= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                float inv, s;
                block_scale<FMT>(amax, inv, s);
                *reinterpret_cast<uint2*>(qr + (r0 + rr) * cols + c0 + ch * 8) = encode8<FMT>(f, inv);
                if (ch == 0) sr[(c0 >> 7) * sldr + r0 + rr] = s;
            }
        }
    }
    __shared__ float warp_max[8];
    if (TENSOR && amax_out) {
#pragma unroll
        for (int off = 1; off <= 16; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = tmax;
    }
    __syncthreads();
    if (TENSOR && amax_out && threadIdx.x == 0) {
        // one atomic per CTA (thousands of CTAs finish together); non-negative
        // floats order like their bit patterns
        float m = warp_max[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) m = fmaxf(m, warp_max[i]);
        atomicMax(amax_out, __float_as_uint(m));
    }

    const int cp = threadIdx.x >> 2;  // column pair 0..63
    const int p = threadIdx.x & 3;    // 32-row part
    const int64_t c = c0 + 2 * cp;
    // two passes over the staged tile (amax, then encode) instead of holding
    // 64 values in registers: the lower register count keeps more tiles, and
    // so more loads, in flight per SM
    float inv_lo = inv_t, s_lo = s_t, inv_hi = inv_t, s_hi = s_t;
    if (!TENSOR) {
        float amax_lo = 0.0f, amax_hi = 0.0f;
        float sum_lo = 0.0f, sum_hi = 0.0f;  // DBIAS
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t w = tile[32 * p + i][(cp + 8 * p) & 63];
            amax_lo = fmaxf(amax_lo, fabsf(bf16_lo(w)));
            amax_hi = fmaxf(amax_hi, fabsf(bf16_hi(w)));
            if (DBIAS) {
                sum_lo = __fadd_rn(sum_lo, bf16_lo(w));
                sum_hi = __fadd_rn(sum_hi, bf16_hi(w));
            }
        }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            amax_lo = fmaxf(amax_lo, __shfl_xor_sync(0xffffffffu, amax_lo, off));
            amax_hi = fmaxf(amax_hi, __shfl_xor_sync(0xffffffffu, amax_hi, off));
            if (DBIAS) {
                // a + b on one lane, b + a on its partner: the same bits on all four
                sum_lo = __fadd_rn(sum_lo, __shfl_xor_sync(0xffffffffu, sum_lo, off));
                sum_hi = __fadd_rn(sum_hi, __shfl_xor_sync(0xffffffffu, sum_hi, off));
            }
        }
        block_scale<FMT>(amax_lo, inv_lo, s_lo);
        block_scale<FMT>(amax_hi, inv_hi, s_hi);
        if (DBIAS && p == 0 && c < cols) {
            // cols is even: c + 1 < cols too
            dpart[static_cast<int64_t>(blockIdx.y) * cols + c] = sum_lo;
            dpart[static_cast<int64_t>(blockIdx.y) * cols + c + 1] = sum_hi;
        }
    }
    if (c < cols) {
        uint32_t wl[8], wh[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t lo16[2], hi16[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint32_t w0 = tile[32 * p + 4 * i + 2 * k][(cp + 8 * p) & 63];
                const uint32_t w1 = tile[32 * p + 4 * i + 2 * k + 1][(cp + 8 * p) & 63];
                lo16[k] = Fp8Fmt<FMT>::cvt2(__fmul_rn(bf16_lo(w0), inv_lo), __fmul_rn(bf16_lo(w1), inv_lo));
                hi16[k] = Fp8Fmt<FMT>::cvt2(__fmul_rn(bf16_hi(w0), inv_hi), __fmul_rn(bf16_hi(w1), inv_hi));
            }
            wl[i] = lo16[0] | (lo16[1] << 16);
            wh[i] = hi16[0] | (hi16[1] << 16);
        }
        uint4* dl = reinterpret_cast<uint4*>(q + c * rows + r0 + 32 * p);
        uint4* dh = reinterpret_cast<uint4*>(q + (c + 1) * rows + r0 + 32 * p);
        dl[0] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        dl[1] = make_uint4(wl[4], wl[5], wl[6], wl[7]);
        dh[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        dh[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
        if (!TENSOR && p == 0) {
            scale[static_cast<int64_t>(blockIdx.y) * sld + c] = s_lo;
            scale[static_cast<int64_t>(blockIdx.y) * sld + c + 1] = s_hi;
        }
    }
}

constexpr int kPipeCtas = 3;                                    // CTAs per SM
constexpr size_t kPipeSmem = 2 * 128 * 64 * sizeof(uint32_t);  // two staged tiles

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    // src_bytes 0 fills the 16 bytes with zeros and reads nothing
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <int FMT, bool DBIAS>
__global__ void __launch_bounds__(256, kPipeCtas) quantize_cols_pipe_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* __restrict__ q,
    float* __restrict__ scale, int64_t sld, float* __restrict__ dpart) {
    extern __shared__ __align__(16) uint32_t stage[];  // [2][128][64]
    const int64_t ncb = (cols + 127) / 128;
    const int64_t ntiles = (rows / 128) * ncb;

    // thread t, copy it: row (t + 256 it) / 16 of the tile, columns
    // 8 ((t + 256 it) % 16) .. +7, to its rotated place in the stage
    auto fetch = [&](int64_t t, int buf) {
        const int64_t rb = t / ncb;
        const int64_t r0 = rb * 128, c0 = (t - rb * ncb) * 128;
        const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(stage)) + buf * (128 * 64 * 4);
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int i = threadIdx.x + it * 256;
            const int rr = i >> 4;
            const int ch = i & 15;
            const int64_t c = c0 + ch * 8;
            const bool in = c < cols;
            cp_async16(base + (rr * 64 + staged_word(rr, ch)) * 4, x + (r0 + rr) * ldx + (in ? c : 0),
                       in ? 16u : 0u);
        }
    };

    int64_t t = blockIdx.x;
    if (t < ntiles) fetch(t, 0);
    cp_async_commit();
    for (int k = 0; t < ntiles; ++k, t += gridDim.x) {
        const uint32_t(*tile)[64] = reinterpret_cast<const uint32_t(*)[64]>(stage + (k & 1) * 128 * 64);
        // every thread is done with the previous tile: its stage is refilled now
        __syncthreads();
        if (t + gridDim.x < ntiles) fetch(t + gridDim.x, (k + 1) & 1);
        cp_async_commit();
        cp_async_wait_all_but_one();  // this thread's copies of this tile have landed
        __syncthreads();              // ... and every thread's
        const int64_t rb = t / ncb;
        cast_tile_cols<FMT, DBIAS>(tile, rows, cols, rb * 128, (t - rb * ncb) * 128, rb, q, scale, sld, dpart);
    }
}

// The column-blocked cast (with ROWS also the row-blocked one): the one-tile
// kernel where rows or a per-tensor scale are involved, the persistent one
// otherwise.
template <int FMT, bool ROWS, bool TENSOR, bool DBIAS>
int launch_cols(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q, float* scale, int64_t sld,
                uint8_t* qr, float* sr, int64_t sldr, const float* amax_in, unsigned* amax_out, float* dpart,
                cudaStream_t stream, int num_sms) {
    if constexpr (ROWS || TENSOR) {
        dim3 grid(static_cast<unsigned>((cols + 127) / 128), static_cast<unsigned>(rows / 128));
        quantize_cols_kernel<FMT, ROWS, TENSOR, DBIAS><<<grid, 256, 0, stream>>>(x, rows, cols, ldx, q, scale, sld, qr,
                                                                                sr, sldr, amax_in, amax_out, dpart);
        return cudaGetLastError() == cudaSuccess ? 0 : -3;
    } else {
        auto kern = quantize_cols_pipe_kernel<FMT, DBIAS>;
        static unsigned long long configured = 0;  // one bit per device ordinal
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -3;
        if (!(configured & (1ull << dev))) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kPipeSmem)) !=
                cudaSuccess)
                return -3;
            configured |= 1ull << dev;
        }
        const int64_t ntiles = (rows / 128) * ((cols + 127) / 128);
        if (ntiles == 0) return 0;
        const int64_t cap = static_cast<int64_t>(num_sms) * kPipeCtas;
        const unsigned grid = static_cast<unsigned>(ntiles < cap ? ntiles : cap);
        kern<<<grid, 256, kPipeSmem, stream>>>(x, rows, cols, ldx, q, scale, sld, dpart);
        return cudaGetLastError() == cudaSuccess ? 0 : -3;
    }
}

// --------------------------------------------------------------- per-tensor
// max|x| over a bf16 matrix: each warp walks rows, its lanes 16 bytes apart
// along the row; one atomic max per warp on the bit pattern (non-negative
// floats order like their bits), into a word the launcher zeroed first.
__global__ void __launch_bounds__(256) tensor_amax_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                          int64_t cols, int64_t ldx, unsigned* __restrict__ amax) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * 8;
    float m = 0.0f;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); r < rows; r += warps) {
        const uint16_t* row = x + r * ldx;
#pragma unroll 4
        for (int64_t c = 8 * lane; c < cols; c += 256) {
            const uint4 v = __ldcs(reinterpret_cast<const uint4*>(row + c));
            m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                               fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))));
            m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))),
                               fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)))));
        }
    }
#pragma unroll
    for (int off = 1; off <= 16; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) atomicMax(amax, __float_as_uint(m));
}

// Per-tensor cast along rows: q [rows][cols] (packed), 8 codes per lane from
// one 16-byte load, the scale from the given amax (the first thread stores it);
// with amax_out, max|x| of the tensor is folded in as in tensor_amax_kernel.
template <int FMT>
__global__ void __launch_bounds__(256) tensor_quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                   int64_t cols, int64_t ldx, const float* amax_in,
                                                                   uint8_t* __restrict__ q, float* scale,
                                                                   unsigned* amax_out) {
    float inv, s;
    block_scale<FMT>(*amax_in, inv, s);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * 8;
    float m = 0.0f;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); r < rows; r += warps) {
        const uint16_t* row = x + r * ldx;
#pragma unroll 4
        for (int64_t c = 8 * lane; c < cols; c += 256) {
            const uint4 v = __ldcs(reinterpret_cast<const uint4*>(row + c));
            const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                                bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
            for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(f[k]));
            *reinterpret_cast<uint2*>(q + r * cols + c) = encode8<FMT>(f, inv);
        }
    }
    if (amax_out) {
#pragma unroll
        for (int off = 1; off <= 16; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) atomicMax(amax_out, __float_as_uint(m));
    }
}

// For each of `count` histories h: history[h][len] <- (amax_new[h],
// history[h][0 .. len-2]) and amax_use[h] = its maximum.  One thread per
// history: each holds a handful of floats.
__global__ void amax_history_kernel(float* hist, int64_t count, int64_t len, const float* amax_new,
                                    float* amax_use) {
    const int64_t h = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (h >= count) return;
    float* row = hist + h * len;
    const float a = amax_new[h];
    for (int64_t i = len - 1; i > 0; --i) row[i] = row[i - 1];
    row[0] = a;
    float m = 0.0f;
    for (int64_t i = 0; i < len; ++i) m = fmaxf(m, row[i]);
    amax_use[h] = m;
}

// -------------------------------------------------------------------- MXFP8
// One power-of-two scale per 32 consecutive elements (the MX block format),
// e = the smallest integer in [-127, 127] with amax <= FMAX 2^e (no element
// saturates; 0 for an all-zero block), codes = fp8(x 2^-e) with a single
// rounding (scaling by a power of two is exact).  The scale bytes (UE8M0,
// e + 127) are written in the layout the GEMM copies into tensor memory:
// 512-byte atoms per (128-element K block kb, 128-row group g), row
// r = 128 g + rr and 32-element group k of the block at byte
//   (kb * G + g) * 512 + (rr % 32) * 16 + (rr / 32) * 4 + k,
// G = 2 * ceil(rows / 256) (an even number of groups, so that the two atoms of
// a 256-row tile are adjacent).  Bytes of rows beyond the matrix are 127.

template <int FMT>
__device__ __forceinline__ int mx_exponent(float amax) {
    // FMAX = 1.75 * 2^F; amax = (1 + m) 2^(E - 127) <= 1.75 2^(F + e)
    //   <=> e >= E - 127 - F + (m > 0.75)
    constexpr int F = (FMT == 0) ? 8 : 15;
    const uint32_t b = __float_as_uint(amax);
    if (b == 0u) return 0;
    const int E = static_cast<int>(b >> 23);
    if (E == 0) return -127;  // subnormal amax: far below FMAX 2^-127
    int e = E - 127 - F + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    e = e < -127 ? -127 : e;
    return e > 127 ? 127 : e;
}

// 2^-e as an fp32 (2^-127 is subnormal)
__device__ __forceinline__ float mx_inverse_scale(int e) {
    return e < 127 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : __uint_as_float(0x400000u);
}

__device__ __forceinline__ int64_t mx_sf_offset(int64_t kb, int64_t groups, int64_t r, int k) {
    const int64_t rr = r & 127;
    return (kb * groups + (r >> 7)) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + k;
}

// Rows: a half-warp per (row, 128-block) task as in the 1x128 cast; lane l of
// the half holds elements 8l..8l+7, so lanes 4k..4k+3 form MX group k.
template <int FMT, int U, bool PACKED>
__global__ void __launch_bounds__(256) mx_quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                               int64_t cols, int64_t ldx, uint8_t* __restrict__ q,
                                                               uint8_t* __restrict__ sf, int64_t groups) {
    const int64_t nb = cols / 128;
    const int64_t total = rows * nb;
    const int lane = threadIdx.x & 31;
    const int hl = lane & 15;
    const int hw = lane >> 4;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp * 2 * U; base < total; base += nwarps * 2 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t task = base + 2 * u + hw;
            v[u] = make_uint4(0, 0, 0, 0);
            if (task < total) {
                const uint16_t* src;
                if (PACKED) {
                    src = x + task * 128 + hl * 8;
                } else {
                    const int64_t r = task / nb;
                    src = x + r * ldx + (task - r * nb) * 128 + hl * 8;
                }
                v[u] = __ldcs(reinterpret_cast<const uint4*>(src));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t task = base + 2 * u + hw;
            float f[8];
            f[0] = bf16_lo(v[u].x); f[1] = bf16_hi(v[u].x);
            f[2] = bf16_lo(v[u].y); f[3] = bf16_hi(v[u].y);
            f[4] = bf16_lo(v[u].z); f[5] = bf16_hi(v[u].z);
            f[6] = bf16_lo(v[u].w); f[7] = bf16_hi(v[u].w);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int e = mx_exponent<FMT>(amax);
            const uint2 codes = encode8<FMT>(f, mx_inverse_scale(e));
            if (task < total) {
                *reinterpret_cast<uint2*>(q + task * 128 + hl * 8) = codes;
                if ((hl & 3) == 0) {
                    int64_t r, b;
                    if (total <= 0xFFFFFFFFll) {
                        const uint32_t t32 = static_cast<uint32_t>(task), nb32 = static_cast<uint32_t>(nb);
                        const uint32_t r32 = t32 / nb32;
                        r = r32;
                        b = t32 - r32 * nb32;
                    } else {
                        r = task / nb;
                        b = task - r * nb;
                    }
                    sf[mx_sf_offset(b, groups, r, hl >> 2)] = static_cast<uint8_t>(e + 127);
                }
            }
        }
    }
}

// Transposed: the 1x128 kernel's staged 128 x 128 tile; a thread's 32 rows of
// a column are exactly one MX group (group p of the 128-token block).
// With DBIAS the cast also adds each thread's 32 values of a column (one MX
// block) in row order and combines the quad's four parts, in the same order as
// the 1x128 transposed cast, so the per-128-row partials in dpart (and the
// bias gradient the finalize makes of them) are bit-identical to that cast's.
template <int FMT, bool DBIAS = false>
__global__ void __launch_bounds__(256, 3) mx_quantize_cols_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                  int64_t cols, int64_t ldx, uint8_t* __restrict__ q,
                                                                  uint8_t* __restrict__ sf, int64_t groups,
                                                                  float* __restrict__ dpart = nullptr) {
    __shared__ __align__(16) uint32_t tile[128][64];
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int i = threadIdx.x + it * 256;
        const int rr = i >> 4;
        const int ch = i & 15;
        const int64_t c = c0 + ch * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (c < cols) v = __ldcs(reinterpret_cast<const uint4*>(x + (r0 + rr) * ldx + c));
        const int w = (ch * 4 + 8 * (rr >> 5)) & 63;
        *reinterpret_cast<uint4*>(&tile[rr][w]) = v;
    }
    __syncthreads();
    const int cp = threadIdx.x >> 2;
    const int p = threadIdx.x & 3;
    const int64_t c = c0 + 2 * cp;
    float amax_lo = 0.0f, amax_hi = 0.0f;
    float sum_lo = 0.0f, sum_hi = 0.0f;  // DBIAS
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t w = tile[32 * p + i][(cp + 8 * p) & 63];
        amax_lo = fmaxf(amax_lo, fabsf(bf16_lo(w)));
        amax_hi = fmaxf(amax_hi, fabsf(bf16_hi(w)));
        if (DBIAS) {
            sum_lo = __fadd_rn(sum_lo, bf16_lo(w));
            sum_hi = __fadd_rn(sum_hi, bf16_hi(w));
        }
    }
    if (DBIAS) {
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            sum_lo = __fadd_rn(sum_lo, __shfl_xor_sync(0xffffffffu, sum_lo, off));
            sum_hi = __fadd_rn(sum_hi, __shfl_xor_sync(0xffffffffu, sum_hi, off));
        }
        if (p == 0 && c < cols) {  // cols is even: c + 1 < cols too
            dpart[static_cast<int64_t>(blockIdx.y) * cols + c] = sum_lo;
            dpart[static_cast<int64_t>(blockIdx.y) * cols + c + 1] = sum_hi;
        }
    }
    const int e_lo = mx_exponent<FMT>(amax_lo), e_hi = mx_exponent<FMT>(amax_hi);
    const float inv_lo = mx_inverse_scale(e_lo), inv_hi = mx_inverse_scale(e_hi);
    if (c < cols) {
        uint32_t wl[8], wh[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t lo16[2], hi16[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint32_t w0 = tile[32 * p + 4 * i + 2 * k][(cp + 8 * p) & 63];
                const uint32_t w1 = tile[32 * p + 4 * i + 2 * k + 1][(cp + 8 * p) & 63];
                lo16[k] = Fp8Fmt<FMT>::cvt2(__fmul_rn(bf16_lo(w0), inv_lo), __fmul_rn(bf16_lo(w1), inv_lo));
                hi16[k] = Fp8Fmt<FMT>::cvt2(__fmul_rn(bf16_hi(w0), inv_hi), __fmul_rn(bf16_hi(w1), inv_hi));
            }
            wl[i] = lo16[0] | (lo16[1] << 16);
            wh[i] = hi16[0] | (hi16[1] << 16);
        }
        uint4* dl = reinterpret_cast<uint4*>(q + c * rows + r0 + 32 * p);
        uint4* dh = reinterpret_cast<uint4*>(q + (c + 1) * rows + r0 + 32 * p);
        dl[0] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        dl[1] = make_uint4(wl[4], wl[5], wl[6], wl[7]);
        dh[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        dh[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
        sf[mx_sf_offset(blockIdx.y, groups, c, p)] = static_cast<uint8_t>(e_lo + 127);
        sf[mx_sf_offset(blockIdx.y, groups, c + 1, p)] = static_cast<uint8_t>(e_hi + 127);
    }
}

// ---------------------------------------------------------------- plain cast
template <int FMT>
__global__ void cast_f32_kernel(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ q) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 4;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i < n; i += stride) {
        if (i + 4 <= n) {
            const float4 v = *reinterpret_cast<const float4*>(x + i);
            const uint32_t a = Fp8Fmt<FMT>::cvt2(v.x, v.y);
            const uint32_t b = Fp8Fmt<FMT>::cvt2(v.z, v.w);
            *reinterpret_cast<uint32_t*>(q + i) = a | (b << 16);
        } else {
            for (int64_t k = i; k < n; ++k) q[k] = static_cast<uint8_t>(Fp8Fmt<FMT>::cvt2(x[k], 0.0f) & 0xFF);
        }
    }
}

// -------------------------------------------------------------- host launch

int launch_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, int transpose, uint8_t* q,
                    float* scale, int64_t sld, cudaStream_t stream, int num_sms) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    if (!transpose) {
        constexpr int U = 4;
        const int64_t total = rows * (cols / 128);
        const int64_t pairs = (total + 1) / 2;
        int64_t blocks = (pairs + 8 * U - 1) / (8 * U);
        const int64_t cap = static_cast<int64_t>(num_sms) * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        const unsigned g = static_cast<unsigned>(blocks);
        const bool packed = ldx == cols;
        if (fmt == 0) {
            if (packed)
                quantize_rows_kernel<0, U, true><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, q, scale, sld);
            else
                quantize_rows_kernel<0, U, false><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, q, scale, sld);
        } else {
            if (packed)
                quantize_rows_kernel<1, U, true><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, q, scale, sld);
            else
                quantize_rows_kernel<1, U, false><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, q, scale, sld);
        }
    } else {
        return fmt == 0 ? launch_cols<0, false, false, false>(xb, rows, cols, ldx, q, scale, sld, nullptr, nullptr, 0,
                                                              nullptr, nullptr, nullptr, stream, num_sms)
                        : launch_cols<1, false, false, false>(xb, rows, cols, ldx, q, scale, sld, nullptr, nullptr, 0,
                                                              nullptr, nullptr, nullptr, stream, num_sms);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q_rows,
                         float* scale_rows, int64_t sld_rows, uint8_t* q_cols, float* scale_cols, int64_t sld_cols,
                         cudaStream_t stream, int num_sms) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    return fmt == 0 ? launch_cols<0, true, false, false>(xb, rows, cols, ldx, q_cols, scale_cols, sld_cols, q_rows,
                                                         scale_rows, sld_rows, nullptr, nullptr, nullptr, stream,
                                                         num_sms)
                    : launch_cols<1, true, false, false>(xb, rows, cols, ldx, q_cols, scale_cols, sld_cols, q_rows,
                                                         scale_rows, sld_rows, nullptr, nullptr, nullptr, stream,
                                                         num_sms);
}

int launch_quantize_dbias(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q_cols,
                          float* scale_cols, int64_t sld_cols, uint8_t* q_rows, float* scale_rows, int64_t sld_rows,
                          float* dpart, float* dbias, cudaStream_t stream, int num_sms) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    int rc;
    if (q_rows)
        rc = fmt == 0 ? launch_cols<0, true, false, true>(xb, rows, cols, ldx, q_cols, scale_cols, sld_cols, q_rows,
                                                          scale_rows, sld_rows, nullptr, nullptr, dpart, stream, num_sms)
                      : launch_cols<1, true, false, true>(xb, rows, cols, ldx, q_cols, scale_cols, sld_cols, q_rows,
                                                          scale_rows, sld_rows, nullptr, nullptr, dpart, stream, num_sms);
    else
        rc = fmt == 0 ? launch_cols<0, false, false, true>(xb, rows, cols, ldx, q_cols, scale_cols, sld_cols, nullptr,
                                                           nullptr, 0, nullptr, nullptr, dpart, stream, num_sms)
                      : launch_cols<1, false, false, true>(xb, rows, cols, ldx, q_cols, scale_cols, sld_cols, nullptr,
                                                           nullptr, 0, nullptr, nullptr, dpart, stream, num_sms);
    if (rc != 0) return rc;
    return launch_bgrad_finalize(dpart, rows / 128, cols, dbias, stream, num_sms);
}

static int grid_rows(int64_t rows, int num_sms) {
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
    return static_cast<int>(blocks < 1 ? 1 : blocks);
}

int launch_tensor_amax(const void* x, int64_t rows, int64_t cols, int64_t ldx, float* amax, cudaStream_t stream,
                       int num_sms) {
    if (cudaMemsetAsync(amax, 0, sizeof(float), stream) != cudaSuccess) return -3;
    tensor_amax_kernel<<<grid_rows(rows, num_sms), 256, 0, stream>>>(static_cast<const uint16_t*>(x), rows, cols,
                                                                     ldx, reinterpret_cast<unsigned*>(amax));
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_tensor_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, const float* amax_in,
                           uint8_t* q_rows, uint8_t* q_cols, float* scale, float* amax_out, cudaStream_t stream,
                           int num_sms) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    unsigned* am = reinterpret_cast<unsigned*>(amax_out);
    if (am && cudaMemsetAsync(am, 0, sizeof(float), stream) != cudaSuccess) return -3;
    if (q_cols) {
        if (q_rows)
            return fmt == 0 ? launch_cols<0, true, true, false>(xb, rows, cols, ldx, q_cols, scale, 0, q_rows, nullptr,
                                                                0, amax_in, am, nullptr, stream, num_sms)
                            : launch_cols<1, true, true, false>(xb, rows, cols, ldx, q_cols, scale, 0, q_rows, nullptr,
                                                                0, amax_in, am, nullptr, stream, num_sms);
        return fmt == 0 ? launch_cols<0, false, true, false>(xb, rows, cols, ldx, q_cols, scale, 0, nullptr, nullptr, 0,
                                                             amax_in, am, nullptr, stream, num_sms)
                        : launch_cols<1, false, true, false>(xb, rows, cols, ldx, q_cols, scale, 0, nullptr, nullptr, 0,
                                                             amax_in, am, nullptr, stream, num_sms);
    } else {
        const int g = grid_rows(rows, num_sms);
        if (fmt == 0)
            tensor_quantize_rows_kernel<0><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, amax_in, q_rows, scale, am);
        else
            tensor_quantize_rows_kernel<1><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, amax_in, q_rows, scale, am);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_amax_history(float* hist, int64_t count, int64_t len, const float* amax_new, float* amax_use,
                        cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((count + 127) / 128);
    amax_history_kernel<<<blocks, 128, 0, stream>>>(hist, count, len, amax_new, amax_use);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int64_t mx_sf_groups(int64_t rows) { return 2 * ((rows + 255) / 256); }

int launch_mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, int transpose, uint8_t* q,
                       uint8_t* sf, cudaStream_t stream, int num_sms) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    // rows of the quantized operand and its K extent
    const int64_t orows = transpose ? cols : rows;
    const int64_t kext = transpose ? rows : cols;
    const int64_t groups = mx_sf_groups(orows);
    if (orows % 256 != 0) {
        // rows beyond the matrix in the last group pair read as scale 1
        if (cudaMemsetAsync(sf, 127, static_cast<size_t>(kext / 128) * groups * 512, stream) != cudaSuccess)
            return -3;
    }
    if (!transpose) {
        constexpr int U = 4;
        const int64_t total = rows * (cols / 128);
        int64_t blocks = ((total + 1) / 2 + 8 * U - 1) / (8 * U);
        const int64_t cap = static_cast<int64_t>(num_sms) * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        const unsigned g = static_cast<unsigned>(blocks);
        const bool packed = ldx == cols;
        if (fmt == 0) {
            if (packed)
                mx_quantize_rows_kernel<0, U, true><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, q, sf, groups);
            else
                mx_quantize_rows_kernel<0, U, false><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, q, sf, groups);
        } else {
            if (packed)
                mx_quantize_rows_kernel<1, U, true><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, q, sf, groups);
            else
                mx_quantize_rows_kernel<1, U, false><<<g, 256, 0, stream>>>(xb, rows, cols, ldx, q, sf, groups);
        }
    } else {
        dim3 grid(static_cast<unsigned>((cols + 127) / 128), static_cast<unsigned>(rows / 128));
        if (fmt == 0)
            mx_quantize_cols_kernel<0><<<grid, 256, 0, stream>>>(xb, rows, cols, ldx, q, sf, groups);
        else
            mx_quantize_cols_kernel<1><<<grid, 256, 0, stream>>>(xb, rows, cols, ldx, q, sf, groups);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_mx_quantize_dbias(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q,
                             uint8_t* sf, float* dpart, float* dbias, cudaStream_t stream, int num_sms) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    const int64_t groups = mx_sf_groups(cols);
    if (cols % 256 != 0) {
        // rows beyond the matrix in the last group pair read as scale 1
        if (cudaMemsetAsync(sf, 127, static_cast<size_t>(rows / 128) * groups * 512, stream) != cudaSuccess)
            return -3;
    }
    dim3 grid(static_cast<unsigned>((cols + 127) / 128), static_cast<unsigned>(rows / 128));
    if (fmt == 0)
        mx_quantize_cols_kernel<0, true><<<grid, 256, 0, stream>>>(xb, rows, cols, ldx, q, sf, groups, dpart);
    else
        mx_quantize_cols_kernel<1, true><<<grid, 256, 0, stream>>>(xb, rows, cols, ldx, q, sf, groups, dpart);
    if (cudaGetLastError() != cudaSuccess) return -3;
    return launch_bgrad_finalize(dpart, rows / 128, cols, dbias, stream, num_sms);
}

int launch_cast_f32(const float* x, int64_t n, int fmt, uint8_t* q, cudaStream_t stream, int num_sms) {
    int64_t blocks = (n + 1023) / 1024;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (fmt == 0)
        cast_f32_kernel<0><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, n, q);
    else
        cast_f32_kernel<1><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, n, q);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace fp8ll
