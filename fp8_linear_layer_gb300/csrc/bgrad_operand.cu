// bgrad_operand.cu -- bias gradient reduced from the weight-gradient GEMM's
// fp8 operand.
//
// "Replaced cublasLt calls with rocblas gemm + 6 manually crafted epilogues"
// (the backward pass; the BGRADB epilogue) takes db together with dW by
// reducing the gradient operand of the weight-gradient GEMM over that GEMM's
// k, the tokens.  With the operand cast by 1x128 blocks,
//   db[r] = (accumulate ? db[r] : 0) + sum_kb scale[kb][r] sum_{k in kb} dec(q[r][k]).
//
// HBM-bound: K code bytes + 4 K/128 scale bytes read and 4 bytes written per
// row.  A CTA of 256 threads takes two rows at a time, four warps to a row,
// and walks over row pairs with a stride of the grid (one wave of resident
// CTAs).  A warp reads 512-byte chunks of its row (16 contiguous bytes a lane,
// so lanes 8b..8b+7 hold one 128-byte block), four chunks a group, and issues
// the next group's loads before it adds up the current one.  Codes become f16
// exactly (e5m2 is the high byte of an f16: a byte permute; e4m3: cvt), and
// each f16 is added to an fp32 sum by the mixed-precision add, which converts
// exactly and rounds once.  The sums run in a fixed order (four chains of four
// codes and a tree per 16 bytes, the groups in turn, a butterfly over the
// lanes, the four warps of a row in turn), so results are deterministic.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"

namespace fp8ll {
namespace {

constexpr int kRowsPerCta = 2;
constexpr int kWarpsPerRow = 4;
constexpr int kChunksPerGroup = 4;
constexpr int kThreadsPerCta = kRowsPerCta * kWarpsPerRow * 32;

// two fp8 codes (bytes 0-1 or 2-3 of w) -> their values as one f16x2
template <int FMT, int HALF>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t w) {
    uint32_t r;
    if constexpr (FMT == 1) {
        // e5m2 -> f16: the code is the f16's high byte, the low byte is zero
        asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(w), "n"(HALF ? 0x3424 : 0x1404));
    } else {
        const uint16_t v = static_cast<uint16_t>(HALF ? (w >> 16) : (w & 0xFFFFu));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    }
    return r;
}

// acc + lo + hi of an f16x2, each added exactly converted, one rounding each
__device__ __forceinline__ float add_f16x2(uint32_t x, float acc) {
    float r;
    asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 t;\n\tmov.b32 {l, h}, %1;\n\t"
        "add.rn.f32.f16 t, l, %2;\n\tadd.rn.f32.f16 %0, h, t;\n\t}"
        : "=f"(r)
        : "r"(x), "f"(acc));
    return r;
}

// the sum of 16 consecutive codes: a chain of four per 32-bit word, then a tree
template <int FMT>
__device__ __forceinline__ float sum16(const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = add_f16x2(fp8x2_to_f16x2<FMT, 1>(w[i]), add_f16x2(fp8x2_to_f16x2<FMT, 0>(w[i]), 0.0f));
    return (c[0] + c[1]) + (c[2] + c[3]);
}

struct Group {
    uint4 v[kChunksPerGroup];
    float s[kChunksPerGroup];
};

// group g of this warp's share of row r: chunks c = 16 g + 4 u + w; a
// segment past the row (or a row past the operand) reads as zero
__device__ __forceinline__ void load_group(Group& G, const uint8_t* __restrict__ q, int64_t ldq,
                                           const float* __restrict__ scale, int64_t sld, int64_t rows, int64_t nseg,
                                           int64_t r, int64_t g, int w, int lane) {
#pragma unroll
    for (int u = 0; u < kChunksPerGroup; ++u) {
        const int64_t j = ((g * kChunksPerGroup + u) * kWarpsPerRow + w) * 32 + lane;
        if (r < rows && j < nseg) {
            G.v[u] = __ldg(reinterpret_cast<const uint4*>(q + r * ldq) + j);
            G.s[u] = __ldg(scale + (j / 8) * sld + r);
        } else {
            G.v[u] = make_uint4(0u, 0u, 0u, 0u);
            G.s[u] = 0.0f;
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kThreadsPerCta) operand_rowsum_kernel(const uint8_t* __restrict__ q, int64_t ldq,
                                                                        const float* __restrict__ scale, int64_t sld,
                                                                        int64_t rows, int64_t K,
                                                                        float* __restrict__ db, int accumulate) {
    __shared__ float part[2][kRowsPerCta][kWarpsPerRow];  // by iteration parity
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rloc = warp / kWarpsPerRow, w = warp % kWarpsPerRow;
    const int64_t nseg = K / 16;  // 16-byte segments in a row
    const int64_t nchunk = (nseg + 31) / 32;
    const int64_t per_group = static_cast<int64_t>(kChunksPerGroup) * kWarpsPerRow;
    const int64_t ngroups = nchunk > 0 ? (nchunk + per_group - 1) / per_group : 1;
    const int64_t npairs = (rows + kRowsPerCta - 1) / kRowsPerCta;

    // every thread walks the same (pair, group) sequence: the barriers stay uniform
    int64_t pair = blockIdx.x, g = 0;
    Group nxt, cur;
    if (pair < npairs) load_group(nxt, q, ldq, scale, sld, rows, nseg, pair * kRowsPerCta + rloc, 0, w, lane);
    float acc = 0.0f;
    int it = 0;
    while (pair < npairs) {
        cur = nxt;
        const int64_t cur_pair = pair;
        const bool last = (g == ngroups - 1);
        if (++g == ngroups) {
            g = 0;
            pair += gridDim.x;
        }
        if (pair < npairs) load_group(nxt, q, ldq, scale, sld, rows, nseg, pair * kRowsPerCta + rloc, g, w, lane);
#pragma unroll
        for (int u = 0; u < kChunksPerGroup; ++u) acc = __fmaf_rn(cur.s[u], sum16<FMT>(cur.v[u]), acc);
        if (last) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
            if (lane == 0) part[it & 1][rloc][w] = acc;
            __syncthreads();
            if (threadIdx.x < kRowsPerCta) {
                const int64_t rr = cur_pair * kRowsPerCta + threadIdx.x;
                if (rr < rows) {
                    float total = part[it & 1][threadIdx.x][0];
#pragma unroll
                    for (int i = 1; i < kWarpsPerRow; ++i) total += part[it & 1][threadIdx.x][i];
                    db[rr] = accumulate ? db[rr] + total : total;
                }
            }
            acc = 0.0f;
            ++it;
        }
    }
}

template <int FMT>
int launch_fmt(const uint8_t* q, int64_t ldq, const float* scale, int64_t sld, int64_t rows, int64_t K, float* db,
               int accumulate, cudaStream_t stream, int num_sms) {
    // resident CTAs per SM, from the occupancy calculator once (callers on
    // several host threads may all compute it: they store the same value)
    static std::atomic<int> cached{0};
    int per_sm = cached.load(std::memory_order_relaxed);
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, operand_rowsum_kernel<FMT>, kThreadsPerCta, 0) !=
                cudaSuccess ||
            per_sm < 1)
            return -1;
        cached.store(per_sm, std::memory_order_relaxed);
    }
    const int64_t npairs = (rows + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t wave = static_cast<int64_t>(num_sms) * per_sm;
    const int64_t blocks = npairs < wave ? npairs : wave;
    if (blocks <= 0) return -1;
    operand_rowsum_kernel<FMT><<<static_cast<unsigned>(blocks), kThreadsPerCta, 0, stream>>>(q, ldq, scale, sld, rows,
                                                                                          K, db, accumulate);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_operand_rowsum(const uint8_t* q, int64_t ldq, const float* scale, int64_t sld, int fmt, int64_t rows,
                          int64_t K, float* db, int accumulate, cudaStream_t stream, int num_sms) {
    return fmt == 0 ? launch_fmt<0>(q, ldq, scale, sld, rows, K, db, accumulate, stream, num_sms)
                    : launch_fmt<1>(q, ldq, scale, sld, rows, K, db, accumulate, stream, num_sms);
}

}  // namespace fp8ll
