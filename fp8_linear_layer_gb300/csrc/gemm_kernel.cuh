// gemm_kernel.cuh -- persistent block-scaled FP8 GEMM for sm_103a (tcgen05 + TMA + TMEM).
//
// Computes, for every output tile, C[i][j] = sum_kb sA[kb][i] sB[kb][j] P_kb[i][j]
// with P_kb[i][j] = sum_{k in block kb} qA[i][k] qB[j][k] (raw fp8 products,
// fp32 in TMEM), i.e. the 1x128 block-scaled "nt" GEMM of "Weight gradient
// kernels for dense and MoE models", then applies one of the fused epilogues
// of "Replaced cublasLt calls with rocblas gemm + 6 manually crafted
// epilogues" (bias, tanh-GELU, GELU derivative, bias-gradient column sums) or
// the fp32 weight-gradient read-modify-write (out += C).
//
// CTA = 3 warpgroups (12 warps), one CTA per SM, persistent over a
// rasterized tile list of 128 x 256 output tiles:
//   warp 0      TMA producer: operand tiles (128 x 128 B of A, 256 x 128 B of
//               B, 128-byte swizzle) into a 4-stage ring, block scales into
//               an 8-stage ring.
//   warp 1      TMEM owner and MMA issuer: per K block, 4 x tcgen05.mma
//               (M=128, N=256, K=32, kind::f8f6f4) into one of two TMEM
//               accumulators (2 x 256 fp32 columns), so the MMAs of block
//               k+1 run while block k is promoted.  An N=256 MMA does twice
//               the work of an N=128 one for the same A operand read, and
//               the tensor core only reaches its full rate at this width.
//   warps 2-3   idle (they complete the first warpgroup).
//   warps 4-11  promotion + epilogue, two warpgroups of 128 columns each:
//               warp w reads TMEM lanes 32*(w%4)..+31 (its rows).  Per K
//               block a thread loads its raw fp32 partial sums in two
//               64-column TMEM loads, hands the buffer back to the MMA warp
//               after the second and adds sA*sB*P into a 128-wide fp32
//               register accumulator ("promotion") with packed fp32x2
//               multiplies and fmas.
// Registers: launched at kLaunchRegs per thread (the most 384 threads can
// have), the first warpgroup gives registers back (setmaxnreg.dec to
// kRegsCtrl) and the two epilogue warpgroups take them (setmaxnreg.inc to
// kRegsEpi); 128 * kRegsCtrl + 256 * kRegsEpi <= 384 * kLaunchRegs.  The host
// refuses to launch if the compiled kernel's register count differs from
// kLaunchRegs, so the split can never ask for more than the pool.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8ll {

constexpr int kBM = kTileM;
constexpr int kBN = kTileN;
constexpr int kBK = 128;  // K bytes per stage == one scale block
constexpr int kStages = 4;
constexpr int kSStages = 8;
constexpr int kEpiGroups = 2;               // epilogue warpgroups
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kFirstEpiWarp = 4;
constexpr int kThreads = 128 + 32 * kEpiWarps;
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtrl = 40;
constexpr int kRegsEpi = 232;
static_assert(128 * kRegsCtrl + 128 * kEpiGroups * kRegsEpi <= kThreads * kLaunchRegs,
              "register split exceeds the pool");
constexpr int kHalfN = kBN / kEpiGroups;  // columns per epilogue thread (128)
static_assert(kHalfN == 128, "two 64-column TMEM loads per thread and K block");
constexpr int kNumAcc = 2;               // TMEM accumulator buffers
constexpr uint32_t kTmemCols = 512;      // kNumAcc * kBN, a power of two
static_assert(kNumAcc * kBN <= 512, "TMEM capacity");
constexpr int kRasterM = 16;

struct __align__(1024) SmemLayout {
    uint8_t a[kStages][kBM * kBK];
    uint8_t b[kStages][kBN * kBK];
    float sa[kSStages][kBM];
    float sb[kSStages][kBN];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t sfull[kSStages];
    uint64_t sempty[kSStages];
    uint64_t acc_full[kNumAcc];
    uint64_t acc_empty[kNumAcc];
    uint64_t drain;
    uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(SmemLayout) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

template <int N>
__device__ __forceinline__ void ring_advance(int& idx, uint32_t& phase) {
    if (++idx == N) {
        idx = 0;
        phase ^= 1u;
    }
}

// tile index -> (group, m tile, n tile); within a group, bands of kRasterM
// row-tiles are walked column by column so that concurrently running CTAs
// share operand rows in L2.
__device__ __forceinline__ void decode_tile(const GemmParams& p, int t, int& g, int& mt, int& nt) {
    g = t / p.tiles_per_group;
    const int local = t - g * p.tiles_per_group;
    const int band_tiles = kRasterM * p.num_n_tiles;
    const int band = local / band_tiles;
    const int first_m = band * kRasterM;
    const int rem_m = p.num_m_tiles - first_m;
    const int bm = rem_m < kRasterM ? rem_m : kRasterM;
    const int r = local - band * band_tiles;
    mt = first_m + r % bm;
    nt = r / bm;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v) != 0; }

// ------------------------------------------------------------------ stores

// wgrad: out (+)= acc, fp32
// out += acc is a single fp32 add per element, done in L2 by a vector
// reduction (no load round trip; each element receives exactly one add per
// call, so the result is deterministic).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void store_wgrad(const GemmParams& p, int out_index, int r, int cbase,
                                            float2 (&acc)[kHalfN / 2]) {
    if (r >= p.M) return;
    float* orow = static_cast<float*>(p.out) + (static_cast<int64_t>(out_index) * p.M + r) * p.N + cbase;
    if ((p.N & 3) == 0 && cbase + kHalfN <= p.N) {
        if (p.accumulate) {
#pragma unroll
            for (int j = 0; j < kHalfN; j += 4)
                red_add_v4(orow + j, acc[j / 2].x, acc[j / 2].y, acc[j / 2 + 1].x, acc[j / 2 + 1].y);
        } else {
#pragma unroll
            for (int j = 0; j < kHalfN; j += 4)
                *reinterpret_cast<float4*>(orow + j) =
                    make_float4(acc[j / 2].x, acc[j / 2].y, acc[j / 2 + 1].x, acc[j / 2 + 1].y);
        }
    } else {
#pragma unroll
        for (int j = 0; j < kHalfN; ++j) {
            const float v = (j & 1) ? acc[j / 2].y : acc[j / 2].x;
            if (cbase + j < p.N) orow[j] = (p.accumulate ? orow[j] : 0.0f) + v;
        }
    }
}

// fprop: Z = acc + bias[j]; Y = gelu(Z) or Z; bf16 out (+ bf16 aux Z)
template <int EPI>
__device__ __forceinline__ void store_fprop(const GemmParams& p, int r, int cbase, float2 (&acc)[kHalfN / 2]) {
    if (r >= p.M) return;
    const int64_t off = static_cast<int64_t>(r) * p.N + cbase;
    uint16_t* out = static_cast<uint16_t*>(p.out) + off;
    uint16_t* aux = (EPI == kEpiBiasGelu && p.aux) ? static_cast<uint16_t*>(p.aux) + off : nullptr;
    const uint16_t* bias = static_cast<const uint16_t*>(p.bias) + cbase;
    if ((p.N & 7) == 0 && cbase + kHalfN <= p.N) {
#pragma unroll
        for (int j = 0; j < kHalfN; j += 8) {
            float z[8];
            if (EPI == kEpiNone) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    z[2 * i] = acc[j / 2 + i].x;
                    z[2 * i + 1] = acc[j / 2 + i].y;
                }
            } else {
                const uint4 bv = __ldg(reinterpret_cast<const uint4*>(bias + j));
                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    z[2 * i] = acc[j / 2 + i].x + bf16_lo(bw[i]);
                    z[2 * i + 1] = acc[j / 2 + i].y + bf16_hi(bw[i]);
                }
            }
            uint32_t yw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (EPI == kEpiBiasGelu)
                    yw[i] = pack_bf16x2(gelu_tanh(z[2 * i]), gelu_tanh(z[2 * i + 1]));
                else
                    yw[i] = pack_bf16x2(z[2 * i], z[2 * i + 1]);
            }
            *reinterpret_cast<uint4*>(out + j) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
            if (aux) {
                *reinterpret_cast<uint4*>(aux + j) =
                    make_uint4(pack_bf16x2(z[0], z[1]), pack_bf16x2(z[2], z[3]), pack_bf16x2(z[4], z[5]),
                               pack_bf16x2(z[6], z[7]));
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < kHalfN; ++j) {
            if (cbase + j < p.N) {
                float z = (j & 1) ? acc[j / 2].y : acc[j / 2].x;
                if (EPI != kEpiNone) z += __uint_as_float(static_cast<uint32_t>(bias[j]) << 16);
                const float y = (EPI == kEpiBiasGelu) ? gelu_tanh(z) : z;
                out[j] = static_cast<uint16_t>(pack_bf16x2(y, 0.0f) & 0xFFFFu);
                if (aux) aux[j] = static_cast<uint16_t>(pack_bf16x2(z, 0.0f) & 0xFFFFu);
            }
        }
    }
}

// Column sums of 32 consecutive columns over the 32 rows held by a warp:
// a butterfly that halves the column set at each step.  Afterwards lane l
// holds the sum for column l.  The summation order is fixed, so results are
// deterministic.
__device__ __forceinline__ float warp_column_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0];
}

// dgrad: dZ = acc * gelu'(Z) -> bf16 out, 32 columns at a time.  With BGRAD,
// each 32-column chunk's fp32 dZ (zero outside the matrix) is summed over the
// warp's 32 rows and written to the workspace band of this warp.
template <bool BGRAD>
__device__ __forceinline__ void store_dgrad(const GemmParams& p, int r, int cbase, float2 (&acc)[kHalfN / 2],
                                            float* band, int lane) {
    const bool row_ok = r < p.M;
    const int64_t off = static_cast<int64_t>(row_ok ? r : 0) * p.N + cbase;
    uint16_t* out = static_cast<uint16_t*>(p.out) + off;
    const uint16_t* zp = static_cast<const uint16_t*>(p.aux) + off;
    const bool vec = (p.N & 7) == 0 && cbase + kHalfN <= p.N;
#pragma unroll
    for (int c = 0; c < kHalfN / 32; ++c) {
        float v[32];
        if (row_ok && vec) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                const uint4 zv = *reinterpret_cast<const uint4*>(zp + c * 32 + j);
                const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
                uint32_t ow[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 a = acc[(c * 32 + j) / 2 + i];
                    v[j + 2 * i] = a.x * dgelu_tanh(bf16_lo(zw[i]));
                    v[j + 2 * i + 1] = a.y * dgelu_tanh(bf16_hi(zw[i]));
                    ow[i] = pack_bf16x2(v[j + 2 * i], v[j + 2 * i + 1]);
                }
                *reinterpret_cast<uint4*>(out + c * 32 + j) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int col = cbase + c * 32 + j;
                const float a = (j & 1) ? acc[(c * 32 + j) / 2].y : acc[(c * 32 + j) / 2].x;
                v[j] = 0.0f;
                if (row_ok && col < p.N) {
                    const float z = __uint_as_float(static_cast<uint32_t>(zp[c * 32 + j]) << 16);
                    v[j] = a * dgelu_tanh(z);
                    out[c * 32 + j] = static_cast<uint16_t>(pack_bf16x2(v[j], 0.0f) & 0xFFFFu);
                }
            }
        }
        if (BGRAD) {
            const float s = warp_column_sum32(v, lane);
            const int col = cbase + c * 32 + lane;
            if (col < p.N) band[col] = s;
        }
    }
}

// acc[i] += P[i] * (sA * sB[2i, 2i+1]) for 32 columns of this thread, as
// packed fp32x2 multiplies and fmas (two columns per instruction, each rounded
// to nearest as the scalar multiply and fma would be).  acc points into the
// thread's register accumulator at a compile-time offset.
__device__ __forceinline__ void promote32(uint64_t* acc, const uint64_t* p, uint64_t sa2, const float* sbp) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const ulonglong2 sb = *reinterpret_cast<const ulonglong2*>(sbp + 4 * j);
        acc[2 * j] = fma_f32x2(p[2 * j], mul_f32x2(sa2, sb.x), acc[2 * j]);
        acc[2 * j + 1] = fma_f32x2(p[2 * j + 1], mul_f32x2(sa2, sb.y), acc[2 * j + 1]);
    }
}

// -------------------------------------------------------------------- kernel

template <int EPI, bool FAST>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ TensorMaps maps, const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    SmemLayout& sm = *reinterpret_cast<SmemLayout*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                    ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.budget_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        for (int s = 0; s < kSStages; ++s) {
            mbar_init(smem_addr(&sm.sfull[s]), 1);
            mbar_init(smem_addr(&sm.sempty[s]), kEpiWarps);
        }
        for (int b = 0; b < kNumAcc; ++b) {
            mbar_init(smem_addr(&sm.acc_full[b]), 1);
            mbar_init(smem_addr(&sm.acc_empty[b]), kEpiWarps);
        }
        mbar_init(smem_addr(&sm.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;

    if (warp < kFirstEpiWarp) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.a);
            tma_prefetch_desc(&maps.b);
            tma_prefetch_desc(&maps.sa);
            tma_prefetch_desc(&maps.sb);
            int s = 0, ss = 0;
            uint32_t ph = 0, sph = 0;
            int n_issued = 0, ns_issued = 0;
            bool ok = true;
            if (!p.debug_starve) {
                for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                    int g, mt, nt;
                    decode_tile(p, t, g, mt, nt);
                    const GroupEntry ge = p.groups[g];
                    const int m0 = mt * kBM, n0 = nt * kBN;
                    for (int kb = 0; kb < ge.nkb; ++kb) {
                        const int kbg = ge.kb_start + kb;
                        if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_addr(&sm.full[s]);
                        mbar_arrive_expect_tx(fb, kBM * kBK + kBN * kBK);
                        tma_load_2d(smem_addr(sm.a[s]), &maps.a, fb, kbg * kBK, m0);
                        tma_load_2d(smem_addr(sm.b[s]), &maps.b, fb, kbg * kBK, n0);
                        ++n_issued;
                        ring_advance<kStages>(s, ph);
                        if (!mbar_wait(smem_addr(&sm.sempty[ss]), sph ^ 1u, budget)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sfb = smem_addr(&sm.sfull[ss]);
                        mbar_arrive_expect_tx(sfb, (kBM + kBN) * 4);
                        tma_load_2d(smem_addr(sm.sa[ss]), &maps.sa, sfb, m0, kbg);
                        tma_load_2d(smem_addr(sm.sb[ss]), &maps.sb, sfb, n0, kbg);
                        ++ns_issued;
                        ring_advance<kSStages>(ss, sph);
                    }
                }
            }
            if (ok) {
                // every stage must be released by its consumer before exit
                for (int i = 0; i < kStages; ++i) {
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) ok = false;
                    ring_advance<kStages>(s, ph);
                }
                for (int i = 0; i < kSStages; ++i) {
                    if (!mbar_wait(smem_addr(&sm.sempty[ss]), sph ^ 1u, budget)) ok = false;
                    ring_advance<kSStages>(ss, sph);
                }
            }
            if (!ok) {
                record_status(p.status, kStatusTimeout);
                // let the loads still in flight land before shared memory goes away
                for (int i = 1; i <= (n_issued < kStages ? n_issued : kStages); ++i) {
                    int si = s - i;
                    uint32_t pi = ph;
                    if (si < 0) {
                        si += kStages;
                        pi ^= 1u;
                    }
                    mbar_wait(smem_addr(&sm.full[si]), pi, budget);
                }
                for (int i = 1; i <= (ns_issued < kSStages ? ns_issued : kSStages); ++i) {
                    int si = ss - i;
                    uint32_t pi = sph;
                    if (si < 0) {
                        si += kSStages;
                        pi ^= 1u;
                    }
                    mbar_wait(smem_addr(&sm.sfull[si]), pi, budget);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        int s = 0, ab = 0;
        uint32_t ph = 0, aph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            int g, mt, nt;
            decode_tile(p, t, g, mt, nt);
            const int nkb = p.groups[g].nkb;
            for (int kb = 0; kb < nkb; ++kb) {
                ok = warp_all(mbar_wait(smem_addr(&sm.acc_empty[ab]), aph ^ 1u, budget));
                if (ok) ok = warp_all(mbar_wait(smem_addr(&sm.full[s]), ph, budget));
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t d = tmem_base + static_cast<uint32_t>(ab * kBN);
                    const uint64_t adesc = smem_desc_k_sw128(smem_addr(sm.a[s]));
                    const uint64_t bdesc = smem_desc_k_sw128(smem_addr(sm.b[s]));
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        mma_f8f6f4(d, adesc + 2u * k, bdesc + 2u * k, p.idesc, k > 0 ? 1u : 0u);
                    mma_commit(smem_addr(&sm.empty[s]));
                    mma_commit(smem_addr(&sm.acc_full[ab]));
                }
                __syncwarp();
                ring_advance<kStages>(s, ph);
                ring_advance<kNumAcc>(ab, aph);
            }
        }
        if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
        // all MMAs issued by this warp must complete before TMEM is released
        if (lane == 0) mma_commit(smem_addr(&sm.drain));
        __syncwarp();
        mbar_wait(smem_addr(&sm.drain), 0, budget);
        __syncwarp();
    } else if (warp >= kFirstEpiWarp) {
        // ------------------------------------------ promotion and epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
        const int ew = warp - kFirstEpiWarp;
        const int q = warp & 3;        // TMEM lane quadrant of this warp
        const int half = ew >> 2;      // which 64 columns of the tile
        const int row = q * 32 + lane; // row within the tile
        int ab = 0, ss = 0;
        uint32_t aph = 0, sph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            int g, mt, nt;
            decode_tile(p, t, g, mt, nt);
            const GroupEntry ge = p.groups[g];
            const int m0 = mt * kBM, n0 = nt * kBN;
            uint64_t acc[kHalfN / 2];  // packed fp32 pairs: columns 2i, 2i+1
#pragma unroll
            for (int j = 0; j < kHalfN / 2; ++j) acc[j] = 0ull;
            const uint32_t tlane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(half * kHalfN);
            for (int kb = 0; kb < ge.nkb; ++kb) {
                ok = warp_all(mbar_wait2(smem_addr(&sm.acc_full[ab]), aph, smem_addr(&sm.sfull[ss]), sph, budget));
                if (!ok) break;
                tc_fence_after();
                const uint32_t tbuf = tlane + ab * kBN;
                const float sa = sm.sa[ss][row];
                const uint64_t sa2 = pack_f32x2(sa, sa);
                const float* sbp = &sm.sb[ss][half * kHalfN];
                // two 64-column TMEM loads; the buffer goes back to the MMA warp
                // as soon as the second one has landed
                {
                    uint64_t pr[32];
                    tmem_ld_32x32b_x64_pairs(tbuf, pr);
                    promote32(&acc[0], &pr[0], sa2, sbp);
                    promote32(&acc[16], &pr[16], sa2, sbp + 32);
                }
                {
                    uint64_t pr[32];
                    tmem_ld_32x32b_x64_pairs(tbuf + 64, pr);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&sm.acc_empty[ab]));
                    promote32(&acc[32], &pr[0], sa2, sbp + 64);
                    promote32(&acc[48], &pr[16], sa2, sbp + 96);
                }
                // the scale stage was read with ordinary loads and is refilled by
                // TMA: order the reads before the release (cross-proxy hazard)
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&sm.sempty[ss]));
                ring_advance<kNumAcc>(ab, aph);
                ring_advance<kSStages>(ss, sph);
            }
            if (!ok) break;
            float2 accf[kHalfN / 2];
#pragma unroll
            for (int j = 0; j < kHalfN / 2; ++j) accf[j] = unpack_f32x2(acc[j]);
            const int r = m0 + row;
            const int cbase = n0 + half * kHalfN;
            if (EPI == kEpiWgrad) {
                store_wgrad(p, ge.out_index, r, cbase, accf);
            } else if (EPI == kEpiNone || EPI == kEpiBias || EPI == kEpiBiasGelu) {
                store_fprop<EPI>(p, r, cbase, accf);
            } else {
                // bias-gradient partials of this warp's 32 rows -> workspace band (4*mt + q)
                float* band = (EPI == kEpiDgeluBgrad) ? p.workspace + (static_cast<int64_t>(mt) * 4 + q) * p.N
                                                      : nullptr;
                store_dgrad<EPI == kEpiDgeluBgrad>(p, r, cbase, accf, band, lane);
            }
        }
        if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int EPI, bool FAST>
int launch_gemm_impl(const TensorMaps& maps, const GemmParams& p, cudaStream_t stream, int grid) {
    auto kern = gemm_fp8_kernel<EPI, FAST>;
    static unsigned long long configured = 0;  // one bit per device ordinal
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -3;
    if (!(configured & (1ull << dev))) {
        // the register split above assumes exactly kLaunchRegs per thread at launch
        cudaFuncAttributes attr;
        if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess || attr.numRegs != kLaunchRegs) return -3;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes)) != cudaSuccess)
            return -3;
        configured |= 1ull << dev;
    }
    kern<<<grid, kThreads, kSmemBytes, stream>>>(maps, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace fp8ll
