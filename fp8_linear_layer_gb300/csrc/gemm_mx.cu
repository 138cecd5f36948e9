// gemm_mx.cu -- MXFP8 GEMM for sm_103a: the scales are applied by the tensor
// core (tcgen05.mma kind::mxf8f6f4 block_scale, one UE8M0 power-of-two scale
// per 32 K-elements of every row of A and B), so the fp32 accumulator stays in
// tensor memory for the whole K range and no software promotion exists.
//
// Same tiling as the 1x128 kernel (128 x 256 output tiles, 128-deep K blocks,
// persistent CTAs), same epilogues (bias / GELU, GELU derivative with bias
// gradient, fp32 out (+)=).  Per CTA:
//   warp 0      TMA producer: A and B code boxes (128-byte swizzle) plus the
//               block's scale atoms (512 B for A, 1 KB for B, untiled bulk
//               copies) into one 4-stage ring.
//   warp 1      TMEM owner and MMA issuer: per K block, three tcgen05.cp copy
//               the scale atoms into a tensor-memory scale slot (4 slots of
//               16 columns, 12 used: lane l, column c = the four 32-element
//               scales of row l + 32c, B's rows 128..255 four columns
//               further), then
//               four block-scaled MMAs (M=128, N=256, K=32, scale id = the
//               32-element group) accumulate into one 256-column accumulator.
//   warps 4-11  epilogue: once per tile, the accumulator is read (16x256b
//               fragments, as in the 1x128 kernel), handed back to the MMA
//               warp, and stored through the same epilogue functions.
// The scale atoms are the layout the MX cast writes (see quantize.cu).
//
// The per-tensor scaled GEMM (one scale per operand, no scale atoms) runs on
// CTA pairs in gemm_tensor.cu.
#include "gemm_kernel.cuh"

namespace fp8ll {

constexpr int kMxStages = 4;
constexpr int kMxSfSlots = 4;
constexpr uint32_t kMxSfCol0 = 256;   // accumulator in columns 0..255
constexpr uint32_t kMxSfSlotCols = 16;
constexpr uint32_t kMxTmemCols = 512;
static_assert(kMxSfCol0 + kMxSfSlots * kMxSfSlotCols <= kMxTmemCols, "TMEM budget");

struct __align__(1024) MxSmem {
    uint8_t a[kMxStages][kBM * kBK];
    uint8_t b[kMxStages][kBN * kBK];
    uint8_t sfa[kMxStages][512];
    uint8_t sfb[kMxStages][1024];
    uint64_t full[kMxStages];
    uint64_t empty[kMxStages];
    uint64_t acc_full[1];
    uint64_t acc_empty[1];
    uint64_t drain;
    uint32_t tmem_base;
};
constexpr size_t kMxSmemBytes = sizeof(MxSmem) + 1024;
static_assert(kMxSmemBytes <= 232448, "shared memory budget");

// untiled bulk copy global -> shared, completion counted on an mbarrier
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// no-swizzle shared-memory descriptor for a 32-row x 16-byte scale atom
// (8-row x 16-byte core matrices, 128 bytes apart)
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(128 >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ void sf_copy(uint32_t taddr, uint32_t saddr) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sf_desc(saddr)) : "memory");
}

__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ TensorMaps maps, const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    MxSmem& sm = *reinterpret_cast<MxSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.budget_ns;
    const int nkb = p.groups[0].nkb;
    // one 256-column accumulator: columns 256.. hold the scale slots
    constexpr int kAccBufs = 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMxStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        mbar_init(smem_addr(&sm.acc_full[0]), 1);
        mbar_init(smem_addr(&sm.acc_empty[0]), kEpiWarps);
        mbar_init(smem_addr(&sm.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sm.tmem_base), kMxTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;

    if (warp < kFirstEpiWarp) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.a);
            tma_prefetch_desc(&maps.b);
            int s = 0;
            uint32_t ph = 0;
            int n_issued = 0;
            bool ok = true;
            if (!p.debug_starve) {
                for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                    int g, mt, nt;
                    decode_tile(p, t, g, mt, nt);
                    const int m0 = mt * kBM, n0 = nt * kBN;
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_addr(&sm.full[s]);
                        mbar_arrive_expect_tx(fb, kBM * kBK + kBN * kBK + 512 + 1024);
                        tma_load_2d(smem_addr(sm.a[s]), &maps.a, fb, kb * kBK, m0);
                        tma_load_2d(smem_addr(sm.b[s]), &maps.b, fb, kb * kBK, n0);
                        bulk_load(smem_addr(sm.sfa[s]), p.sfa + (static_cast<int64_t>(kb) * p.sfa_groups + mt) * 512,
                                  512, fb);
                        bulk_load(smem_addr(sm.sfb[s]),
                                  p.sfb + (static_cast<int64_t>(kb) * p.sfb_groups + 2 * nt) * 512, 1024, fb);
                        ++n_issued;
                        ring_advance<kMxStages>(s, ph);
                    }
                }
            }
            if (ok) {
                for (int i = 0; i < kMxStages; ++i) {
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) ok = false;
                    ring_advance<kMxStages>(s, ph);
                }
            }
            if (!ok) {
                record_status(p.status, kStatusTimeout);
                for (int i = 1; i <= (n_issued < kMxStages ? n_issued : kMxStages); ++i) {
                    int si = s - i;
                    uint32_t pi = ph;
                    if (si < 0) {
                        si += kMxStages;
                        pi ^= 1u;
                    }
                    mbar_wait(smem_addr(&sm.full[si]), pi, budget);
                }
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        int s = 0, ab = 0;
        uint32_t ph = 0, aph = 0;
        uint32_t slot = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            // the accumulator must have been read by the epilogue of the tile that used it last
            ok = mbar_wait_warp(smem_addr(&sm.acc_empty[ab]), aph ^ 1u, budget);
            if (!ok) break;
            tc_fence_after();
            const uint32_t dacc = tmem_base + static_cast<uint32_t>(ab * kBN);
            for (int kb = 0; kb < nkb; ++kb) {
                ok = mbar_wait_warp(smem_addr(&sm.full[s]), ph, budget);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t adesc = smem_desc_k_sw128(smem_addr(sm.a[s]));
                    const uint64_t bdesc = smem_desc_k_sw128(smem_addr(sm.b[s]));
                    const uint32_t tsf = tmem_base + kMxSfCol0 + slot * kMxSfSlotCols;
                    sf_copy(tsf, smem_addr(sm.sfa[s]));
                    sf_copy(tsf + 4, smem_addr(sm.sfb[s]));
                    sf_copy(tsf + 8, smem_addr(sm.sfb[s] + 512));
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k) {
                        const uint32_t idesc =
                            p.idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
                        mma_mx(dacc, adesc + 2u * k, bdesc + 2u * k, idesc, tsf, tsf + 4,
                               (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_addr(&sm.empty[s]));
                    if (kb == nkb - 1) mma_commit(smem_addr(&sm.acc_full[ab]));
                }
                __syncwarp();
                ring_advance<kMxStages>(s, ph);
                slot = (slot + 1) % kMxSfSlots;
            }
            ring_advance<kAccBufs>(ab, aph);
        }
        if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
        if (lane == 0) mma_commit(smem_addr(&sm.drain));
        __syncwarp();
        mbar_wait(smem_addr(&sm.drain), 0, budget);
        __syncwarp();
    } else if (warp >= kFirstEpiWarp) {
        // ---------------------------------------------------------- epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
        const int ew = warp - kFirstEpiWarp;
        const int q = warp & 3;
        const int half = ew >> 2;
        const int g8 = lane >> 2;
        const int cq = lane & 3;
        int ab = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            int g, mt, nt;
            decode_tile(p, t, g, mt, nt);
            const int m0 = mt * kBM, n0 = nt * kBN;
            if (EPI == kEpiDgelu || EPI == kEpiDgeluBgrad) {
                const int prow = m0 + q * 32 + g8 + 8 * cq;
                const int pc0 = n0 + half * kHalfN;
                if (prow < p.M && pc0 < p.N) {
                    const uint16_t* zrow = static_cast<const uint16_t*>(p.aux) + static_cast<int64_t>(prow) * p.N;
                    const int pc1 = min(pc0 + kHalfN - 1, p.N - 1);
                    prefetch_l2(zrow + pc0);
                    prefetch_l2(zrow + min(pc0 + 64, pc1));
                    prefetch_l2(zrow + pc1);
                }
            }
            ok = mbar_wait_warp(smem_addr(&sm.acc_full[ab]), aph, budget);
            if (!ok) break;
            tc_fence_after();
            uint64_t acc[4 * kChunks];
            const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                static_cast<uint32_t>(ab * kBN + half * kHalfN);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint64_t plo[8], phi[8];
                tmem_ld_16x256b_x4_pairs2(tq + 32u * h, tq + (16u << 16) + 32u * h, plo, phi);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = 4 * h + i;
                    acc[4 * c + 0] = plo[2 * i];
                    acc[4 * c + 1] = plo[2 * i + 1];
                    acc[4 * c + 2] = phi[2 * i];
                    acc[4 * c + 3] = phi[2 * i + 1];
                }
            }
            // the tile's sums are in registers: the accumulator goes back to the MMA warp
            tc_fence_before();
            __syncwarp();
            mbar_arrive_lane0(smem_addr(&sm.acc_empty[ab]), lane);
            ring_advance<kAccBufs>(ab, aph);
            const int row0 = m0 + q * 32 + g8;
            const int col0 = n0 + half * kHalfN + 2 * cq;
            if (EPI == kEpiWgrad) {
                store_wgrad(p, 0, row0, col0, acc);
            } else if (EPI == kEpiNone || EPI == kEpiBias || EPI == kEpiBiasGelu) {
                store_fprop<EPI>(p, row0, col0, acc);
            } else {
                float* band = (EPI == kEpiDgeluBgrad) ? p.workspace + (static_cast<int64_t>(mt) * 4 + q) * p.N
                                                      : nullptr;
                store_dgrad<EPI == kEpiDgeluBgrad, false>(p, row0, col0, acc, band, lane, nullptr);
            }
        }
        if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kMxTmemCols);
}

template <int EPI>
int launch_mx_impl(const TensorMaps& maps, const GemmParams& p, cudaStream_t stream, int grid) {
    auto kern = gemm_mx_kernel<EPI>;
    static unsigned long long configured = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -3;
    if (!(configured & (1ull << dev))) {
        cudaFuncAttributes attr;
        if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess || attr.numRegs != kLaunchRegs) return -3;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kMxSmemBytes)) != cudaSuccess)
            return -3;
        configured |= 1ull << dev;
    }
    kern<<<grid, kThreads, kMxSmemBytes, stream>>>(maps, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_gemm_mx(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream, int grid) {
    switch (epi) {
        case kEpiNone: return launch_mx_impl<kEpiNone>(maps, p, stream, grid);
        case kEpiBias: return launch_mx_impl<kEpiBias>(maps, p, stream, grid);
        case kEpiBiasGelu: return launch_mx_impl<kEpiBiasGelu>(maps, p, stream, grid);
        case kEpiDgelu: return launch_mx_impl<kEpiDgelu>(maps, p, stream, grid);
        case kEpiDgeluBgrad: return launch_mx_impl<kEpiDgeluBgrad>(maps, p, stream, grid);
        case kEpiWgrad: return launch_mx_impl<kEpiWgrad>(maps, p, stream, grid);
        default: return -3;
    }
}

}  // namespace fp8ll
