// gemm_mx.cu -- MXFP8 GEMM for sm_103a on CTA pairs: the scales are applied
// by the tensor core (tcgen05.mma kind::mxf8f6f4 block_scale, one UE8M0
// power-of-two scale per 32 K-elements of every row of A and B), so the fp32
// accumulator stays in tensor memory for the whole K range and no software
// promotion exists.
//
// Clusters of two CTAs on two SMs share each MMA (cta_group::2, M = 256,
// N = 256), as the per-tensor kernel does: each CTA loads its 128 rows of A,
// half of B's 256 rows and, per 128-deep K block, the scale atoms its half of
// the MMA reads from its own tensor memory -- the 512-byte atom of its A rows
// and both atoms of B's 256 rows (a probe on the GPU showed each CTA's half of
// a pair's block-scaled MMA takes A's scales for its rows and all of B's from
// its own tensor memory, and tcgen05.cp.cta_group::2 fills each CTA's tensor
// memory from that CTA's shared memory).  Per CTA, 3 warpgroups:
//   warp 0      TMA producer: A and B code boxes (128-byte swizzle) and the
//               scale atoms (as 128-word rows of a 2-D map over the atom
//               array) into a 6-stage ring; both CTAs' bytes are counted on
//               the leader's (rank 0's) stage barrier.
//   warp 1      TMEM owner (the pair allocates together) and, in the leader,
//               MMA issuer: per K block, once the stage and its scales are
//               in place, four block-scaled MMAs (M=256, N=256, K=32, scale
//               id = the 32-element group) accumulate into one 256-column
//               accumulator per CTA.
//   warp 3      in the leader, scale copier: as each stage lands, three
//               tcgen05.cp copy its scale atoms into that stage's 16-column
//               tensor-memory slot of both CTAs (lane l, column c = the four
//               32-element scales of row l + 32c; B's rows 128..255 four
//               columns further) and a commit tells the MMA issuer.  Copies
//               issued by the MMA thread itself, ahead of each block's MMAs,
//               cost the GEMMs 14-17% (they hold up the MMA issue); from this
//               warp the results are bit-identical.  One slot per stage: a
//               slot is refilled only after its stage was, i.e. after the
//               MMAs that read it completed.
//   warps 4-11  epilogue: once per tile each CTA reads its 128 rows of the
//               accumulator (16x256b fragments), hands it back to the leader
//               and stores through the epilogues of the 1x128 kernel.
// The scale atoms are the layout the MX cast writes (see quantize.cu).
//
// The per-tensor scaled GEMM (one scale per operand, no scale atoms) runs on
// CTA pairs in gemm_tensor.cu.
#include "gemm_kernel.cuh"

namespace fp8ll {

constexpr int kMxStages = 6;
constexpr int kMxSfSlots = kMxStages;  // scale slot s belongs to stage s
constexpr uint32_t kMxSfCol0 = 256;   // accumulator in columns 0..255
constexpr uint32_t kMxSfSlotCols = 16;
constexpr uint32_t kMxTmemCols = 512;
static_assert(kMxSfCol0 + kMxSfSlots * kMxSfSlotCols <= kMxTmemCols, "TMEM budget");
constexpr int kMxRows = 2 * kBM;     // output rows of a pair's tile
constexpr int kMxBRows = kBN / 2;    // rows of B each CTA loads
constexpr int kMxRaster = kRasterM / 2;
constexpr uint32_t kMxStageBytes = (kBM + kMxBRows) * kBK + 512 + 1024;  // one CTA's bytes per K block

struct __align__(1024) MxSmem {
    uint8_t b[kMxStages][kMxBRows * kBK];
    uint8_t a[kMxStages][kBM * kBK];
    uint8_t sfa[kMxStages][512];   // the atom of this CTA's 128 rows of A
    uint8_t sfb[kMxStages][1024];  // both atoms of the pair's 256 rows of B
    uint64_t full[kMxStages];      // leader: both CTAs' bytes of stage s have landed
    uint64_t empty[kMxStages];     // stage s read by the pair's copies and MMAs
    uint64_t acc_full[1];
    uint64_t acc_empty[1];         // leader: both CTAs' epilogue warps have read the accumulator
    uint64_t drain;
    uint64_t sf_full[kMxStages];   // leader: stage s's scales are in both CTAs' tensor memory
    uint64_t sf_drain;             // leader: the copier's last copies completed
    uint32_t tmem_base;
};
constexpr size_t kMxSmemBytes = sizeof(MxSmem) + 1024;
static_assert(kMxSmemBytes <= 232448, "shared memory budget");

// no-swizzle shared-memory descriptor for a 32-row x 16-byte scale atom
// (8-row x 16-byte core matrices, 128 bytes apart)
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(128 >> 4) << 32) | (1ull << 46);
}

// each CTA's atom at this shared-memory offset -> the same columns of its own tensor memory
__device__ __forceinline__ void sf_copy_pair(uint32_t taddr, uint32_t saddr) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sf_desc(saddr)) : "memory");
}

__device__ __forceinline__ void mma_mx_pair(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// pair-tile index -> (pair-row tile, n tile), as decode_tile over 256-row tiles
__device__ __forceinline__ void decode_mx_tile(const GemmParams& p, int t, int& mt, int& nt) {
    const int band_tiles = kMxRaster * p.num_n_tiles;
    const int band = t / band_tiles;
    const int first_m = band * kMxRaster;
    const int rem_m = p.num_m_pairs - first_m;
    const int bm = rem_m < kMxRaster ? rem_m : kMxRaster;
    const int r = t - band * band_tiles;
    mt = first_m + r % bm;
    nt = r / bm;
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ TensorMaps maps, const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    MxSmem& sm = *reinterpret_cast<MxSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.budget_ns;
    const int nkb = p.groups[0].nkb;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMxStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        mbar_init(smem_addr(&sm.acc_full[0]), 1);
        mbar_init(smem_addr(&sm.acc_empty[0]), 2 * kEpiWarps);
        mbar_init(smem_addr(&sm.drain), 1);
        for (int s = 0; s < kMxStages; ++s) mbar_init(smem_addr(&sm.sf_full[s]), 1);
        mbar_init(smem_addr(&sm.sf_drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&sm.tmem_base), kMxTmemCols);
        tmem_relinquish_pair();
    }
    // both CTAs' barriers initialised and tensor memory allocated before either signals the other
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;

    if (warp < kFirstEpiWarp) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.a);
            tma_prefetch_desc(&maps.b);
            tma_prefetch_desc(&maps.sa);
            tma_prefetch_desc(&maps.sb);
            int s = 0;
            uint32_t ph = 0;
            int n_issued = 0;
            bool ok = true;
            if (!p.debug_starve) {
                for (int t = pair; t < p.total_tiles && ok; t += num_pairs) {
                    int mt, nt;
                    decode_mx_tile(p, t, mt, nt);
                    const int m0 = mt * kMxRows + static_cast<int>(rank) * kBM;
                    const int nb0 = nt * kBN + static_cast<int>(rank) * kMxBRows;
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_addr(&sm.full[s]);
                        if (leader) mbar_arrive_expect_tx(fb, 2 * kMxStageBytes);
                        const uint32_t fbl = mapa_shared(fb, 0);
                        tma_load_2d_pair(smem_addr(sm.a[s]), &maps.a, fbl, kb * kBK, m0);
                        tma_load_2d_pair(smem_addr(sm.b[s]), &maps.b, fbl, kb * kBK, nb0);
                        // scale atoms: rows of 128 words; A's atom of this CTA's 128-row group,
                        // both atoms of the tile's 256 rows of B
                        tma_load_2d_pair(smem_addr(sm.sfa[s]), &maps.sa, fbl, 0,
                                         static_cast<int32_t>(kb * p.sfa_groups + 2 * mt + static_cast<int>(rank)));
                        tma_load_2d_pair(smem_addr(sm.sfb[s]), &maps.sb, fbl, 0,
                                         static_cast<int32_t>(kb * p.sfb_groups + 2 * nt));
                        ++n_issued;
                        ring_advance<kMxStages>(s, ph);
                    }
                }
            }
            if (ok) {
                // every stage must be released by the pair's MMAs before exit
                for (int i = 0; i < kMxStages; ++i) {
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) ok = false;
                    ring_advance<kMxStages>(s, ph);
                }
            }
            if (!ok) {
                record_status(p.status, kStatusTimeout);
                // the leader's stage barriers count both CTAs' bytes: the loads
                // still in flight land before the leader (and, at the final
                // cluster barrier, the peer) leaves
                if (leader) {
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
        }
    } else if (warp == 1) {
        // -------------------------------------------- MMA issuer (leader only)
        if (leader) {
            int s = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int t = pair; t < p.total_tiles && ok; t += num_pairs) {
                // both CTAs' epilogues must have read the accumulator's last tile
                ok = mbar_wait_warp(smem_addr(&sm.acc_empty[0]), aph ^ 1u, budget);
                if (!ok) break;
                tc_fence_after();
                for (int kb = 0; kb < nkb; ++kb) {
                    ok = mbar_wait2_warp(smem_addr(&sm.full[s]), ph, smem_addr(&sm.sf_full[s]), ph, budget);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t adesc = smem_desc_k_sw128(smem_addr(sm.a[s]));
                        const uint64_t bdesc = smem_desc_k_sw128(smem_addr(sm.b[s]));
                        const uint32_t tsf = tmem_base + kMxSfCol0 + static_cast<uint32_t>(s) * kMxSfSlotCols;
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k) {
                            const uint32_t idesc =
                                p.idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
                            mma_mx_pair(tmem_base, adesc + 2u * k, bdesc + 2u * k, idesc, tsf, tsf + 4,
                                        (kb > 0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit_pair(smem_addr(&sm.empty[s]), 0x3);
                        if (kb == nkb - 1) mma_commit_pair(smem_addr(&sm.acc_full[0]), 0x3);
                    }
                    __syncwarp();
                    ring_advance<kMxStages>(s, ph);
                }
                aph ^= 1u;
            }
            if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
            // every MMA of the pair completes before either CTA frees its memory
            if (lane == 0) mma_commit_pair(smem_addr(&sm.drain), 0x3);
            __syncwarp();
            mbar_wait(smem_addr(&sm.drain), 0, budget);
            __syncwarp();
        }
    } else if (warp == 3) {
        // ------------------------------------------- scale copier (leader only)
        if (leader) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = pair; t < p.total_tiles && ok; t += num_pairs) {
                for (int kb = 0; kb < nkb; ++kb) {
                    // stage s of this block landed in both CTAs; its slot's last
                    // readers (the MMAs of the stage's previous use) completed
                    // before the producer refilled it
                    ok = mbar_wait_warp(smem_addr(&sm.full[s]), ph, budget);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t tsf = tmem_base + kMxSfCol0 + static_cast<uint32_t>(s) * kMxSfSlotCols;
                        sf_copy_pair(tsf, smem_addr(sm.sfa[s]));
                        sf_copy_pair(tsf + 4, smem_addr(sm.sfb[s]));
                        sf_copy_pair(tsf + 8, smem_addr(sm.sfb[s] + 512));
                        mma_commit_pair(smem_addr(&sm.sf_full[s]), 0x1);
                    }
                    __syncwarp();
                    ring_advance<kMxStages>(s, ph);
                }
            }
            if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
            // the copies complete before either CTA frees its tensor memory
            if (lane == 0) mma_commit_pair(smem_addr(&sm.sf_drain), 0x1);
            __syncwarp();
            mbar_wait(smem_addr(&sm.sf_drain), 0, budget);
            __syncwarp();
        }
    } else if (warp >= kFirstEpiWarp) {
        // ---------------------------------------------------------- epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
        const int ew = warp - kFirstEpiWarp;
        const int q = warp & 3;
        const int half = ew >> 2;
        const int g8 = lane >> 2;
        const int cq = lane & 3;
        const uint32_t acc_empty_leader = mapa_shared(smem_addr(&sm.acc_empty[0]), 0);
        uint32_t aph = 0;
        bool ok = true;
        for (int t = pair; t < p.total_tiles && ok; t += num_pairs) {
            int mt, nt;
            decode_mx_tile(p, t, mt, nt);
            const int m0 = mt * kMxRows + static_cast<int>(rank) * kBM, n0 = nt * kBN;
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
            ok = mbar_wait_warp(smem_addr(&sm.acc_full[0]), aph, budget);
            if (!ok) break;
            tc_fence_after();
            uint64_t acc[4 * kChunks];
            const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(half * kHalfN);
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
            // the tile's sums are in registers: the accumulator goes back to the leader
            tc_fence_before();
            __syncwarp();
            mbar_arrive_remote_lane0(acc_empty_leader, lane);
            aph ^= 1u;
            // the peer of a pair whose tile ends inside the leader's rows holds
            // only rows outside the matrix and stores nothing
            if (m0 >= p.M) continue;
            const int row0 = m0 + q * 32 + g8;
            const int col0 = n0 + half * kHalfN + 2 * cq;
            if (EPI == kEpiWgrad) {
                store_wgrad(p, 0, row0, col0, acc);
            } else if (EPI == kEpiNone || EPI == kEpiBias || EPI == kEpiBiasGelu) {
                store_fprop<EPI>(p, row0, col0, acc);
            } else {
                float* band = (EPI == kEpiDgeluBgrad) ? p.workspace + (static_cast<int64_t>(m0 / kBM) * 4 + q) * p.N
                                                      : nullptr;
                store_dgrad<EPI == kEpiDgeluBgrad, false>(p, row0, col0, acc, band, lane, nullptr);
            }
        }
        if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
    }

    // neither CTA leaves (or frees its tensor memory) while the other may still
    // use its shared memory, tensor memory or barriers
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        // the leader waited for the pair's MMAs above; the peer's drain barrier
        // received the same commit
        if (!leader) mbar_wait_warp(smem_addr(&sm.drain), 0, budget);
        tmem_dealloc_pair(tmem_base, kMxTmemCols);
    }
}

template <int EPI>
int launch_mx_impl(const TensorMaps& maps, const GemmParams& p, cudaStream_t stream) {
    auto kern = gemm_mx_kernel<EPI>;
    static unsigned long long configured = 0;
    static int pairs_on[64] = {0};  // resident CTA pairs per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -3;
    if (!(configured & (1ull << dev))) {
        cudaFuncAttributes attr;
        if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess || attr.numRegs != kLaunchRegs) return -3;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kMxSmemBytes)) != cudaSuccess)
            return -3;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kMxSmemBytes;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -3;
            n = sms / 2;
        }
        pairs_on[dev] = n;
        configured |= 1ull << dev;
    }
    const int pairs = pairs_on[dev];
    const int grid = 2 * (p.total_tiles < pairs ? p.total_tiles : pairs);
    kern<<<grid, kThreads, kMxSmemBytes, stream>>>(maps, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_gemm_mx(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream) {
    switch (epi) {
        case kEpiNone: return launch_mx_impl<kEpiNone>(maps, p, stream);
        case kEpiBias: return launch_mx_impl<kEpiBias>(maps, p, stream);
        case kEpiBiasGelu: return launch_mx_impl<kEpiBiasGelu>(maps, p, stream);
        case kEpiDgelu: return launch_mx_impl<kEpiDgelu>(maps, p, stream);
        case kEpiDgeluBgrad: return launch_mx_impl<kEpiDgeluBgrad>(maps, p, stream);
        case kEpiWgrad: return launch_mx_impl<kEpiWgrad>(maps, p, stream);
        default: return -3;
    }
}

}  // namespace fp8ll
