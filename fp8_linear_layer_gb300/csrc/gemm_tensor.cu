// gemm_tensor.cu -- per-tensor scaled FP8 GEMM for sm_103a on CTA pairs.
//
// "FP8 GEMM for the fprop should use fast accumulation": with one fp32 scale
// per operand tensor, plain kind::f8f6f4 MMAs accumulate the raw fp8 products
// over the whole K range in tensor memory and the epilogue multiplies the
// fp32 sums by fl32(sA * sB) once per tile -- no promotion inside the K loop,
// so this kernel is bound by how fast operands reach the tensor core.
//
// Clusters of two CTAs on two SMs share each MMA (cta_group::2, M = 256,
// N = 256): each CTA loads its 128 rows of A and half of B's 256 rows, 32 KB
// per 128-deep K block where a lone CTA computing a 128 x 256 tile loads
// 48 KB, and the same shared-memory budget holds six stages instead of four.
// Per CTA, 3 warpgroups (12 warps):
//   warp 0      TMA producer: its A and B boxes (128-byte swizzle) into a
//               6-stage ring; both CTAs' bytes are counted on the leader's
//               (rank 0's) stage barrier.
//   warp 1      TMEM owner (the pair allocates together) and, in the leader,
//               MMA issuer: per K block four M256 x N256 x K32 MMAs into one
//               of two 256-column accumulators (alternating per tile, so a
//               tile's MMAs need not wait for the previous tile's epilogue);
//               its commits arrive on the barriers of both CTAs.
//   warps 4-11  epilogue: once per tile each CTA reads its 128 rows of the
//               accumulator (16x256b fragments), hands the buffer back to the
//               leader and stores through the epilogues of the 1x128 kernel.
#include "gemm_kernel.cuh"

namespace fp8ll {

constexpr int kTpStages = 6;
constexpr int kTpRows = 2 * kBM;     // output rows of a pair's tile
constexpr int kTpBRows = kBN / 2;    // rows of B each CTA loads
constexpr int kTpRaster = kRasterM / 2;
constexpr uint32_t kTpStageBytes = (kBM + kTpBRows) * kBK;

struct __align__(1024) TpSmem {
    uint8_t b[kTpStages][kTpBRows * kBK];
    uint8_t a[kTpStages][kBM * kBK];
    uint64_t full[kTpStages];   // leader: both CTAs' bytes of stage s have landed
    uint64_t empty[kTpStages];  // stage s read by the pair's MMAs (commit to both CTAs)
    uint64_t acc_full[2];       // accumulator b holds a finished tile (commit to both CTAs)
    uint64_t acc_empty[2];      // leader: both CTAs' epilogue warps have read it
    uint64_t drain;
    uint32_t tmem_base;
};
constexpr size_t kTpSmemBytes = sizeof(TpSmem) + 1024;
static_assert(kTpSmemBytes <= 232448, "shared memory budget");

// pair-tile index -> (pair-row tile, n tile): bands of kTpRaster pair rows
// walked column by column, as decode_tile does for 128-row tiles
__device__ __forceinline__ void decode_pair_tile(const GemmParams& p, int t, int& mt, int& nt) {
    const int band_tiles = kTpRaster * p.num_n_tiles;
    const int band = t / band_tiles;
    const int first_m = band * kTpRaster;
    const int rem_m = p.num_m_pairs - first_m;
    const int bm = rem_m < kTpRaster ? rem_m : kTpRaster;
    const int r = t - band * band_tiles;
    mt = first_m + r % bm;
    nt = r / bm;
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tensor_kernel(const __grid_constant__ TensorMaps maps, const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    TpSmem& sm = *reinterpret_cast<TpSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
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
        for (int s = 0; s < kTpStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&sm.acc_full[b]), 1);
            mbar_init(smem_addr(&sm.acc_empty[b]), 2 * kEpiWarps);
        }
        mbar_init(smem_addr(&sm.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&sm.tmem_base), 512);
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
            int s = 0;
            uint32_t ph = 0;
            int n_issued = 0;
            bool ok = true;
            if (!p.debug_starve) {
                for (int t = pair; t < p.total_tiles && ok; t += num_pairs) {
                    int mt, nt;
                    decode_pair_tile(p, t, mt, nt);
                    const int m0 = mt * kTpRows + static_cast<int>(rank) * kBM;
                    const int nb0 = nt * kBN + static_cast<int>(rank) * kTpBRows;
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_addr(&sm.full[s]);
                        if (leader) mbar_arrive_expect_tx(fb, 2 * kTpStageBytes);
                        const uint32_t fbl = mapa_shared(fb, 0);
                        tma_load_2d_pair(smem_addr(sm.a[s]), &maps.a, fbl, kb * kBK, m0);
                        tma_load_2d_pair(smem_addr(sm.b[s]), &maps.b, fbl, kb * kBK, nb0);
                        ++n_issued;
                        ring_advance<kTpStages>(s, ph);
                    }
                }
            }
            if (ok) {
                // every stage must be released by the pair's MMAs before exit
                for (int i = 0; i < kTpStages; ++i) {
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) ok = false;
                    ring_advance<kTpStages>(s, ph);
                }
            }
            if (!ok) {
                record_status(p.status, kStatusTimeout);
                // the leader's stage barriers count both CTAs' bytes: the loads
                // still in flight land before the leader (and, at the final
                // cluster barrier, the peer) leaves
                if (leader) {
                    for (int i = 1; i <= (n_issued < kTpStages ? n_issued : kTpStages); ++i) {
                        int si = s - i;
                        uint32_t pi = ph;
                        if (si < 0) {
                            si += kTpStages;
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
            int s = 0, ab = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int t = pair; t < p.total_tiles && ok; t += num_pairs) {
                // both CTAs' epilogues must have read this accumulator's last tile
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
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            mma_f8f6f4_pair(dacc, adesc + 2u * k, bdesc + 2u * k, p.idesc,
                                            (kb > 0 || k > 0) ? 1u : 0u);
                        mma_commit_pair(smem_addr(&sm.empty[s]), 0x3);
                        if (kb == nkb - 1) mma_commit_pair(smem_addr(&sm.acc_full[ab]), 0x3);
                    }
                    __syncwarp();
                    ring_advance<kTpStages>(s, ph);
                }
                ring_advance<2>(ab, aph);
            }
            if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
            // every MMA of the pair completes before either CTA frees its memory
            if (lane == 0) mma_commit_pair(smem_addr(&sm.drain), 0x3);
            __syncwarp();
            mbar_wait(smem_addr(&sm.drain), 0, budget);
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
        const uint32_t acc_empty0 = mapa_shared(smem_addr(&sm.acc_empty[0]), 0);
        const uint32_t acc_empty_step = smem_addr(&sm.acc_empty[1]) - smem_addr(&sm.acc_empty[0]);
        int ab = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int t = pair; t < p.total_tiles && ok; t += num_pairs) {
            int mt, nt;
            decode_pair_tile(p, t, mt, nt);
            const int m0 = mt * kTpRows + static_cast<int>(rank) * kBM, n0 = nt * kBN;
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
            // the tile's sums are in registers: the accumulator goes back to the leader
            tc_fence_before();
            __syncwarp();
            mbar_arrive_remote_lane0(acc_empty0 + static_cast<uint32_t>(ab) * acc_empty_step, lane);
            ring_advance<2>(ab, aph);
            const float st = __fmul_rn(*p.tsa, *p.tsb);
            const uint64_t st2 = pack_f32x2(st, st);
#pragma unroll
            for (int j = 0; j < 4 * kChunks; ++j) acc[j] = mul_f32x2(acc[j], st2);
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
        tmem_dealloc_pair(tmem_base, 512);
    }
}

template <int EPI>
int launch_tensor_impl(const TensorMaps& maps, const GemmParams& p, cudaStream_t stream) {
    auto kern = gemm_tensor_kernel<EPI>;
    static unsigned long long configured = 0;
    static int pairs_on[64] = {0};  // resident CTA pairs per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -3;
    if (!(configured & (1ull << dev))) {
        cudaFuncAttributes attr;
        if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess || attr.numRegs != kLaunchRegs) return -3;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kTpSmemBytes)) != cudaSuccess)
            return -3;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kTpSmemBytes;
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
    kern<<<grid, kThreads, kTpSmemBytes, stream>>>(maps, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_gemm_tensor(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream) {
    switch (epi) {
        case kEpiNone: return launch_tensor_impl<kEpiNone>(maps, p, stream);
        case kEpiBias: return launch_tensor_impl<kEpiBias>(maps, p, stream);
        case kEpiBiasGelu: return launch_tensor_impl<kEpiBiasGelu>(maps, p, stream);
        case kEpiDgelu: return launch_tensor_impl<kEpiDgelu>(maps, p, stream);
        case kEpiDgeluBgrad: return launch_tensor_impl<kEpiDgeluBgrad>(maps, p, stream);
        case kEpiWgrad: return launch_tensor_impl<kEpiWgrad>(maps, p, stream);
        default: return -3;
    }
}

}  // namespace fp8ll
