// CTA-pair tcgen05 GEMM: one 256 x BN output tile per cluster of two CTAs
// (tcgen05.mma.cta_group::2, M = 256).
//
// Each CTA of the pair TMA-loads its own 128 rows of the X tile and its half
// (BN/2 rows) of the Y tile, so an SM receives 16 KB + BN*64 bytes per 64-wide
// K-step instead of 16 KB + BN*128: the bytes each SM must stream per flop
// drop by a third (BN = 256), which is what keeps the tensor core fed from L2
// with the ring depth shared memory allows.  The accumulator of each CTA's 128
// rows x BN columns lives in its own TMEM; its four epilogue warps store them.
//
//   even CTA (leader)   warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 epilogue
//   odd CTA             warp 0 TMA producer, warp 1 forwarder,  warps 2-5 epilogue
//
// Synchronisation across the pair uses only mbarriers:
//   full[s]     leader: armed with both CTAs' bytes; the odd CTA's TMA loads
//               complete their transactions on it directly (cta_group::2);
//   empty[s]    in both CTAs, arrived by the leader's multicast commit;
//   tfull[b]    in both CTAs, arrived by the leader's multicast commit when
//               accumulator b is final;
//   tempty[b]   each CTA's epilogue threads (local, 128 arrivals);
//   ptempty[b]  leader only: the forwarder arrives (remote) once the odd
//               CTA's epilogue has released accumulator b.
// Every wait is bounded; a cluster barrier after set-up (barriers initialised,
// TMEM allocated) and another before TMEM is freed keep the pair in step.
#pragma once
#include <atomic>

#include "common.cuh"

namespace qg {

template <int BN>
struct PairCfg {
    static constexpr int BH = BN / 2;  // Y rows per CTA
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BYTES = BH * BK * 2;
    static constexpr uint32_t STAGE_BYTES = (A_BYTES + B_BYTES + 1023) / 1024 * 1024;
    static constexpr uint32_t TMEM_COLS = tmem_cols_for(2 * BN);
    static constexpr int MAX_STAGES = 12;
    // the epilogue keeps four C/D buffers per warp (16-bit D; fp32 D uses the
    // register path).  With stages of two K-steps the ring depth is the same
    // as with two buffers at every tile width (3 stages at 224 and 256, 4 at
    // 128), and the deeper C prefetch shortens the exposed epilogue of a
    // program's last tile
    static constexpr uint32_t EPI_BYTES = EPI_SMEM_BYTES;
    static constexpr uint32_t AUX_BYTES = (2 * MAX_STAGES + 7 + FIX_BARS + EPI_CBARS) * 8 + 16;
    static constexpr uint32_t FIXED_BYTES = 1024 + EPI_BYTES + AUX_BYTES;
    // a stage holds ks 64-wide K-steps of both operands
    static size_t smem_bytes(int stages, int ks) { return FIXED_BYTES + (size_t)stages * ks * STAGE_BYTES; }
    static int max_stages(int ks) {
        int s = (int)((232448 - FIXED_BYTES) / (ks * STAGE_BYTES));
        return s > MAX_STAGES ? MAX_STAGES : s;
    }
};

__device__ __forceinline__ bool wait_bar_cluster(uint64_t* bar, uint32_t parity, const Guard& g, uint32_t site) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*g.abort) return false;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((n & 31u) == 0) {
            if (*g.abort) return false;
            if (globaltimer_ns() - t0 > g.limit_ns) {
                record_timeout(g, site);
                return false;
            }
        }
    }
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    umma_pair_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                          const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                          const __grid_constant__ GemmKernelParams P) {
    using Cfg = PairCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = P.stages;
    const int KS = P.ks;  // K-steps per stage: 1, or 2-3 with K-chunk tensor maps (one box per operand per stage)
    const uint32_t stage_bytes = (uint32_t)KS * Cfg::STAGE_BYTES;
    const uint32_t a_region = (uint32_t)KS * Cfg::A_BYTES;
    uint8_t* ring = smem;
    uint8_t* esmem = smem + (size_t)S * stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(esmem + Cfg::EPI_BYTES);
    uint64_t* empty = full + Cfg::MAX_STAGES;
    uint64_t* tfull = empty + Cfg::MAX_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* ptempty = tempty + 2;
    uint64_t* done = ptempty + 2;
    uint64_t* cbar = done + 1;
    uint64_t* fixbar = cbar + EPI_CBARS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fixbar + FIX_BARS);
    volatile uint32_t* bcast = tmem_slot + 1;
    volatile uint32_t* abort_flag = tmem_slot + 2;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 128);
            mbar_init(&ptempty[b], 1);
        }
        mbar_init(done, 1);
        for (int i = 0; i < EPI_CBARS; ++i) mbar_init(&cbar[i], 1);
        for (int i = 0; i < FIX_BARS; ++i) mbar_init(&fixbar[i], 1);
        *bcast = 0;
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmY);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // set-up overlaps the previous kernel's tail; no global memory is
    // touched before the previous grid is done
    griddep_launch_dependents();
    griddep_wait();
    const Guard g{P.status, P.timeout_ns, abort_flag};

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            WorkIter w;
            w.init(P.sched, unit_pid(P));
            Unit u;
            int s = 0;
            uint32_t ph = 0, armed = 0, armed_par = 0;
            bool ok = true;
            while (ok && next_unit(P, w, u, BN)) {
                // this CTA's half of the Y tile
                const int32_t y0 = (int32_t)(u.y_row0 + (int64_t)rank * Cfg::BH);
                for (int k = u.k_begin; k < u.k_end; k += KS) {
                    if (!wait_bar(&empty[s], ph ^ 1, g, SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    uint8_t* a = ring + (size_t)s * stage_bytes;
                    uint8_t* b = a + a_region;
                    if (KS > 1) {
                        // K-chunk maps: coordinates (0, row, chunk), boxes of KS 64-wide chunks
                        // (past the last chunk TMA fills zeros and still counts the bytes)
                        // (a batched / grouped Y operand adds the batch or expert coordinate)
                        if (leader) {
                            mbar_arrive_expect_tx(&full[s], 2 * KS * (Cfg::A_BYTES + Cfg::B_BYTES));
                            tma_load_3d(a, &tmX, &full[s], 0, (int32_t)u.x_row0, k);
                            if (P.y3d)
                                tma_load_4d(b, &tmY, &full[s], 0, y0, k, u.batch);
                            else
                                tma_load_3d(b, &tmY, &full[s], 0, y0, k);
                        } else {
                            const uint32_t lf = mapa_shared(smem_u32(&full[s]), 0);
                            tma_load_3d_pair(a, &tmX, lf, 0, (int32_t)u.x_row0, k);
                            if (P.y3d)
                                tma_load_4d_pair(b, &tmY, lf, 0, y0, k, u.batch);
                            else
                                tma_load_3d_pair(b, &tmY, lf, 0, y0, k);
                        }
                    } else if (leader) {
                        mbar_arrive_expect_tx(&full[s], 2 * (Cfg::A_BYTES + Cfg::B_BYTES));
                        if (P.x3d)
                            tma_load_3d(a, &tmX, &full[s], k * P.kstep, (int32_t)u.x_row0, u.batch);
                        else
                            tma_load_2d(a, &tmX, &full[s], k * P.kstep, (int32_t)u.x_row0);
                        if (P.y3d)
                            tma_load_3d(b, &tmY, &full[s], k * P.kstep, y0, u.batch);
                        else
                            tma_load_2d(b, &tmY, &full[s], k * P.kstep, y0);
                    } else {
                        const uint32_t lf = mapa_shared(smem_u32(&full[s]), 0);
                        if (P.x3d)
                            tma_load_3d_pair(a, &tmX, lf, k * P.kstep, (int32_t)u.x_row0, u.batch);
                        else
                            tma_load_2d_pair(a, &tmX, lf, k * P.kstep, (int32_t)u.x_row0);
                        if (P.y3d)
                            tma_load_3d_pair(b, &tmY, lf, k * P.kstep, y0, u.batch);
                        else
                            tma_load_2d_pair(b, &tmY, lf, k * P.kstep, y0);
                    }
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (leader) {
                for (int i = 0; i < S; ++i)
                    if (armed & (1u << i)) wait_bar_drain(&full[i], (armed_par >> i) & 1u, g);
            } else if (!ok) {
                // the odd CTA cannot observe its copies' completion (they land
                // on the leader's barriers); after an abort give them time to land
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 100000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (even CTA) ----------------
            WorkIter w;
            w.init(P.sched, unit_pid(P));
            Unit u;
            int s = 0;
            uint32_t ph = 0, acc_it = 0;
            bool ok = true, issued = false;
            while (ok && next_unit(P, w, u, BN)) {
                const int buf = acc_it & 1;
                const uint32_t aph = (acc_it >> 1) & 1;
                ++acc_it;
                if (!wait_bar(&tempty[buf], aph ^ 1, g, SITE_MMA_TMEM_EMPTY) ||
                    !wait_bar_cluster(&ptempty[buf], aph ^ 1, g, SITE_MMA_TMEM_EMPTY))
                    break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + (uint32_t)(buf * BN);
                // the K loop of one unit, for one MMA kind (chosen once per
                // launch, outside the loop): four instructions per K-step, 32
                // bytes of each operand row apiece
                auto k_loop = [&](auto f8) {
                    for (int k = u.k_begin; k < u.k_end; k += KS) {
                        if (!wait_bar(&full[s], ph, g, SITE_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t a_addr = smem_u32(ring + (size_t)s * stage_bytes);
                        const int nk = u.k_end - k < KS ? u.k_end - k : KS;
                        for (int h = 0; h < nk; ++h) {
                            const uint64_t ad = make_sw128_kmajor_desc(a_addr + h * Cfg::A_BYTES);
                            const uint64_t bd = make_sw128_kmajor_desc(a_addr + a_region + h * Cfg::B_BYTES);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint32_t acc = (k + h > u.k_begin || kk > 0) ? 1u : 0u;
                                if constexpr (decltype(f8)::value)
                                    umma_f8_ss_pair(d, ad + 2 * kk, bd + 2 * kk, P.idesc, acc);
                                else
                                    umma_f16_ss_pair(d, ad + 2 * kk, bd + 2 * kk, P.idesc, acc);
                            }
                        }
                        issued = true;
                        umma_commit_pair_mc(&empty[s], 0x3);
                        if (++s == S) {
                            s = 0;
                            ph ^= 1;
                        }
                    }
                };
                if (P.mma_f8)
                    k_loop(std::true_type{});
                else
                    k_loop(std::false_type{});
                if (!ok) break;
                umma_commit_pair_mc(&tfull[buf], 0x3);
            }
            if (issued) {
                umma_commit_pair_mc(done, 0x1);
                wait_bar_drain(done, 0, g);
            }
        } else if (lane == 0) {
            // ---------------- forwarder (odd CTA) ----------------
            // Tells the leader, in the order its MMA loop waits, that this
            // CTA's accumulator b was released (from the third unit on).
            const uint32_t l_ptempty = mapa_shared(smem_u32(ptempty), 0);
            WorkIter w;
            w.init(P.sched, unit_pid(P));
            Unit u;
            uint32_t acc_it = 0;
            while (next_unit(P, w, u, BN)) {
                const int buf = acc_it & 1;
                const uint32_t aph = (acc_it >> 1) & 1;
                if (acc_it >= 2) {
                    if (!wait_bar(&tempty[buf], aph ^ 1, g, SITE_EPI_TMEM_FULL)) break;
                    mbar_arrive_remote(l_ptempty + 8u * buf);
                }
                ++acc_it;
            }
        }
    } else {
        const FixupSmem fx{ring, (uint32_t)((size_t)S * stage_bytes), fixbar};
        epilogue<BN>(P, &tmC, &tmD, tmem_base, tfull, tempty, esmem, cbar, bcast, fx, g, 64);
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // the leader's MMAs and all cross-CTA arrivals are done
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BN>
cudaError_t launch_pair_bn(const GemmMaps& m, const GemmKernelParams& p, int grid, cudaStream_t st) {
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(umma_pair_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    return launch_pdl(umma_pair_gemm_kernel<BN>, grid, 192, PairCfg<BN>::smem_bytes(p.stages, p.ks), st, m.x, m.y,
                      m.c, m.d, p);
}

template <int BN>
int pair_stages_bn(int ks) {
    return PairCfg<BN>::max_stages(ks);
}

// Clusters of two that can be resident at once with the largest ring.
template <int BN>
int pair_max_clusters_bn() {
    const size_t smem = PairCfg<BN>::smem_bytes(PairCfg<BN>::max_stages(1), 1);
    if (cudaFuncSetAttribute(umma_pair_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, umma_pair_gemm_kernel<BN>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace qg
