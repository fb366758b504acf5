// The dense tcgen05 GEMM kernel for sm_103a.
//
// One persistent, warp-specialised kernel per output-tile width BN serves the
// dense, swapped-operand (decode), batched and grouped problems under the
// data-parallel, split-K and stream-K schedules:
//
//   warp 0      TMA producer: one elected thread streams the 128 x 64 tile of
//               the X operand and the BN x 64 tile of the Y operand into an
//               S-stage shared-memory ring (SWIZZLE_128B), arming full[s] with
//               the transaction bytes and waiting on empty[s].
//   warp 1      allocates TMEM (two BN-column fp32 accumulators) and, from
//               one thread, issues four tcgen05.mma (K = 16 each) per stage,
//               releasing the stage with tcgen05.commit -> empty[s] and the
//               finished accumulator with tcgen05.commit -> tmem_full[b].
//   warps 2-5   epilogue: TMEM -> registers -> fma(alpha, acc, beta*C) ->
//               cast -> global, or the split-K / stream-K partial path.
//
// This replaces the cp.async multi-stage mainloop of "InternLM Lmdeploy Gemm
// MainloopSm80V2" (sections Overview / Description: N-stage ring, prologue and
// steady state, wait for the stage the MMA needs) with the Blackwell data
// path: TMA + mbarrier ring, UMMA from shared memory into TMEM.  Tail tiles
// need no special code: TMA fills out-of-range elements with zeros (the
// zero-fill rule of the DeepGEMM kernel-set blog, section 4.3) and the
// epilogue masks the stores.
#pragma once
#include <atomic>

#include "common.cuh"

namespace qg {

template <int BN>
struct UmmaCfg {
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BYTES = BN * BK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = tmem_cols_for(2 * BN);
    static constexpr uint32_t STAGING_BYTES = EPI_SMEM_BYTES;
    static constexpr int MAX_STAGES = 16;
    static constexpr uint32_t AUX_BYTES = (2 * MAX_STAGES + 5 + FIX_BARS + EPI_CBARS) * 8 + 16;
    static constexpr uint32_t FIXED_BYTES = 1024 /*alignment slack*/ + STAGING_BYTES + AUX_BYTES;
    // a stage holds ks 64-wide K-steps of both operands
    static size_t smem_bytes(int stages, int ks) { return FIXED_BYTES + (size_t)stages * ks * STAGE_BYTES; }
    static int max_stages(int ks) {
        const size_t budget = 232448;  // 227 KB opt-in shared memory per block
        int s = (int)((budget - FIXED_BYTES) / (ks * STAGE_BYTES));
        return s > MAX_STAGES ? MAX_STAGES : s;
    }
};

template <int BN>
__global__ void __launch_bounds__(192, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ GemmKernelParams P) {
    using Cfg = UmmaCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = P.stages;
    const int KS = P.ks;  // K-steps per stage: 1, or 2 with K-chunk tensor maps (one box per operand per stage)
    const uint32_t stage_bytes = (uint32_t)KS * Cfg::STAGE_BYTES;
    const uint32_t a_region = (uint32_t)KS * Cfg::A_BYTES;
    uint8_t* ring = smem;
    float* staging = reinterpret_cast<float*>(smem + (size_t)S * stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes + Cfg::STAGING_BYTES);
    uint64_t* empty = full + Cfg::MAX_STAGES;
    uint64_t* tfull = empty + Cfg::MAX_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint64_t* cbar = done + 1;
    uint64_t* fixbar = cbar + EPI_CBARS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fixbar + FIX_BARS);
    volatile uint32_t* bcast = tmem_slot + 1;
    volatile uint32_t* abort_flag = tmem_slot + 2;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 128);
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
        // warm L2 with the first stages' operands while the previous kernel in
        // the stream finishes (grouped problems read their tile map from memory
        // the previous kernel may write, so they wait)
        if (!P.sched.grouped) {
            WorkIter w;
            w.init(P.sched, blockIdx.x);
            Unit u;
            if (w.next(P.sched, blockIdx.x, BM, BN, u)) {
                const int kend = u.k_end < u.k_begin + S * KS ? u.k_end : u.k_begin + S * KS;
                for (int k = u.k_begin; k < kend; k += KS) {
                    if (KS > 1) {
                        tma_prefetch_l2_3d(&tmX, 0, (int32_t)u.x_row0, k);
                        tma_prefetch_l2_3d(&tmY, 0, (int32_t)u.y_row0, k);
                    } else {
                        if (P.x3d)
                            tma_prefetch_l2_3d(&tmX, k * P.kstep, (int32_t)u.x_row0, u.batch);
                        else
                            tma_prefetch_l2_2d(&tmX, k * P.kstep, (int32_t)u.x_row0);
                        if (P.y3d)
                            tma_prefetch_l2_3d(&tmY, k * P.kstep, (int32_t)u.y_row0, u.batch);
                        else
                            tma_prefetch_l2_2d(&tmY, k * P.kstep, (int32_t)u.y_row0);
                    }
                }
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // set-up (barriers, TMEM, descriptor prefetch) overlaps the previous
    // kernel's tail; no global memory is touched before the previous grid is done
    griddep_launch_dependents();
    griddep_wait();
    const Guard g{P.status, P.timeout_ns, abort_flag};

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            WorkIter w;
            w.init(P.sched, blockIdx.x);
            Unit u;
            int s = 0;
            uint32_t ph = 0, armed = 0, armed_par = 0;
            bool ok = true;
            while (ok && w.next(P.sched, blockIdx.x, BM, BN, u)) {
                for (int k = u.k_begin; k < u.k_end; k += KS) {
                    if (!wait_bar(&empty[s], ph ^ 1, g, SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    uint8_t* a = ring + (size_t)s * stage_bytes;
                    uint8_t* b = a + a_region;
                    mbar_arrive_expect_tx(&full[s], stage_bytes);
                    if (KS > 1) {
                        // K-chunk maps: coordinates (0, row, chunk); past the
                        // last chunk TMA fills zeros and still counts the bytes
                        tma_load_3d(a, &tmX, &full[s], 0, (int32_t)u.x_row0, k);
                        tma_load_3d(b, &tmY, &full[s], 0, (int32_t)u.y_row0, k);
                    } else {
                        if (P.x3d)
                            tma_load_3d(a, &tmX, &full[s], k * P.kstep, (int32_t)u.x_row0, u.batch);
                        else
                            tma_load_2d(a, &tmX, &full[s], k * P.kstep, (int32_t)u.x_row0);
                        if (P.y3d)
                            tma_load_3d(b, &tmY, &full[s], k * P.kstep, (int32_t)u.y_row0, u.batch);
                        else
                            tma_load_2d(b, &tmY, &full[s], k * P.kstep, (int32_t)u.y_row0);
                    }
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            // never leave with copies in flight into this CTA's shared memory
            for (int i = 0; i < S; ++i)
                if (armed & (1u << i)) wait_bar_drain(&full[i], (armed_par >> i) & 1u, g);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            WorkIter w;
            w.init(P.sched, blockIdx.x);
            Unit u;
            int s = 0;
            uint32_t ph = 0, acc_it = 0;
            bool ok = true, issued = false;
            while (ok && w.next(P.sched, blockIdx.x, BM, BN, u)) {
                const int buf = acc_it & 1;
                const uint32_t aph = (acc_it >> 1) & 1;
                ++acc_it;
                if (!wait_bar(&tempty[buf], aph ^ 1, g, SITE_MMA_TMEM_EMPTY)) break;
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
                                    umma_f8_ss(d, ad + 2 * kk, bd + 2 * kk, P.idesc, acc);
                                else
                                    umma_f16_ss(d, ad + 2 * kk, bd + 2 * kk, P.idesc, acc);
                            }
                        }
                        issued = true;
                        umma_commit(&empty[s]);
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
                umma_commit(&tfull[buf]);
            }
            if (issued) {  // every issued MMA has finished before TMEM is freed
                umma_commit(done);
                wait_bar_drain(done, 0, g);
            }
        }
    } else {
        const FixupSmem fx{ring, (uint32_t)((size_t)S * stage_bytes), fixbar};
        epilogue<BN>(P, &tmC, &tmD, tmem_base, tfull, tempty, reinterpret_cast<uint8_t*>(staging), cbar, bcast, fx, g, 64);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BN>
cudaError_t launch_umma_bn(const GemmMaps& m, const GemmKernelParams& p, int grid, cudaStream_t st) {
    const size_t smem = UmmaCfg<BN>::smem_bytes(p.stages, p.ks);
    // raise the dynamic shared-memory limit once per device (to the largest ring)
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(umma_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    return launch_pdl(umma_gemm_kernel<BN>, grid, 192, smem, st, m.x, m.y, m.c, m.d, p);
}

template <int BN>
int umma_stages_bn(int ks) {
    return UmmaCfg<BN>::max_stages(ks);
}

}  // namespace qg
