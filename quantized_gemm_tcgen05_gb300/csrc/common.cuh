// Device pieces shared by the tcgen05 GEMM kernels: bounded waits with the
// device status record, the persistent-unit iteration, and the epilogue
// (TMEM -> registers -> alpha/beta/cast -> global), including the split-K /
// stream-K partial write and the last-arriver reduction.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kparams.h"
#include "ptx.cuh"

namespace qg {

constexpr int BM = 128;  // UMMA M: rows of the X operand per tile (TMEM lanes)
constexpr int BK = 64;   // K per pipeline stage: one 128-byte swizzle row of 16-bit values
constexpr int UMMA_K = 16;

// ---- bounded waits -------------------------------------------------------------

struct Guard {
    uint32_t* status;
    uint64_t limit_ns;
    volatile uint32_t* abort;  // shared flag: once set, every role stops waiting
};

static __device__ __noinline__ void record_timeout(const Guard& g, uint32_t site) {
    *g.abort = 1u;
    if (g.status) {
        atomicExch(&g.status[1], site);
        atomicExch(&g.status[2], blockIdx.x);
        atomicAdd(&g.status[3], 1u);
        atomicOr(&g.status[0], 1u);
    }
}

// Wait until the phase of `bar` with parity `parity` has completed.  Gives
// up (returns false) when another role aborted or after g.limit_ns.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Guard& g, uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*g.abort) return false;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 31u) == 0) {
            if (*g.abort) return false;
            if (globaltimer_ns() - t0 > g.limit_ns) {
                record_timeout(g, site);
                return false;
            }
        }
    }
}

// Wait used when a role drains its own in-flight work before exit: bounded,
// and it does not stop early on abort.
__device__ __forceinline__ bool wait_bar_drain(uint64_t* bar, uint32_t parity, const Guard& g) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > g.limit_ns) {
            record_timeout(g, SITE_DRAIN);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// ---- element access ------------------------------------------------------------------

__device__ __forceinline__ float ld_elem(const void* p, int32_t t, int64_t i) {
    if (t == DT_F32) return static_cast<const float*>(p)[i];
    if (t == DT_F16) return __half2float(static_cast<const __half*>(p)[i]);
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ __forceinline__ void st_elem(void* p, int32_t t, int64_t i, float x) {
    if (t == DT_F32)
        static_cast<float*>(p)[i] = x;
    else if (t == DT_F16)
        static_cast<__half*>(p)[i] = __float2half_rn(x);
    else
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
}

// Four consecutive elements, 16-byte (f32) or 8-byte (16-bit) aligned.
__device__ __forceinline__ float4 ld4(const void* p, int32_t t, int64_t i) {
    if (t == DT_F32) return *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i);
    float4 r;
    if (t == DT_F16) {
        float2 a = __half22float2(*reinterpret_cast<__half2*>(&raw.x));
        float2 b = __half22float2(*reinterpret_cast<__half2*>(&raw.y));
        r = make_float4(a.x, a.y, b.x, b.y);
    } else {
        float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.x));
        float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.y));
        r = make_float4(a.x, a.y, b.x, b.y);
    }
    return r;
}

__device__ __forceinline__ void st4(void* p, int32_t t, int64_t i, float4 v) {
    if (t == DT_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p) + i) = v;
        return;
    }
    uint2 raw;
    if (t == DT_F16) {
        __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        raw.x = *reinterpret_cast<uint32_t*>(&a);
        raw.y = *reinterpret_cast<uint32_t*>(&b);
    } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        raw.x = *reinterpret_cast<uint32_t*>(&a);
        raw.y = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p) + i) = raw;
}

__device__ __forceinline__ float epi_value(const EpiParams& e, float acc, float c) {
    return e.beta != 0.0f ? fmaf(e.alpha, acc, e.beta * c) : e.alpha * acc;
}

// ---- epilogue --------------------------------------------------------------------------

// Column chunk handled per TMEM load: 32 fp32 columns (16 when BN is 16).
template <int BN>
struct Chunk {
    static constexpr int W = BN < 32 ? BN : 32;
    static constexpr int N = BN / W;
    static constexpr int Q = W / 4;  // float4 quads per row
};

template <int W>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float (&v)[W]) {
    if constexpr (W == 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    } else {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
    }
}

// The C values one thread combines for one chunk, loaded before they are
// needed so the epilogue does not wait on global-memory latency per row.
template <int W>
struct CChunk {
    float v[W];
};

// Row-per-thread layout (non-swapped): iteration `it` of a thread covers tile
// row ew*32 + it*(32/Q) + lane/Q and the 4 columns 4*(lane%Q) .. +3.
template <int W>
__device__ __forceinline__ void load_c_chunk(const EpiParams& e, const Unit& u, int ew, int lane, int col0,
                                             CChunk<W>& cc) {
    if (e.beta == 0.0f) return;
    constexpr int Q = W / 4;
    const int64_t boff_c = (int64_t)u.batch * e.c_bstride;
    if (e.swap) {
        const int64_t n = u.x_row0 + ew * 32 + lane;
        const bool nok = n < e.N && ew * 32 + lane < u.x_rows;
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const int64_t m = u.y_row0 + col0 + j;
            cc.v[j] = (nok && m < e.M) ? ld_elem(e.C, e.d_type, boff_c + m * e.ldc + n) : 0.0f;
        }
        return;
    }
    constexpr int ROWS_PER_IT = 32 / Q;
#pragma unroll
    for (int it = 0; it < Q; ++it) {
        const int rr = it * ROWS_PER_IT + lane / Q;
        const int j = lane % Q;
        const int rt = ew * 32 + rr;
        const int64_t m = u.x_row0 + rt;
        const int64_t n0 = u.y_row0 + col0 + 4 * j;
        float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rt < u.x_rows && m < e.M && n0 < e.N) {
            const int64_t ci = boff_c + m * e.ldc + n0;
            if (e.vec_ok && n0 + 3 < e.N) {
                c = ld4(e.C, e.d_type, ci);
            } else {
                c.x = ld_elem(e.C, e.d_type, ci);
                if (n0 + 1 < e.N) c.y = ld_elem(e.C, e.d_type, ci + 1);
                if (n0 + 2 < e.N) c.z = ld_elem(e.C, e.d_type, ci + 2);
                if (n0 + 3 < e.N) c.w = ld_elem(e.C, e.d_type, ci + 3);
            }
        }
        cc.v[4 * it] = c.x;
        cc.v[4 * it + 1] = c.y;
        cc.v[4 * it + 2] = c.z;
        cc.v[4 * it + 3] = c.w;
    }
}

// Store one chunk of W accumulator columns held by this thread for tile row
// r = ew*32 + lane, combined with the prefetched C values.  `staging` is this
// warp's private 32 x W fp32 buffer (swizzled by 16-byte quads) that turns the
// row-per-thread TMEM layout into row-contiguous global stores.
template <int W>
__device__ __forceinline__ void store_chunk(const EpiParams& e, const Unit& u, int ew, int lane, int col0,
                                            const float (&v)[W], const CChunk<W>& cc, float4* staging) {
    constexpr int Q = W / 4;
    const int64_t boff_d = (int64_t)u.batch * e.d_bstride;
    if (e.swap) {
        // tile row -> output column n; tile column -> output row m.  Lanes
        // hold consecutive n, so each store instruction is row-contiguous.
        const int64_t n = u.x_row0 + ew * 32 + lane;
        if (n >= e.N || ew * 32 + lane >= u.x_rows) return;
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const int64_t m = u.y_row0 + col0 + j;
            if (m < e.M) st_elem(e.D, e.d_type, boff_d + m * e.ldd + n, epi_value(e, v[j], cc.v[j]));
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < Q; ++j)
        staging[lane * Q + (j ^ (lane & (Q - 1)))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    constexpr int ROWS_PER_IT = 32 / Q;
#pragma unroll
    for (int it = 0; it < Q; ++it) {
        const int rr = it * ROWS_PER_IT + lane / Q;  // row within this warp's 32
        const int j = lane % Q;
        const float4 a = staging[rr * Q + (j ^ (rr & (Q - 1)))];
        const int rt = ew * 32 + rr;                 // row within the tile
        const int64_t m = u.x_row0 + rt;
        const int64_t n0 = u.y_row0 + col0 + 4 * j;
        if (rt >= u.x_rows || m >= e.M || n0 >= e.N) continue;
        const int64_t di = boff_d + m * e.ldd + n0;
        const float4 o = make_float4(epi_value(e, a.x, cc.v[4 * it]), epi_value(e, a.y, cc.v[4 * it + 1]),
                                     epi_value(e, a.z, cc.v[4 * it + 2]), epi_value(e, a.w, cc.v[4 * it + 3]));
        if (e.vec_ok && n0 + 3 < e.N) {
            st4(e.D, e.d_type, di, o);
        } else {
            const float ov[4] = {o.x, o.y, o.z, o.w};
            for (int q = 0; q < 4 && n0 + q < e.N; ++q) st_elem(e.D, e.d_type, di + q, ov[q]);
        }
    }
    __syncwarp();
}

// Partial tile layout in the workspace: for chunk c and quad j, the 128 rows'
// float4 values are contiguous, so a warp's 32 lanes write 512 bytes at once.
template <int BN>
__device__ __forceinline__ float4* partial_quad(float* partials, int64_t slot, int c, int j, int r) {
    constexpr int Q = Chunk<BN>::Q;
    return reinterpret_cast<float4*>(partials + slot * (int64_t)(BM * BN)) + ((int64_t)(c * Q + j) * BM + r);
}

// The epilogue role: 4 warps (128 threads), warp w reads TMEM lanes
// 32*(w%4) .. 32*(w%4)+31.  For every unit: wait for the accumulator, then
// either store it (whole tile) or write it as a partial and, if this unit is
// the last of its tile to arrive, reduce all partials in K order and store.
template <int BN>
__device__ void epilogue_role(const GemmKernelParams& P, uint32_t tmem_base, uint64_t* tfull, uint64_t* tempty,
                              float* staging_all, volatile uint32_t* bcast, const Guard& g) {
    using CK = Chunk<BN>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ew = warp % 4;
    const int r = ew * 32 + lane;
    float4* staging = reinterpret_cast<float4*>(staging_all) + ew * 32 * CK::Q;
    WorkIter w;
    w.init(P.sched, blockIdx.x);
    Unit u;
    uint32_t acc_it = 0;
    while (w.next(P.sched, blockIdx.x, BM, BN, u)) {
        const int buf = acc_it & 1;
        const uint32_t aph = (acc_it >> 1) & 1;
        ++acc_it;
        if (!wait_bar(&tfull[buf], aph, g, SITE_EPI_TMEM_FULL)) break;
        tc_fence_after_sync();
        const uint32_t tbase = tmem_base + (uint32_t)(buf * BN) + ((uint32_t)(ew * 32) << 16);
        if (u.mode == UNIT_FULL) {
            // C for chunk c+1 is fetched while chunk c is stored (two buffers,
            // alternated by a two-step loop so they stay in registers)
            CChunk<CK::W> c0, c1;
            load_c_chunk<CK::W>(P.epi, u, ew, lane, 0, c0);
#pragma unroll 1
            for (int c = 0; c < CK::N; c += 2) {
                if (c + 1 < CK::N) load_c_chunk<CK::W>(P.epi, u, ew, lane, (c + 1) * CK::W, c1);
                {
                    float v[CK::W];
                    tmem_load_chunk<CK::W>(tbase + c * CK::W, v);
                    if (c == CK::N - 1) {
                        tc_fence_before_sync();
                        mbar_arrive(&tempty[buf]);
                    }
                    store_chunk<CK::W>(P.epi, u, ew, lane, c * CK::W, v, c0, staging);
                }
                if (c + 1 < CK::N) {
                    if (c + 2 < CK::N) load_c_chunk<CK::W>(P.epi, u, ew, lane, (c + 2) * CK::W, c0);
                    float v[CK::W];
                    tmem_load_chunk<CK::W>(tbase + (c + 1) * CK::W, v);
                    if (c + 1 == CK::N - 1) {
                        tc_fence_before_sync();
                        mbar_arrive(&tempty[buf]);
                    }
                    store_chunk<CK::W>(P.epi, u, ew, lane, (c + 1) * CK::W, v, c1, staging);
                }
            }
            continue;
        }
        // partial unit
#pragma unroll 1
        for (int c = 0; c < CK::N; ++c) {
            float v[CK::W];
            tmem_load_chunk<CK::W>(tbase + c * CK::W, v);
#pragma unroll
            for (int j = 0; j < CK::Q; ++j)
                *partial_quad<BN>(P.partials, u.slot, c, j, r) =
                    make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        tc_fence_before_sync();
        mbar_arrive(&tempty[buf]);
        __threadfence();
        epi_bar_sync();
        if (threadIdx.x == 64) {
            const int old = atomicAdd(&P.counters[u.tile], 1);
            const bool last = (old == u.ncontrib - 1);
            if (last) atomicExch(&P.counters[u.tile], 0);  // every contributor has arrived
            *bcast = last ? 1u : 0u;
        }
        epi_bar_sync();
        if (*bcast == 0u) continue;
        __threadfence();
#pragma unroll 1
        for (int c = 0; c < CK::N; ++c) {
            CChunk<CK::W> cc;
            load_c_chunk<CK::W>(P.epi, u, ew, lane, c * CK::W, cc);
            float v[CK::W];
#pragma unroll
            for (int i = 0; i < CK::W; ++i) v[i] = 0.0f;
            // contributors in K order, two at a time so their loads overlap
#pragma unroll 1
            for (int q0 = 0; q0 < u.ncontrib; q0 += 2) {
                const bool two = q0 + 1 < u.ncontrib;
                const int64_t s0 = partial_slot(P.sched, u.tile, q0);
                const int64_t s1 = two ? partial_slot(P.sched, u.tile, q0 + 1) : s0;
                float4 p0[CK::Q], p1[CK::Q];
#pragma unroll
                for (int j = 0; j < CK::Q; ++j) {
                    p0[j] = __ldcg(partial_quad<BN>(P.partials, s0, c, j, r));
                    p1[j] = __ldcg(partial_quad<BN>(P.partials, s1, c, j, r));
                }
#pragma unroll
                for (int j = 0; j < CK::Q; ++j) {
                    v[4 * j] += p0[j].x;
                    v[4 * j + 1] += p0[j].y;
                    v[4 * j + 2] += p0[j].z;
                    v[4 * j + 3] += p0[j].w;
                }
                if (two) {
#pragma unroll
                    for (int j = 0; j < CK::Q; ++j) {
                        v[4 * j] += p1[j].x;
                        v[4 * j + 1] += p1[j].y;
                        v[4 * j + 2] += p1[j].z;
                        v[4 * j + 3] += p1[j].w;
                    }
                }
            }
            store_chunk<CK::W>(P.epi, u, ew, lane, c * CK::W, v, cc, staging);
        }
    }
}

}  // namespace qg
