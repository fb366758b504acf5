// tcgen05 GEMM with in-mainloop operand transforms: int4 dequantisation and
// group-wise scaling (the U/V scale operands that advance at K-group
// boundaries, "InternLM Lmdeploy Gemm MainloopSm80V2", section Description).
//
// Same persistent warp-specialised structure as the dense kernel, plus eight
// transform warps between the TMA ring and the tensor core:
//
//   warp 0      TMA: X tile (128 x 64 16-bit, SWIZZLE_128B, or 128 x 32 bytes
//               of packed int4) and Y tile (BN x 64 16-bit, or BN x 32 bytes
//               of int4) into stage s, arming full[s].
//   warp 1      TMEM owner / MMA issuer; waits ready[s], not full[s].
//   warps 2-5   epilogue (shared with the dense kernel).
//   warps 6-13  transform: wait full[s]; for every 16-byte chunk of 8 K
//               values of a transformed operand, form RN(x * scale) in fp32
//               and write the chunk where the SWIZZLE_128B canonical layout
//               wants it; fence the writes to the async proxy; arrive ready[s].
//
// The product of a nibble or a 16-bit value with an fp16/bf16 scale is exact
// in fp32, so each operand element is rounded exactly once, to the MMA input
// type (A's type).
#pragma once
#include <atomic>

#include "common.cuh"

namespace qg {

template <int BN>
struct DqCfg {
    static constexpr uint32_t X_OP = BM * BK * 2;   // 16 KB
    static constexpr uint32_t Y_OP = BN * BK * 2;
    static constexpr uint32_t X_RAW = BM * 32;      // packed int4 rows
    static constexpr uint32_t Y_RAW = BN * 32;
    // up to 8 scale rows (group 8) of 16-bit scales; the X side's rows are
    // XS_PITCH wide: a copy starts at the 8-aligned column below the tile's
    // first row (a grouped problem's token blocks start anywhere), since a
    // tensor copy's innermost coordinate must be a multiple of 16 bytes
    static constexpr int XS_PITCH = BM + 8;
    static constexpr uint32_t X_SC = XS_PITCH * 2 * 8;
    static constexpr uint32_t Y_SC = BN * 2 * 8;
    static constexpr uint32_t X_ZP = BM * 8;        // up to 8 zero-point rows, one byte per value
    static constexpr uint32_t Y_ZP = BN * 8;
    static constexpr uint32_t STAGE_BYTES =
        ((X_OP + Y_OP + X_RAW + Y_RAW + X_SC + Y_SC + X_ZP + Y_ZP) + 1023) / 1024 * 1024;
    static constexpr uint32_t TMEM_COLS = tmem_cols_for(2 * BN);
    static constexpr uint32_t STAGING_BYTES = EPI_SMEM_BYTES;
    static constexpr int MAX_STAGES = 12;
    static constexpr uint32_t AUX_BYTES = (3 * MAX_STAGES + 5 + FIX_BARS + EPI_CBARS) * 8 + 16;
    static constexpr uint32_t FIXED_BYTES = 1024 + STAGING_BYTES + AUX_BYTES;
    static size_t smem_bytes(int stages) { return FIXED_BYTES + (size_t)stages * STAGE_BYTES; }
    static int max_stages() {
        int s = (int)((232448 - FIXED_BYTES) / STAGE_BYTES);
        return s > MAX_STAGES ? MAX_STAGES : s;
    }
};

__device__ __forceinline__ uint32_t pack2(float a, float b, int out_bf16) {
    if (out_bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack2(uint32_t w, int is_bf16) {
    if (is_bf16) return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
    return __half22float2(*reinterpret_cast<__half2*>(&w));
}

// Chunk i of a transform thread covers 16-byte chunk c = tid + XF_THREADS*i of a
// ROWS x 64 tile: row c/8 and logical K-chunk j (8 values at k0 + 8j).  For a
// packed int4 operand j = c % 8 (the destination is permuted); for a 16-bit
// operand already in the swizzled layout the physical chunk is c % 8 and the
// logical one is (c % 8) ^ (row % 8).
// Transform threads per CTA: eight warps, two per SM sub-partition, so the
// dependent integer/float chains of one warp hide behind the other's.
constexpr int XF_THREADS = 256;

template <int ROWS>
struct XformChunks {
    static constexpr int TOTAL = ROWS * 8;  // 16-byte chunks in a ROWS x 64 tile
    static constexpr int N = (TOTAL + XF_THREADS - 1) / XF_THREADS;  // per transform thread
};

// Scale of row r for logical K-chunk j, from the stage's scale rows
// ([sc_rows][pitch] 16-bit values, the tile's row 0 at column off; row t
// covers K-group k0/group + t).  Branch free so the chunks of a thread
// interleave.
struct ScaleRows {
    const uint8_t* p;
    int pitch, off;
};

__device__ __forceinline__ float stage_scale(const OperandXform& o, const ScaleRows& sc, int r, int j) {
    const int t = o.group >= 64 ? 0 : (8 * j) / o.group;
    const uint32_t bits = reinterpret_cast<const uint16_t*>(sc.p)[t * sc.pitch + sc.off + r];
    const float as_f16 = __half2float(__ushort_as_half((unsigned short)bits));
    const float as_bf16 = __uint_as_float(bits << 16);
    const float v = o.scale_type == DT_F16 ? as_f16 : as_bf16;
    return o.has_scale ? v : 1.0f;
}

// Zero point of row r for logical K-chunk j, from the stage's zero-point rows
// ([sc_rows][ROWS] bytes, laid out like the scale rows): the two's-complement
// value of the byte's low nibble; 0 without zero points.
template <int ROWS>
__device__ __forceinline__ int stage_zero(const OperandXform& o, const uint8_t* zp, int r, int j) {
    const int t = o.group >= 64 ? 0 : (8 * j) / o.group;
    const int z = (int)((uint32_t)zp[t * ROWS + r] << 28) >> 28;
    return o.has_zero ? z : 0;
}

template <bool OUT_BF16>
__device__ __forceinline__ uint32_t pack2t(float a, float b) {
    if constexpr (OUT_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Transform one operand tile of ROWS rows.  op: the SWIZZLE_128B operand
// tile; raw: the packed int4 tile (ROWS x 32 bytes); sc: the scale rows; zp:
// the zero-point rows (int4 only).  All chunks of a thread are independent;
// scales and raw words are read first so their shared-memory latency overlaps.
template <int ROWS, bool INT4, bool OUT_BF16>
__device__ __forceinline__ void transform_tile(const OperandXform& o, uint8_t* op, const uint8_t* raw,
                                               const ScaleRows& sc, const uint8_t* zp, int tid) {
    constexpr int NC = XformChunks<ROWS>::N;
    float s[NC];
    float zoff[NC];  // int4: 2^23 + 8 + z, the bias subtracted from the magic-number float
    uint32_t w[NC];
    uint4 in[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = tid + XF_THREADS * i;
        if (XformChunks<ROWS>::TOTAL % XF_THREADS != 0 && c >= XformChunks<ROWS>::TOTAL) break;
        const int r = c >> 3;
        const int j = INT4 ? (c & 7) : ((c & 7) ^ (r & 7));
        s[i] = stage_scale(o, sc, r, j);
        if constexpr (INT4) {
            w[i] = *reinterpret_cast<const uint32_t*>(raw + r * 32 + 4 * (c & 7));
            zoff[i] = 8388616.0f + (float)stage_zero<ROWS>(o, zp, r, j);  // exact in fp32
        }
        else
            in[i] = *reinterpret_cast<const uint4*>(op + r * 128 + ((c & 7) << 4));
    }
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = tid + XF_THREADS * i;
        if (XformChunks<ROWS>::TOTAL % XF_THREADS != 0 && c >= XformChunks<ROWS>::TOTAL) break;
        const int r = c >> 3;
        uint4 out;
        if constexpr (INT4) {
            // chunk j = c % 8 holds k = k0 + 8j .. +7 (raw bytes 4j .. 4j+3);
            // biased nibble b = q + 8 becomes the float 2^23 + b, so
            // q - z = f - (2^23 + 8 + z), exactly
            const uint32_t x = w[i] ^ 0x88888888u;
            const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
            float q[8];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                q[2 * t] = (__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7650u | t)) - zoff[i]) * s[i];
                q[2 * t + 1] = (__uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7650u | t)) - zoff[i]) * s[i];
            }
            out.x = pack2t<OUT_BF16>(q[0], q[1]);
            out.y = pack2t<OUT_BF16>(q[2], q[3]);
            out.z = pack2t<OUT_BF16>(q[4], q[5]);
            out.w = pack2t<OUT_BF16>(q[6], q[7]);
            *reinterpret_cast<uint4*>(op + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = out;
        } else {
            const uint32_t iw[4] = {in[i].x, in[i].y, in[i].z, in[i].w};
            uint32_t ow[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 f = unpack2(iw[t], OUT_BF16);
                ow[t] = pack2t<OUT_BF16>(f.x * s[i], f.y * s[i]);
            }
            *reinterpret_cast<uint4*>(op + r * 128 + ((c & 7) << 4)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
    }
}

// Scale v split for packed bf16 arithmetic: v = vhi + vlo with both parts
// exact in bf16 (vhi = v's top 8 significant bits, vlo = the rest: at most 3
// bits for an fp16 scale, 0 for a bf16 one).  Returned as two bf16 pairs.
__device__ __forceinline__ void split_scale_bf16(float v, uint32_t& vhi2, uint32_t& vlo2) {
    const uint32_t sb = __float_as_uint(v);
    const uint32_t hb = sb & 0xFFFF0000u;
    const float vlo = (sb & 0x7F800000u) != 0x7F800000u ? v - __uint_as_float(hb) : 0.0f;
    vhi2 = (hb >> 16) * 0x10001u;
    vlo2 = (__float_as_uint(vlo) >> 16) * 0x10001u;
}

// Two int4 values -> RN_bf16((q - z) * v) each, as a bf16 pair.  p holds the
// even K value's nibble in bits 0-3 and the odd one's in bits 16-19 (other
// bits ignored).  (b & 0xF) ^ 8 | 0x4300 is the bf16 number 128 + q + 8;
// off2 holds the bf16 number 136 + z twice (128 + 8 + z, exact for a zero
// point z in [-8, 7]; 136 without one), so q - z is exact after the
// subtraction; (q - z) * vlo is exact in bf16 (<= 4 + 3 significant bits), and
// one fma rounds the exact (q - z) * vhi + (q - z) * vlo = (q - z) * v once.
__device__ __forceinline__ uint32_t int4_off2(int z) { return (0x4300u + (uint32_t)(8 + z)) * 0x10001u; }

__device__ __forceinline__ uint32_t int4_pair_bf16(uint32_t p, uint32_t vhi2, uint32_t vlo2, uint32_t off2) {
    uint32_t m;
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(m) : "r"(p), "r"(0x000F000Fu), "r"(0x43084308u));  // (a & b) ^ c
    const __nv_bfloat162 q2 = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&m),
                                      *reinterpret_cast<const __nv_bfloat162*>(&off2));
    const __nv_bfloat162 r = __hfma2(q2, *reinterpret_cast<const __nv_bfloat162*>(&vhi2),
                                     __hmul2(q2, *reinterpret_cast<const __nv_bfloat162*>(&vlo2)));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// The int4 operand of a stage (ROWS rows x 32 bytes) expanded to a bf16
// SWIZZLE_128B tile, row per thread: threads_per_row = XF_THREADS/ROWS
// clamped to [2, 8] threads share a tile row, each taking 8/threads_per_row
// 16-byte chunks, so a thread reads contiguous raw bytes and, for groups of
// 64 or more, one scale.  Same bits as the chunk-per-thread fp32 formulation
// (RN of the exact product); about 1.7x fewer instructions.
template <int ROWS>
__device__ __forceinline__ void transform_int4_bf16_rows(const OperandXform& o, uint8_t* op, const uint8_t* raw,
                                                         const ScaleRows& sc, const uint8_t* zp, int tid) {
    constexpr int TPR = (XF_THREADS / ROWS) < 2 ? 2 : ((XF_THREADS / ROWS) > 8 ? 8 : (XF_THREADS / ROWS));
    constexpr int CPT = 8 / TPR;                                     // chunks per thread
    constexpr int RPT = (ROWS * TPR + XF_THREADS - 1) / XF_THREADS;  // rows per thread
    constexpr int RSTEP = XF_THREADS / TPR;
    const int sub = tid % TPR;
    const bool per_chunk = o.has_scale && o.group < 64;
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
        const int r = tid / TPR + rr * RSTEP;
        if (ROWS * TPR < XF_THREADS && r >= ROWS) break;
        const uint8_t* src = raw + r * 32 + sub * CPT * 4;
        uint32_t ws[CPT];
        if constexpr (CPT == 4) {
            const uint4 a = *reinterpret_cast<const uint4*>(src);
            ws[0] = a.x; ws[1] = a.y; ws[2] = a.z; ws[3] = a.w;
        } else if constexpr (CPT == 2) {
            const uint2 a = *reinterpret_cast<const uint2*>(src);
            ws[0] = a.x; ws[1] = a.y;
        } else {
            ws[0] = *reinterpret_cast<const uint32_t*>(src);
        }
        uint32_t vhi2 = 0x3F803F80u, vlo2 = 0u;  // unscaled: v = 1
        uint32_t off2 = int4_off2(0);
        if (o.has_scale && !per_chunk) {
            split_scale_bf16(stage_scale(o, sc, r, 0), vhi2, vlo2);
            off2 = int4_off2(stage_zero<ROWS>(o, zp, r, 0));
        }
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int jj = sub * CPT + q;
            if (per_chunk) {
                split_scale_bf16(stage_scale(o, sc, r, jj), vhi2, vlo2);
                off2 = int4_off2(stage_zero<ROWS>(o, zp, r, jj));
            }
            const uint32_t w = ws[q], w4 = w >> 4;
            uint32_t out[4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                out[t] = int4_pair_bf16(__byte_perm(w, w4, (uint32_t)t * 0x11u | (uint32_t)(4 + t) * 0x1100u), vhi2, vlo2,
                                        off2);
            *reinterpret_cast<uint4*>(op + r * 128 + ((jj ^ (r & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
}

template <int ROWS>
__device__ __forceinline__ void transform_any(const OperandXform& o, uint8_t* op, const uint8_t* raw,
                                              const ScaleRows& sc, const uint8_t* zp, int out_bf16, int tid) {
    if (o.int4) {
        if (out_bf16)
            transform_int4_bf16_rows<ROWS>(o, op, raw, sc, zp, tid);
        else
            transform_tile<ROWS, true, false>(o, op, raw, sc, zp, tid);
    } else {
        if (out_bf16)
            transform_tile<ROWS, false, true>(o, op, raw, sc, zp, tid);
        else
            transform_tile<ROWS, false, false>(o, op, raw, sc, zp, tid);
    }
}

// Kernel variants.  DQ_GENERAL decides per launch which operands it
// transforms (and how) and which epilogue form it runs.  DQ_W4A16 is the
// weight-only int4 case with bf16 operands and the TMA epilogue (int4 B with
// group scales and optional zero points, A untouched, 16-bit aligned D): it
// compiles only the packed int4 -> bf16 transform and the TMA epilogue.  The
// smaller kernel keeps its registers (no spills) and its instruction stream
// short; measured on the W4A16 workload (M=128 N=11008 K=4096) it ran 36.3 us
// against 39.3 us for the general kernel.
enum DqMode : int { DQ_GENERAL = 0, DQ_W4A16 = 1 };

template <int BN, int MODE>
__global__ void __launch_bounds__(192 + XF_THREADS, 1)
    umma_dq_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                        const __grid_constant__ CUtensorMap tmXs, const __grid_constant__ CUtensorMap tmYs,
                        const __grid_constant__ CUtensorMap tmZ, const __grid_constant__ GemmKernelParams P) {
    using Cfg = DqCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = P.stages;
    uint8_t* ring = smem;
    float* staging = reinterpret_cast<float*>(smem + (size_t)S * Cfg::STAGE_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * Cfg::STAGE_BYTES + Cfg::STAGING_BYTES);
    uint64_t* ready = full + Cfg::MAX_STAGES;
    uint64_t* empty = ready + Cfg::MAX_STAGES;
    uint64_t* tfull = empty + Cfg::MAX_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint64_t* cbar = done + 1;
    uint64_t* fixbar = cbar + EPI_CBARS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fixbar + FIX_BARS);
    volatile uint32_t* bcast = tmem_slot + 1;
    volatile uint32_t* abort_flag = tmem_slot + 2;

    const DqParams& dq = P.dq;
    const uint32_t x_bytes = (dq.x.int4 ? Cfg::X_RAW : Cfg::X_OP) +
                             (dq.x.has_scale ? Cfg::XS_PITCH * 2 * dq.x.sc_rows : 0) +
                             (dq.x.has_zero ? BM * dq.x.sc_rows : 0);
    const uint32_t y_bytes = (dq.y.int4 ? Cfg::Y_RAW : Cfg::Y_OP) + (dq.y.has_scale ? BN * 2 * dq.y.sc_rows : 0) +
                             (dq.y.has_zero ? BN * dq.y.sc_rows : 0);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&ready[s], XF_THREADS / 32);  // one arrival per transform warp
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
        if (P.dq.x.has_scale) tma_prefetch_desc(&tmXs);
        if (P.dq.y.has_scale) tma_prefetch_desc(&tmYs);
        if (P.dq.x.has_zero || P.dq.y.has_zero) tma_prefetch_desc(&tmZ);
        // warm L2 with the first stages' operands while the previous kernel in
        // the stream finishes (not for grouped problems: their tile map reads
        // memory the previous kernel may write)
        if (!P.sched.grouped) {
            WorkIter w;
            w.init(P.sched, blockIdx.x);
            Unit u;
            if (w.next(P.sched, blockIdx.x, BM, BN, u)) {
                const int kend = u.k_end < u.k_begin + S ? u.k_end : u.k_begin + S;
                for (int k = u.k_begin; k < kend; ++k) {
                    tma_prefetch_l2_2d(&tmX, P.dq.x.int4 ? k * (BK / 2) : k * BK, (int32_t)u.x_row0);
                    tma_prefetch_l2_2d(&tmY, P.dq.y.int4 ? k * (BK / 2) : k * BK, (int32_t)u.y_row0);
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

    auto x_op = [&](int s) { return ring + (size_t)s * Cfg::STAGE_BYTES; };
    auto y_op = [&](int s) { return x_op(s) + Cfg::X_OP; };
    auto x_raw = [&](int s) { return y_op(s) + Cfg::Y_OP; };
    auto y_raw = [&](int s) { return x_raw(s) + Cfg::X_RAW; };
    auto x_sc = [&](int s) { return y_raw(s) + Cfg::Y_RAW; };
    auto y_sc = [&](int s) { return x_sc(s) + Cfg::X_SC; };
    auto x_zp = [&](int s) { return y_sc(s) + Cfg::Y_SC; };
    auto y_zp = [&](int s) { return x_zp(s) + Cfg::X_ZP; };

    if (warp == 0) {
        if (lane == 0) {
            WorkIter w;
            w.init(P.sched, blockIdx.x);
            Unit u;
            int s = 0;
            uint32_t ph = 0, armed = 0, armed_par = 0;
            bool ok = true;
            while (ok && w.next(P.sched, blockIdx.x, BM, BN, u)) {
                for (int k = u.k_begin; k < u.k_end; ++k) {
                    if (!wait_bar(&empty[s], ph ^ 1, g, SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], x_bytes + y_bytes);
                    // int4 tiles are addressed in bytes: K-step k starts at byte k*32
                    if (dq.x.int4)
                        tma_load_2d(x_raw(s), &tmX, &full[s], k * (BK / 2), (int32_t)u.x_row0);
                    else
                        tma_load_2d(x_op(s), &tmX, &full[s], k * BK, (int32_t)u.x_row0);
                    // a grouped problem's Y operand, scales and zero points
                    // carry the expert as their last coordinate
                    const int32_t yr = (int32_t)u.y_row0;
                    if (P.y3d) {
                        if (dq.y.int4)
                            tma_load_3d(y_raw(s), &tmY, &full[s], k * (BK / 2), yr, u.batch);
                        else
                            tma_load_3d(y_op(s), &tmY, &full[s], k * BK, yr, u.batch);
                    } else if (dq.y.int4) {
                        tma_load_2d(y_raw(s), &tmY, &full[s], k * (BK / 2), yr);
                    } else {
                        tma_load_2d(y_op(s), &tmY, &full[s], k * BK, yr);
                    }
                    // the scale (and zero-point) rows of this K-step: groups
                    // (k*64)/group .. + sc_rows - 1
                    if (dq.x.has_scale)  // from the 8-aligned column at or below the tile's first row
                        tma_load_2d(x_sc(s), &tmXs, &full[s], (int32_t)(u.x_row0 & ~int64_t(7)), (k * BK) / dq.x.group);
                    if (dq.x.has_zero)
                        tma_load_2d(x_zp(s), &tmZ, &full[s], (int32_t)u.x_row0, (k * BK) / dq.x.group);
                    if (dq.y.has_scale) {
                        if (P.y3d)
                            tma_load_3d(y_sc(s), &tmYs, &full[s], yr, (k * BK) / dq.y.group, u.batch);
                        else
                            tma_load_2d(y_sc(s), &tmYs, &full[s], yr, (k * BK) / dq.y.group);
                    }
                    if (dq.y.has_zero) {
                        if (P.y3d)
                            tma_load_3d(y_zp(s), &tmZ, &full[s], yr, (k * BK) / dq.y.group, u.batch);
                        else
                            tma_load_2d(y_zp(s), &tmZ, &full[s], yr, (k * BK) / dq.y.group);
                    }
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            for (int i = 0; i < S; ++i)
                if (armed & (1u << i)) wait_bar_drain(&full[i], (armed_par >> i) & 1u, g);
        }
    } else if (warp == 1) {
        if (lane == 0) {
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
                for (int k = u.k_begin; k < u.k_end; ++k) {
                    if (!wait_bar(&ready[s], ph, g, SITE_MMA_OPERAND)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t ad = make_sw128_kmajor_desc(smem_u32(x_op(s)));
                    const uint64_t bd = make_sw128_kmajor_desc(smem_u32(y_op(s)));
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        umma_f16_ss(d, ad + 2 * kk, bd + 2 * kk, P.idesc, (k > u.k_begin || kk > 0) ? 1u : 0u);
                    issued = true;
                    umma_commit(&empty[s]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[buf]);
            }
            if (issued) {
                umma_commit(done);
                wait_bar_drain(done, 0, g);
            }
        }
    } else if (warp < 6) {
        const FixupSmem fx{ring, (uint32_t)((size_t)S * Cfg::STAGE_BYTES), fixbar};
        if constexpr (MODE == DQ_W4A16)
            epilogue_tma<BN>(P, &tmC, &tmD, tmem_base, tfull, tempty, reinterpret_cast<uint8_t*>(staging), cbar, bcast,
                             fx, g, 64);
        else
            epilogue<BN>(P, &tmC, &tmD, tmem_base, tfull, tempty, reinterpret_cast<uint8_t*>(staging), cbar, bcast, fx,
                         g, 64);
    } else {
        // transform warps
        const int tid = threadIdx.x - 192;
        WorkIter w;
        w.init(P.sched, blockIdx.x);
        Unit u;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        while (ok && w.next(P.sched, blockIdx.x, BM, BN, u)) {
            for (int k = u.k_begin; k < u.k_end; ++k) {
                // warp-uniform outcome, so no lane is left behind at the
                // __syncwarp below when another lane's wait gives up
                if (!__all_sync(0xffffffffu, wait_bar(&full[s], ph, g, SITE_DQ_RAW))) {
                    ok = false;
                    break;
                }
                if constexpr (MODE == DQ_W4A16) {
                    transform_int4_bf16_rows<BN>(dq.y, y_op(s), y_raw(s), ScaleRows{y_sc(s), BN, 0}, y_zp(s), tid);
                } else {
                    if (dq.x.active)
                        transform_any<BM>(dq.x, x_op(s), x_raw(s),
                                          ScaleRows{x_sc(s), Cfg::XS_PITCH, (int)(u.x_row0 & 7)}, x_zp(s),
                                          dq.out_bf16, tid);
                    if (dq.y.active)
                        transform_any<BN>(dq.y, y_op(s), y_raw(s), ScaleRows{y_sc(s), BN, 0}, y_zp(s), dq.out_bf16,
                                          tid);
                }
                // each thread orders its generic-proxy writes before the
                // tensor core's reads; the warp then arrives once
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ready[s]);
                if (++s == S) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// Raise a kernel's dynamic shared-memory limit once per device (to the
// largest ring).
template <typename K>
static cudaError_t configure_dq_once(K kernel, std::atomic<uint64_t>& configured, size_t max_smem) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    return cudaSuccess;
}

// Whether a launch is the W4A16 case that the DQ_W4A16 variant serves.
template <int BN>
static bool dq_w4a16_launch(const GemmKernelParams& p) {
    return BN >= 32 && p.epi.tma && p.dq.y.int4 && p.dq.out_bf16 && !p.dq.x.active;
}

template <int BN>
cudaError_t launch_dq_bn(const GemmMaps& m, const GemmKernelParams& p, int grid, cudaStream_t st) {
    const size_t smem = DqCfg<BN>::smem_bytes(p.stages);
    const size_t max_smem = DqCfg<BN>::smem_bytes(DqCfg<BN>::max_stages());
    static std::atomic<uint64_t> configured[2] = {{0}, {0}};
    if constexpr (BN >= 32) {
        if (dq_w4a16_launch<BN>(p)) {
            cudaError_t e = configure_dq_once(umma_dq_gemm_kernel<BN, DQ_W4A16>, configured[1], max_smem);
            if (e != cudaSuccess) return e;
            return launch_pdl(umma_dq_gemm_kernel<BN, DQ_W4A16>, grid, 192 + XF_THREADS, smem, st, m.x, m.y, m.c, m.d,
                              m.xs, m.ys, m.z, p);
        }
    }
    cudaError_t e = configure_dq_once(umma_dq_gemm_kernel<BN, DQ_GENERAL>, configured[0], max_smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(umma_dq_gemm_kernel<BN, DQ_GENERAL>, grid, 192 + XF_THREADS, smem, st, m.x, m.y, m.c, m.d, m.xs,
                      m.ys, m.z, p);
}

template <int BN>
int dq_stages_bn() {
    return DqCfg<BN>::max_stages();
}

}  // namespace qg
