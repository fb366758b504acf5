// Device pieces shared by the tcgen05 GEMM kernels: bounded waits with the
// device status record, the persistent-unit iteration, and the epilogue
// (TMEM -> registers -> alpha/beta/cast -> global), including the split-K /
// stream-K partial write and the last-arriver reduction.
#pragma once
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdlib.h>
#include <string.h>

#include <utility>

#include "kparams.h"
#include "ptx.cuh"

namespace qg {

constexpr int BM = 128;  // UMMA M: rows of the X operand per tile (TMEM lanes)
constexpr int BK = 64;   // K per pipeline stage: one 128-byte swizzle row of 16-bit values
constexpr int UMMA_K = 16;
// Shared memory the epilogue owns: 16 KB of staging (register path) or the
// per-warp C/D tile buffers (TMA path), whichever the launch uses.
constexpr uint32_t EPI_SMEM_BYTES = 32 * 1024;
constexpr int EPI_CBARS = 16;  // 4 epilogue warps x up to 4 buffers
constexpr int FIX_BARS = 4;    // completion barriers of the split-tile reduction's bulk copies

// TMEM is allocated in power-of-two column counts of at least 32.
__host__ __device__ constexpr uint32_t tmem_cols_for(uint32_t cols) {
    uint32_t n = 32;
    while (n < cols) n *= 2;
    return n;
}

// ---- launches ------------------------------------------------------------------

// Programmatic dependent launch is on unless GEMM_PDL=0: a GEMM kernel may
// then be scheduled while the previous kernel in the stream finishes, doing
// its set-up early; it waits for that kernel before touching memory.
inline bool pdl_enabled() {
    static const bool on = [] {
        const char* e = getenv("GEMM_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

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

// ---- device-side bounds checks (debug build) ------------------------------------
//
// Built with QG_DEVICE_CHECKS (the checked library, GEMM_DEVICE_CHECKS=1 at
// build time), every unit's tile coordinates, K range, partial slots and tile
// counter are checked against the problem and the workspace the host passed,
// and every element the register epilogue reads or writes against C's / D's
// extent.  A failed check records its site in the device status words (bit 1
// of the first word) and the access is skipped, so the kernel never touches
// memory outside its operands; gemm_device_status then reports it.  The
// regular build compiles none of this.
#ifdef QG_DEVICE_CHECKS
constexpr bool kDeviceChecks = true;
#else
constexpr bool kDeviceChecks = false;
#endif

static __device__ __noinline__ void record_check(uint32_t* status, uint32_t site) {
    if (!status) return;
    atomicExch(&status[1], site);
    atomicExch(&status[2], blockIdx.x);
    atomicAdd(&status[3], 1u);
    atomicOr(&status[0], 2u);
}

// ---- unit iteration shared by all roles ----------------------------------------
//
// A 1-CTA kernel walks 128-row tiles with program id blockIdx.x.  The CTA-pair
// kernel walks 256-row tiles with program id = cluster id; each CTA of the
// pair owns 128 of the rows (the odd CTA the upper half).

__device__ __forceinline__ int unit_pid(const GemmKernelParams& P) {
    return P.pair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
}

static __device__ bool unit_in_bounds(const GemmKernelParams& P, const Unit& u, int bn);

__device__ __forceinline__ bool next_unit(const GemmKernelParams& P, WorkIter& w, Unit& u, int bn) {
    if (!P.pair) {
        if (!w.next(P.sched, (int)blockIdx.x, BM, bn, u)) return false;
    } else {
        if (!w.next(P.sched, (int)(blockIdx.x >> 1), 2 * BM, bn, u)) return false;
        const int32_t half = (int32_t)(blockIdx.x & 1);
        u.x_row0 += (int64_t)half * BM;
        // a grouped 256-row block may hold fewer rows of its expert: each CTA
        // keeps its share (possibly none; the epilogue then stores nothing)
        const int32_t rows = P.sched.grouped ? u.x_rows - half * BM : BM;
        u.x_rows = rows < 0 ? 0 : (rows > BM ? BM : rows);
    }
    if constexpr (kDeviceChecks) {
        if (!unit_in_bounds(P, u, bn)) return false;  // recorded; this role stops
    }
    return true;
}

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

// Output quantisation for an int8 D (DeepGEMM kernel-set blog, section 6.2):
// round(x * scale + zp) with one fp32 fma, nearest-even, saturated to int8
// (a NaN becomes 0, as the conversion defines).
__device__ __forceinline__ int32_t quant_s8(float x, float scale, int32_t zp) {
    const int32_t q = __float2int_rn(fmaf(x, scale, (float)zp));
    return q < -128 ? -128 : (q > 127 ? 127 : q);
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

// Eight consecutive 16-bit elements (F16 or BF16), 16-byte aligned.
__device__ __forceinline__ void ld8(const void* p, int32_t t, int64_t i, float (&o)[8]) {
    const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p) + i);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = t == DT_F16 ? __half22float2(*reinterpret_cast<const __half2*>(&w[q]))
                                     : __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
        o[2 * q] = f.x;
        o[2 * q + 1] = f.y;
    }
}

__device__ __forceinline__ void st8(void* p, int32_t t, int64_t i, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (t == DT_F16) {
            const __half2 h = __floats2half2_rn(v[2 * q], v[2 * q + 1]);
            w[q] = *reinterpret_cast<const uint32_t*>(&h);
        } else {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
            w[q] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p) + i) = make_uint4(w[0], w[1], w[2], w[3]);
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

// Bias of output column n for the fused epilogue: 0 without the bias flag
// and for columns past N (a tile's overhang).  Callers load it once per
// column and chunk, not per element.
__device__ __forceinline__ float bias_at(const EpiParams& e, int64_t n) {
    return ((e.flags & EPI_BIAS) && n < e.N) ? ld_elem(e.bias, e.bias_type, n) : 0.0f;
}

// Store one output value of row m at element index i: rounded to D's type, or
// (Q8) quantised with the row's scale for an int8 D.  Callers choose Q8 once
// per chunk, so the float store carries no extra per-element test.
// Checked build: element index i (and the three after it for a vector access)
// inside extent; records and returns false otherwise.
__device__ __forceinline__ bool elem_in_bounds(const EpiParams& e, int64_t i, int64_t n, int64_t extent) {
    if constexpr (kDeviceChecks) {
        if (i < 0 || i + n > extent) {
            record_check(e.status, CHECK_ELEMENT);
            return false;
        }
    }
    return true;
}

template <bool Q8 = true>
__device__ __forceinline__ void store_out(const EpiParams& e, int64_t i, float x, int64_t m) {
    if (!elem_in_bounds(e, i, 1, e.d_extent)) return;
    if (Q8 && e.d_type == DT_S8)
        static_cast<int8_t*>(e.D)[i] = (int8_t)quant_s8(x, e.qscale[m], e.qzp);
    else
        st_elem(e.D, e.d_type, i, x);
}

// Four consecutive values of row m (aligned as st4 needs; 4 bytes for int8).
template <bool Q8 = true>
__device__ __forceinline__ void store_out4(const EpiParams& e, int64_t i, float4 v, int64_t m) {
    if (!elem_in_bounds(e, i, 4, e.d_extent)) return;
    if (Q8 && e.d_type == DT_S8) {
        const float s = e.qscale[m];
        const uint32_t b = (uint32_t)(quant_s8(v.x, s, e.qzp) & 0xFF) | ((uint32_t)(quant_s8(v.y, s, e.qzp) & 0xFF) << 8) |
                           ((uint32_t)(quant_s8(v.z, s, e.qzp) & 0xFF) << 16) |
                           ((uint32_t)(quant_s8(v.w, s, e.qzp) & 0xFF) << 24);
        *reinterpret_cast<uint32_t*>(static_cast<int8_t*>(e.D) + i) = b;
    } else {
        st4(e.D, e.d_type, i, v);
    }
}

// Bring the bias of a unit's output columns into L1 before its accumulator is
// ready, so the epilogue's per-chunk bias loads hit L1 (a first touch costs
// about a microsecond under load).  Lane l prefetches the 128-byte line of
// columns first + 32 l .. ; 32 lines cover the widest tile (256 columns) and
// the 128 rows of a swapped one.
__device__ __forceinline__ void prefetch_bias(const EpiParams& e, int64_t first, int64_t count, int lane) {
    if (!(e.flags & EPI_BIAS)) return;
    const int64_t es = e.bias_type == DT_F32 ? 4 : 2;
    const int64_t per_line = 128 / es;
    const int64_t n = first + per_line * lane;
    if (lane * per_line < count && n < e.N) {
        const char* a = static_cast<const char*>(e.bias) + n * es;
        asm volatile("prefetch.global.L1 [%0];" ::"l"(a));
    }
}

// Bring the C block a unit combines into L2 before its accumulator is ready,
// so the register epilogue's per-chunk C loads do not each wait on HBM.  This
// warp's share: its 32 tile rows (output rows, or output columns when the
// operands are swapped) across the tile's bn columns; one prefetch per
// 128-byte line, spread over the lanes.
__device__ __forceinline__ void prefetch_c_l2(const EpiParams& e, const Unit& u, int ew, int lane, int bn) {
    if (e.beta == 0.0f || e.C == nullptr) return;
    const int64_t es = e.d_type == DT_F32 ? 4 : 2;
    const char* base = static_cast<const char*>(e.C) + (int64_t)u.batch * e.c_bstride * es;
    if (!e.swap) {
        // rows x_row0 + ew*32 .. +31, columns y_row0 .. +bn
        const int64_t row_bytes = (e.N - u.y_row0 < bn ? e.N - u.y_row0 : bn) * es;
        const int lines = (int)((row_bytes + 127) / 128);
        for (int i = lane; i < 32 * lines; i += 32) {
            const int rt = ew * 32 + i / lines;
            const int64_t m = u.x_row0 + rt;
            if (rt >= u.x_rows || m >= e.M) continue;
            const char* a = base + (m * e.ldc + u.y_row0) * es + (int64_t)(i % lines) * 128;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        }
    } else {
        // output rows y_row0 .. +bn, columns x_row0 + ew*32 .. +31
        const int64_t n0 = u.x_row0 + ew * 32;
        if (n0 >= e.N || ew * 32 >= u.x_rows) return;
        for (int j = lane; j < bn; j += 32) {
            const int64_t m = u.y_row0 + j;
            if (m >= e.M) break;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(base + (m * e.ldc + n0) * es));
        }
    }
}

// The fused steps after x = alpha * acc + beta * c: + bias, then ReLU (keeps
// NaN) or GELU in the exact form x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)).
__device__ __forceinline__ float epi_finish(const EpiParams& e, float x, float bias) {
    if (e.flags & EPI_BIAS) x += bias;
    if (e.flags & EPI_RELU) x = x < 0.0f ? 0.0f : x;
    if (e.flags & EPI_GELU) x = 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
    return x;
}

// Compile-time form of the fused steps: -1 none; 0 + bias, then ReLU if its
// flag is set (a select, not a branch); 2 + bias, GELU (the bias is 0 without
// the bias flag).  Callers pick it once per chunk, so no element carries a
// branch: per-element branches on the flags cost a third of C2's time.
__device__ __forceinline__ int epi_act(const EpiParams& e) {
    return !e.flags ? -1 : ((e.flags & EPI_GELU) ? 2 : 0);
}

template <int ACT>
using EpiAct = std::integral_constant<int, ACT>;

// Run f(EpiAct<act>) for the epilogue's act.
template <typename F>
__device__ __forceinline__ void with_epi_act(const EpiParams& e, F&& f) {
    switch (epi_act(e)) {
        case -1: f(EpiAct<-1>{}); break;
        case 0: f(EpiAct<0>{}); break;
        default: f(EpiAct<2>{}); break;
    }
}

// The epilogue parameters the per-element arithmetic reads, copied into
// registers once per chunk.  Read through the parameter block instead, they
// would be re-read after every store of the chunk: the compiler cannot tell
// that a store to shared or global memory leaves them unchanged, and the
// re-reads made a chunk's conversion several times slower.
struct EpiArith {
    float alpha, beta;
    int32_t relu, has_bias, bias_type;
    const void* bias;
    int64_t N;
};

__device__ __forceinline__ EpiArith epi_arith(const EpiParams& e) {
    EpiArith a;
    a.alpha = e.alpha;
    a.beta = e.beta;
    a.relu = (e.flags & EPI_RELU) != 0;
    a.has_bias = (e.flags & EPI_BIAS) != 0;
    a.bias_type = e.bias_type;
    a.bias = e.bias;
    a.N = e.N;
    return a;
}

__device__ __forceinline__ float bias_at(const EpiArith& a, int64_t n) {
    return (a.has_bias && n < a.N) ? ld_elem(a.bias, a.bias_type, n) : 0.0f;
}

// The value stored: alpha * acc + beta * c, then the fused steps of ACT with
// the column's bias.
template <int ACT>
__device__ __forceinline__ float epi_value(const EpiArith& e, float acc, float c, float bias) {
    float x = e.beta != 0.0f ? fmaf(e.alpha, acc, e.beta * c) : e.alpha * acc;
    if constexpr (ACT >= 0) {
        x += bias;
        if constexpr (ACT == 0) x = (e.relu && x < 0.0f) ? 0.0f : x;
        if constexpr (ACT == 2) x = 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
    }
    return x;
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

// Whether a non-swapped chunk moves through global memory in 8-column
// pieces (16 bytes of a 16-bit C / D per lane) rather than 4-column ones.
__device__ __forceinline__ bool octet_layout(const EpiParams& e) {
    return e.vec_ok && (e.d_type == DT_F16 || e.d_type == DT_BF16);
}

// Row-per-thread layout (non-swapped): iteration `it` of a thread covers tile
// row ew*32 + it*(32/Q) + lane/Q and the 4 columns 4*(lane%Q) .. +3; in the
// octet layout, tile row ew*32 + it*(32/O) + lane/O and the 8 columns
// 8*(lane%O) .. +7 (O = W/8 pieces per row).
template <int W>
__device__ __forceinline__ void load_c_chunk(const EpiParams& e, const Unit& u, int ew, int lane, int col0,
                                             CChunk<W>& cc) {
    if (e.beta == 0.0f) return;
    if (!e.swap && octet_layout(e)) {
        constexpr int O = W / 8, ROWS = 32 / O;
        const int64_t boff = (int64_t)u.batch * e.c_bstride;
#pragma unroll
        for (int it = 0; it < O; ++it) {
            const int rt = ew * 32 + it * ROWS + lane / O;
            const int64_t m = u.x_row0 + rt;
            const int64_t n0 = u.y_row0 + col0 + 8 * (lane % O);
            float c[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            const int64_t ci = boff + m * e.ldc + n0;
            if (rt < u.x_rows && m < e.M && n0 < e.N &&
                elem_in_bounds(e, ci, e.N - n0 < 8 ? e.N - n0 : 8, e.c_extent)) {
                if (n0 + 7 < e.N) {
                    ld8(e.C, e.d_type, ci, c);
                } else {
                    for (int t = 0; t < 8 && n0 + t < e.N; ++t) c[t] = ld_elem(e.C, e.d_type, ci + t);
                }
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) cc.v[8 * it + t] = c[t];
        }
        return;
    }
    constexpr int Q = W / 4;
    const int64_t boff_c = (int64_t)u.batch * e.c_bstride;
    if (e.swap) {
        const int64_t n = u.x_row0 + ew * 32 + lane;
        const bool nok = n < e.N && ew * 32 + lane < u.x_rows;
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const int64_t m = u.y_row0 + col0 + j;
            cc.v[j] = (nok && m < e.M && elem_in_bounds(e, boff_c + m * e.ldc + n, 1, e.c_extent))
                          ? ld_elem(e.C, e.d_type, boff_c + m * e.ldc + n)
                          : 0.0f;
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
        if (rt < u.x_rows && m < e.M && n0 < e.N &&
            elem_in_bounds(e, boff_c + m * e.ldc + n0, e.N - n0 < 4 ? e.N - n0 : 4, e.c_extent)) {
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
template <int W, int ACT, bool Q8>
__device__ __forceinline__ void store_chunk_t(const EpiParams& ep, const Unit& u, int ew, int lane, int col0,
                                            const float (&v)[W], const CChunk<W>& cc, float4* staging) {
    const EpiParams e = ep;  // in registers: the stores below would otherwise force re-reads of every field used
    constexpr int Q = W / 4;
    const int64_t boff_d = (int64_t)u.batch * e.d_bstride;
    const EpiArith ar = epi_arith(e);
    if (e.swap) {
        // tile row -> output column n; tile column -> output row m.
        const int64_t nb = u.x_row0 + ew * 32;  // this warp's 32 output columns
        if (!Q8 && e.d_type != DT_F32 && e.vec_ok && nb + 32 <= e.N && ew * 32 + 32 <= u.x_rows) {
            // 16-bit D, whole warp in range: through the staging buffer, so
            // that every lane stores 16 bytes (a quarter of one output row's
            // 32 columns) instead of one element per chunk column
            constexpr int PITCH = 40;  // halves per staged row: 80 bytes keeps the 16-byte reads spread over the banks
            uint16_t* t16 = reinterpret_cast<uint16_t*>(staging);
            const float bn = ACT >= 0 ? bias_at(ar, nb + lane) : 0.0f;
#pragma unroll
            for (int j = 0; j < W; ++j) {
                const float x = epi_value<ACT>(ar, v[j], cc.v[j], bn);
                t16[j * PITCH + lane] = e.d_type == DT_F16 ? __half_as_ushort(__float2half_rn(x))
                                                           : __bfloat16_as_ushort(__float2bfloat16_rn(x));
            }
            __syncwarp();
#pragma unroll
            for (int it = 0; it < W / 8; ++it) {
                const int j = it * 8 + lane / 4, part = lane % 4;
                const int64_t m = u.y_row0 + col0 + j;
                const int64_t di = boff_d + m * e.ldd + nb + part * 8;
                const uint4 q = *reinterpret_cast<const uint4*>(t16 + j * PITCH + part * 8);
                if (m < e.M && elem_in_bounds(e, di, 8, e.d_extent))
                    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(e.D) + di) = q;
            }
            __syncwarp();
            return;
        }
        // otherwise one element per store; lanes hold consecutive n, so each
        // store instruction is still row-contiguous
        const int64_t n = nb + lane;
        if (n >= e.N || ew * 32 + lane >= u.x_rows) return;
        const float bn = ACT >= 0 ? bias_at(ar, n) : 0.0f;
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const int64_t m = u.y_row0 + col0 + j;
            if (m < e.M) store_out<Q8>(e, boff_d + m * e.ldd + n, epi_value<ACT>(ar, v[j], cc.v[j], bn), m);
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < Q; ++j)
        staging[lane * Q + (j ^ (lane & (Q - 1)))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    if (!Q8 && octet_layout(e)) {
        // 16-bit D: two staged quads per lane, one 16-byte store
        constexpr int O = W / 8, ROWS = 32 / O;
        const int o = lane % O;
#pragma unroll
        for (int it = 0; it < O; ++it) {
            const int rr = it * ROWS + lane / O;
            const float4 a = staging[rr * Q + ((2 * o) ^ (rr & (Q - 1)))];
            const float4 b = staging[rr * Q + ((2 * o + 1) ^ (rr & (Q - 1)))];
            const int rt = ew * 32 + rr;
            const int64_t m = u.x_row0 + rt;
            const int64_t n0 = u.y_row0 + col0 + 8 * o;
            if (rt >= u.x_rows || m >= e.M || n0 >= e.N) continue;
            const float acc[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            float out[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
                out[t] = epi_value<ACT>(ar, acc[t], cc.v[8 * it + t], ACT >= 0 ? bias_at(ar, n0 + t) : 0.0f);
            const int64_t di = boff_d + m * e.ldd + n0;
            if (n0 + 7 < e.N) {
                if (elem_in_bounds(e, di, 8, e.d_extent)) st8(e.D, e.d_type, di, out);
            } else {
                for (int t = 0; t < 8 && n0 + t < e.N; ++t) store_out<false>(e, di + t, out[t], m);
            }
        }
        __syncwarp();
        return;
    }
    constexpr int ROWS_PER_IT = 32 / Q;
    // this lane's quad of columns is the same in every iteration
    float bq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (ACT >= 0) {
        const int64_t nq = u.y_row0 + col0 + 4 * (lane % Q);
#pragma unroll
        for (int t = 0; t < 4; ++t) bq[t] = bias_at(ar, nq + t);
    }
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
        const float4 o = make_float4(epi_value<ACT>(ar, a.x, cc.v[4 * it], bq[0]),
                                     epi_value<ACT>(ar, a.y, cc.v[4 * it + 1], bq[1]),
                                     epi_value<ACT>(ar, a.z, cc.v[4 * it + 2], bq[2]),
                                     epi_value<ACT>(ar, a.w, cc.v[4 * it + 3], bq[3]));
        if (e.vec_ok && n0 + 3 < e.N) {
            store_out4<Q8>(e, di, o, m);
        } else {
            const float ov[4] = {o.x, o.y, o.z, o.w};
            for (int q = 0; q < 4 && n0 + q < e.N; ++q) store_out<Q8>(e, di + q, ov[q], m);
        }
    }
    __syncwarp();
}

template <int W>
__device__ __forceinline__ void store_chunk(const EpiParams& e, const Unit& u, int ew, int lane, int col0,
                                            const float (&v)[W], const CChunk<W>& cc, float4* staging) {
    if (e.d_type == DT_S8)
        with_epi_act(e, [&](auto act) { store_chunk_t<W, decltype(act)::value, true>(e, u, ew, lane, col0, v, cc, staging); });
    else
        with_epi_act(e, [&](auto act) { store_chunk_t<W, decltype(act)::value, false>(e, u, ew, lane, col0, v, cc, staging); });
}

// Partial tile layout in the workspace: for chunk c and quad j, the 128 rows'
// float4 values are contiguous, so a warp's 32 lanes write 512 bytes at once.
template <int BN>
__device__ __forceinline__ float4* partial_quad(float* partials, int64_t slot, int c, int j, int r) {
    constexpr int Q = Chunk<BN>::Q;
    return reinterpret_cast<float4*>(partials + slot * (int64_t)(BM * BN)) + ((int64_t)(c * Q + j) * BM + r);
}

// Shared memory the last arriver of a split tile may use to reduce the
// partials of its CTA's final unit: the pipeline ring, idle once the final
// unit's accumulator is complete.  base == nullptr: not available.
struct FixupSmem {
    uint8_t* base;
    uint32_t bytes;
    uint64_t* bar;  // FIX_BARS completion barriers of the bulk copies (used on the final unit only)
};

// The CTA pair splits every tile into two 128-row halves, one per CTA, each
// with its own partial slots and arrival counter.
__device__ __forceinline__ int64_t half_slot(const GemmKernelParams& P, int64_t slot) {
    return P.pair ? 2 * slot + (blockIdx.x & 1) : slot;
}
__device__ __forceinline__ int32_t* tile_counter(const GemmKernelParams& P, int64_t tile) {
    return &P.counters[P.pair ? 2 * tile + (blockIdx.x & 1) : tile];
}

// The checked build's unit check: tile coordinates inside the tile grid (or,
// grouped, the expert and its token rows inside the problem), a K range inside
// the K-steps, and for a split tile every contributor's partial slot and the
// tile's counter inside the workspace.
static __device__ __noinline__ bool unit_in_bounds(const GemmKernelParams& P, const Unit& u, int bn) {
    const SchedParams& s = P.sched;
    const int64_t rows_x = (int64_t)s.tiles_x * BM * (P.pair ? 2 : 1), rows_y = (int64_t)s.tiles_y * bn;
    bool ok = u.k_begin >= 0 && u.k_begin < u.k_end && u.k_end <= s.k_iters && u.tile >= 0 && u.tile < total_tiles(s) &&
              u.y_row0 >= 0 && u.y_row0 < rows_y && u.x_rows >= 0 && u.x_rows <= BM;
    if (s.grouped)  // a CTA-pair half with no rows of its expert stores nothing (its copies read zeros)
        ok = ok && u.batch >= 0 && u.batch < s.num_experts && u.x_row0 >= 0 &&
             (u.x_rows == 0 || u.x_row0 + u.x_rows <= (int64_t)s.expert_offsets[s.num_experts]);
    else
        ok = ok && u.batch >= 0 && u.batch < s.batches && u.x_row0 >= 0 && u.x_row0 < rows_x;
    if (!ok) {
        record_check(P.status, CHECK_UNIT);
        return false;
    }
    if (u.mode == UNIT_PARTIAL) {
        // both halves of a CTA pair are checked, so the two CTAs always agree
        const uint64_t slot_bytes = (uint64_t)BM * bn * 4;
        const int64_t halves = P.pair ? 2 : 1;
        for (int q = 0; q <= u.ncontrib; ++q) {
            const int64_t sl = q < u.ncontrib ? partial_slot(s, u.tile, q) : u.slot;
            if (sl < 0 || (uint64_t)(halves * sl + halves) * slot_bytes > P.partials_bytes) {
                record_check(P.status, CHECK_PARTIAL);
                return false;
            }
        }
        if ((uint64_t)(halves * u.tile + halves) * 4 > P.counters_bytes) {
            record_check(P.status, CHECK_COUNTER);
            return false;
        }
    }
    return true;
}

// Whether unit `u` (just returned by the iterator `w`) is this program's last.
__device__ __forceinline__ bool final_unit(const GemmKernelParams& P, WorkIter w, int bn) {
    Unit u2;
    return !next_unit(P, w, u2, bn);
}

// Arrival of a split tile's contributor, after its partial tile is written:
// one CTA barrier orders every epilogue thread's partial stores before the
// lead thread's release fence and counter increment (the fence is cumulative),
// so one thread pays the write-acknowledgement latency instead of each.  The
// last arriver resets the counter and acquires the others' partials.  Returns
// whether this unit's CTA is the tile's last arriver (every epilogue thread).
__device__ __forceinline__ bool split_arrive(const GemmKernelParams& P, const Unit& u, volatile uint32_t* bcast,
                                             int lead) {
    epi_bar_sync();
    if ((int)threadIdx.x == lead) {
        __threadfence();
        const int old = atomicAdd(tile_counter(P, u.tile), 1);
        const bool last = (old == u.ncontrib - 1);
        if (last) {
            atomicExch(tile_counter(P, u.tile), 0);  // every contributor has arrived
            __threadfence();
        }
        *bcast = last ? 1u : 0u;
    }
    epi_bar_sync();
    return *bcast != 0u;
}

// Chunks of a split tile's partials that the idle ring can hold at once for
// all contributors (0: the bulk path does not fit).
template <int BN>
__device__ __forceinline__ int fixup_buffers(const FixupSmem& fx, const Unit& u) {
    constexpr uint32_t CHUNK = BM * Chunk<BN>::W * 4;
    if (fx.base == nullptr) return 0;
    const uint32_t n = fx.bytes / ((uint32_t)u.ncontrib * CHUNK);
    return (int)(n < (uint32_t)FIX_BARS ? (n < (uint32_t)Chunk<BN>::N ? n : Chunk<BN>::N)
                                        : ((uint32_t)FIX_BARS < (uint32_t)Chunk<BN>::N ? FIX_BARS : Chunk<BN>::N));
}

// The last arriver's reduction on its final unit: column chunk c of every
// contributor's partial tile (BM x W fp32, contiguous in a slot) is copied
// into the idle ring with bulk copies, nbuf chunks in flight at once, each
// chunk completing on its own barrier; the epilogue sums a chunk over the
// contributors in K order (fixup_reduce) while the next chunks land.
// fixup_issue(c): the lead thread starts chunk c's copies.
template <int BN>
__device__ __forceinline__ void fixup_issue(const GemmKernelParams& P, const Unit& u, const FixupSmem& fx, int lead,
                                            int nbuf, int c) {
    using CK = Chunk<BN>;
    constexpr uint32_t CHUNK = BM * CK::W * 4;
    if ((int)threadIdx.x != lead || c >= CK::N) return;
    const uint32_t per = (uint32_t)u.ncontrib * CHUNK;
    if (c == 0) fence_proxy_async_global();  // the contributors' partial stores -> bulk reads
    uint64_t* bar = &fx.bar[c % nbuf];
    mbar_arrive_expect_tx(bar, per);
    for (int q = 0; q < u.ncontrib; ++q)
        bulk_load_g2s(fx.base + (size_t)(c % nbuf) * per + (size_t)q * CHUNK,
                      P.partials + half_slot(P, partial_slot(P.sched, u.tile, q)) * (int64_t)(BM * BN) +
                          (int64_t)c * (BM * CK::W),
                      CHUNK, bar);
}

// Sum chunk c of every contributor into v (zeroed by the caller), in K order,
// once its copies have landed; then, after every epilogue thread is done with
// the buffer, start chunk c + nbuf in it.  Returns false if the wait gave up.
template <int BN>
__device__ __forceinline__ bool fixup_reduce(const GemmKernelParams& P, const Unit& u, const FixupSmem& fx,
                                             const Guard& g, int lead, int nbuf, int c, float (&v)[Chunk<BN>::W]) {
    using CK = Chunk<BN>;
    constexpr uint32_t CHUNK = BM * CK::W * 4;
    if (!__all_sync(0xffffffffu, wait_bar(&fx.bar[c % nbuf], (uint32_t)(c / nbuf) & 1u, g, SITE_EPI_TMEM_FULL)))
        return false;
    const int r = (int)(threadIdx.x % 128);
    const float4* src = reinterpret_cast<const float4*>(fx.base + (size_t)(c % nbuf) * u.ncontrib * CHUNK);
#pragma unroll 1
    for (int q = 0; q < u.ncontrib; ++q) {
#pragma unroll
        for (int j = 0; j < CK::Q; ++j) {
            const float4 p = src[(size_t)q * (CK::Q * BM) + j * BM + r];
            v[4 * j] += p.x;
            v[4 * j + 1] += p.y;
            v[4 * j + 2] += p.z;
            v[4 * j + 3] += p.w;
        }
    }
    epi_bar_sync();  // every thread is done with this buffer before it is refilled
    fixup_issue<BN>(P, u, fx, lead, nbuf, c + nbuf);
    return true;
}

// The epilogue role: 4 warps (128 threads, the first of them `lead`), warp w
// reads TMEM lanes 32*(w%4) .. 32*(w%4)+31.  For every unit: wait for the
// accumulator, then either store it (whole tile) or write it as a partial
// and, if this unit is the last of its tile to arrive, reduce all partials in
// K order and store.
template <int BN>
__device__ void epilogue_role(const GemmKernelParams& P, uint32_t tmem_base, uint64_t* tfull, uint64_t* tempty,
                              float* staging_all, volatile uint32_t* bcast, const FixupSmem& fx, const Guard& g,
                              int lead) {
    using CK = Chunk<BN>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ew = warp % 4;
    const int r = ew * 32 + lane;
    float4* staging = reinterpret_cast<float4*>(staging_all) + ew * 32 * CK::Q;
    WorkIter w;
    w.init(P.sched, unit_pid(P));
    Unit u;
    uint32_t acc_it = 0;
    while (next_unit(P, w, u, BN)) {
        if (P.epi.flags) {
            if (P.epi.swap)
                prefetch_bias(P.epi, u.x_row0 + ew * 32, 32, lane);
            else
                prefetch_bias(P.epi, u.y_row0, BN, lane);
        }
        if (u.mode == UNIT_FULL) prefetch_c_l2(P.epi, u, ew, lane, BN);
        const int buf = acc_it & 1;
        const uint32_t aph = (acc_it >> 1) & 1;
        ++acc_it;
        if (!wait_bar(&tfull[buf], aph, g, SITE_EPI_TMEM_FULL)) break;
        tc_fence_after_sync();
        const uint32_t tbase = tmem_base + (uint32_t)(buf * BN) + ((uint32_t)(ew * 32) << 16);
        if (u.mode == UNIT_FULL) {
            // C of a chunk is requested before its TMEM load so the two overlap
#pragma unroll 1
            for (int c = 0; c < CK::N; ++c) {
                CChunk<CK::W> cc;
                load_c_chunk<CK::W>(P.epi, u, ew, lane, c * CK::W, cc);
                float v[CK::W];
                tmem_load_chunk<CK::W>(tbase + c * CK::W, v);
                if (c == CK::N - 1) {
                    tc_fence_before_sync();
                    mbar_arrive(&tempty[buf]);
                }
                store_chunk<CK::W>(P.epi, u, ew, lane, c * CK::W, v, cc, staging);
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
                *partial_quad<BN>(P.partials, half_slot(P, u.slot), c, j, r) =
                    make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        tc_fence_before_sync();
        mbar_arrive(&tempty[buf]);
        if (!split_arrive(P, u, bcast, lead)) continue;
        // on the final unit the idle ring takes the contributors' partials, chunk by chunk
        const int nbuf = final_unit(P, w, BN) ? fixup_buffers<BN>(fx, u) : 0;
        for (int c = 0; c < nbuf; ++c) fixup_issue<BN>(P, u, fx, lead, nbuf, c);
        bool fix_ok = true;
#pragma unroll 1
        for (int c = 0; c < CK::N; ++c) {
            CChunk<CK::W> cc;
            load_c_chunk<CK::W>(P.epi, u, ew, lane, c * CK::W, cc);
            float v[CK::W];
#pragma unroll
            for (int i = 0; i < CK::W; ++i) v[i] = 0.0f;
            if (nbuf > 0) {
                if (!fixup_reduce<BN>(P, u, fx, g, lead, nbuf, c, v)) {
                    fix_ok = false;
                    break;
                }
                store_chunk<CK::W>(P.epi, u, ew, lane, c * CK::W, v, cc, staging);
                continue;
            }
            // contributors in K order, two at a time so their loads overlap
#pragma unroll 1
            for (int q0 = 0; q0 < u.ncontrib; q0 += 2) {
                const bool two = q0 + 1 < u.ncontrib;
                const int64_t s0 = half_slot(P, partial_slot(P.sched, u.tile, q0));
                const int64_t s1 = two ? half_slot(P, partial_slot(P.sched, u.tile, q0 + 1)) : s0;
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
        if (!fix_ok) break;
    }
}

// Position in the per-warp stream of (unit, chunk) pairs, used to fetch C
// ahead of the chunk being stored, across unit boundaries.
struct ChunkStream {
    WorkIter w;
    Unit u;
    int c;
    bool valid;
    __device__ __forceinline__ void init(const GemmKernelParams& P, int bn) {
        w.init(P.sched, unit_pid(P));
        c = 0;
        valid = next_unit(P, w, u, bn);
    }
    __device__ __forceinline__ void advance(const GemmKernelParams& P, int bn, int nch) {
        if (++c == nch) {
            c = 0;
            valid = next_unit(P, w, u, bn);
        }
    }
};

// TMA epilogue (non-swapped, non-grouped, 16-byte aligned C and D): every
// epilogue warp owns `ncb` shared-memory buffers holding a 32-row x 32-column
// slab of C / D in the TMA swizzled layout (64-byte rows for 16-bit types,
// SWIZZLE_64B; 128-byte rows for fp32, SWIZZLE_128B).  C slabs are loaded
// ncb-1 chunks ahead of use -- across unit boundaries, so they arrive while
// the tensor core still works on the tile -- and each finished D slab is
// written back in place and stored with one TMA store.
template <int BN>
__device__ void epilogue_tma(const GemmKernelParams& P, const CUtensorMap* tmC, const CUtensorMap* tmD,
                             uint32_t tmem_base, uint64_t* tfull, uint64_t* tempty, uint8_t* ebuf_all,
                             uint64_t* cbar_all, volatile uint32_t* bcast, const FixupSmem& fx, const Guard& g,
                             int lead) {
    constexpr int W = 32;
    constexpr int NCH = BN / W;
    const EpiParams& e = P.epi;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ew = warp % 4;
    const int r = ew * 32 + lane;
    const bool f32 = e.d_type == DT_F32;
    const bool bf16 = e.d_type == DT_BF16;
    const uint32_t buf_bytes = 32u * W * (f32 ? 4u : 2u);
    const int ncb = e.ncb;
    uint8_t* ebuf = ebuf_all + (size_t)ew * ncb * buf_bytes;
    uint64_t* cbar = cbar_all + ew * 4;
    const bool use_c = e.beta != 0.0f;

    auto slab_x = [&](const Unit& u, int c) { return (int32_t)(u.y_row0 + c * W); };
    auto slab_y = [&](const Unit& u) { return (int32_t)(u.x_row0 + ew * 32); };

    // Store bookkeeping (all lanes; lane 0 issues): stores are numbered as they are committed;
    // a buffer may be rewritten once every store up to its last one has read
    // its source, i.e. once at most nstores - last_store[b] are still reading.
    uint32_t nstores = 0;
    uint32_t last_store[4] = {0, 0, 0, 0};
    auto wait_buffer_read = [&](int b) {
        const uint32_t newer = nstores - last_store[b];
        if (newer == 0)
            bulk_wait_group_read<0>();
        else if (newer == 1)
            bulk_wait_group_read<1>();
        else if (newer == 2)
            bulk_wait_group_read<2>();
        else if (newer == 3)
            bulk_wait_group_read<3>();
        else  // four or more newer stores: waiting for all but the newest four suffices
            bulk_wait_group_read<4>();
    };

    ChunkStream pre;
    pre.init(P, BN);
    uint32_t ppos = 0, gpos = 0;
    auto issue_c = [&]() {
        const int b = ppos % ncb;
        if (lane == 0) {
            mbar_arrive_expect_tx(&cbar[b], buf_bytes);
            if (P.x3d)
                tma_load_3d(ebuf + b * buf_bytes, tmC, &cbar[b], slab_x(pre.u, pre.c), slab_y(pre.u), pre.u.batch);
            else
                tma_load_2d(ebuf + b * buf_bytes, tmC, &cbar[b], slab_x(pre.u, pre.c), slab_y(pre.u));
        }
        pre.advance(P, BN, NCH);
        ++ppos;
    };
    if (use_c)
        for (int i = 0; i < ncb - 1 && pre.valid; ++i) issue_c();

    // Combine chunk `c` of unit `u` (values v) with C and store it; when
    // `store` is false the chunk's C slab is only consumed.
    bool ok = true;
    auto finish_chunk = [&](const Unit& u, int c, const float(&v)[W], bool store) {
        const int b = gpos % ncb;
        uint8_t* buf = ebuf + b * buf_bytes;
        if (use_c) {
            if (!wait_bar(&cbar[b], (gpos / ncb) & 1u, g, SITE_EPI_TMEM_FULL)) {
                ok = false;
                return;
            }
        } else if (store && last_store[b] != 0) {
            // the buffer's previous store must have read it; a buffer never
            // stored from, or not written now, needs no wait (the bulk-group
            // wait costs about a microsecond even with nothing pending)
            if (lane == 0) wait_buffer_read(b);
            __syncwarp();
        }
        if (store) {
            const EpiArith ar = epi_arith(e);
            if (f32) {
                uint8_t* row = buf + lane * 128;
                const int64_t n0 = slab_x(u, c);
                auto put = [&](auto act) {
                    constexpr int F = decltype(act)::value;
                    // lane l holds the bias of the chunk's column l (W = 32 columns)
                    const float bl = F >= 0 ? bias_at(ar, n0 + lane) : 0.0f;
                    auto bcol = [&](int col) { return F >= 0 ? __shfl_sync(0xffffffffu, bl, col) : 0.0f; };
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float4* pp = reinterpret_cast<float4*>(row + ((q ^ (lane & 7)) << 4));
                        const float4 cv = use_c ? *pp : make_float4(0.f, 0.f, 0.f, 0.f);
                        *pp = make_float4(epi_value<F>(ar, v[4 * q], cv.x, bcol(4 * q)),
                                          epi_value<F>(ar, v[4 * q + 1], cv.y, bcol(4 * q + 1)),
                                          epi_value<F>(ar, v[4 * q + 2], cv.z, bcol(4 * q + 2)),
                                          epi_value<F>(ar, v[4 * q + 3], cv.w, bcol(4 * q + 3)));
                    }
                };
                with_epi_act(e, put);
            } else {
                uint8_t* row = buf + lane * 64;
                const int64_t n0 = slab_x(u, c);
                auto put = [&](auto act) {
                    constexpr int F = decltype(act)::value;
                    const float bl = F >= 0 ? bias_at(ar, n0 + lane) : 0.0f;
                    auto bcol = [&](int col) { return F >= 0 ? __shfl_sync(0xffffffffu, bl, col) : 0.0f; };
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4* pp = reinterpret_cast<uint4*>(row + ((q ^ ((lane >> 1) & 3)) << 4));
                        float cv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        if (use_c) {
                            const uint4 in = *pp;
                            const uint32_t iw[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const float2 f = bf16 ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&iw[t]))
                                                      : __half22float2(*reinterpret_cast<const __half2*>(&iw[t]));
                                cv[2 * t] = f.x;
                                cv[2 * t + 1] = f.y;
                            }
                        }
                        uint32_t ow[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float a = epi_value<F>(ar, v[8 * q + 2 * t], cv[2 * t], bcol(8 * q + 2 * t));
                            const float b2 = epi_value<F>(ar, v[8 * q + 2 * t + 1], cv[2 * t + 1], bcol(8 * q + 2 * t + 1));
                            if (bf16) {
                                __nv_bfloat162 h = __floats2bfloat162_rn(a, b2);
                                ow[t] = *reinterpret_cast<uint32_t*>(&h);
                            } else {
                                __half2 h = __floats2half2_rn(a, b2);
                                ow[t] = *reinterpret_cast<uint32_t*>(&h);
                            }
                        }
                        *pp = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                };
                with_epi_act(e, put);
            }
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (store) {
            if (lane == 0) {
                if (P.x3d)
                    tma_store_3d(tmD, buf, slab_x(u, c), slab_y(u), u.batch);
                else
                    tma_store_2d(tmD, buf, slab_x(u, c), slab_y(u));
                bulk_commit_group();
            }
            // every lane keeps the count, so the waits below are taken (or
            // skipped) by the whole warp
            last_store[b] = ++nstores;
        }
        ++gpos;
        if (use_c && pre.valid) {
            if (last_store[ppos % ncb] != 0) {
                if (lane == 0) wait_buffer_read(ppos % ncb);  // the next slab's buffer is free
                __syncwarp();
            }
            issue_c();
        }
    };

    WorkIter w;
    w.init(P.sched, unit_pid(P));
    Unit u;
    uint32_t acc_it = 0;
    while (ok && next_unit(P, w, u, BN)) {
        if (e.flags) prefetch_bias(e, u.y_row0, BN, lane);
        // this warp's C slabs of the unit into L2 while its accumulator is
        // computed: the slab copies issued during the epilogue then find them
        // there instead of each waiting on HBM
        if (use_c && lane < NCH) {
            if (P.x3d)
                tma_prefetch_l2_3d(tmC, slab_x(u, lane), slab_y(u), u.batch);
            else
                tma_prefetch_l2_2d(tmC, slab_x(u, lane), slab_y(u));
        }
        const int buf = acc_it & 1;
        const uint32_t aph = (acc_it >> 1) & 1;
        ++acc_it;
        if (!wait_bar(&tfull[buf], aph, g, SITE_EPI_TMEM_FULL)) break;
        tc_fence_after_sync();
        const uint32_t tbase = tmem_base + (uint32_t)(buf * BN) + ((uint32_t)(ew * 32) << 16);
        if (u.mode == UNIT_FULL) {
#pragma unroll 1
            for (int c = 0; c < NCH && ok; ++c) {
                float v[W];
                tmem_load_chunk<W>(tbase + c * W, v);
                if (c == NCH - 1) {
                    tc_fence_before_sync();
                    mbar_arrive(&tempty[buf]);
                }
                finish_chunk(u, c, v, true);
            }
            continue;
        }
#pragma unroll 1
        for (int c = 0; c < NCH; ++c) {
            float v[W];
            tmem_load_chunk<W>(tbase + c * W, v);
#pragma unroll
            for (int j = 0; j < W / 4; ++j)
                *partial_quad<BN>(P.partials, half_slot(P, u.slot), c, j, r) =
                    make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        tc_fence_before_sync();
        mbar_arrive(&tempty[buf]);
        const bool last = split_arrive(P, u, bcast, lead);
        // on the final unit the idle ring takes the contributors' partials, chunk by chunk
        const int nbuf = last && final_unit(P, w, BN) ? fixup_buffers<BN>(fx, u) : 0;
        for (int c = 0; c < nbuf; ++c) fixup_issue<BN>(P, u, fx, lead, nbuf, c);
#pragma unroll 1
        for (int c = 0; c < NCH && ok; ++c) {
            float v[W];
#pragma unroll
            for (int i = 0; i < W; ++i) v[i] = 0.0f;
            if (nbuf > 0) {
                if (!fixup_reduce<BN>(P, u, fx, g, lead, nbuf, c, v)) {
                    ok = false;
                    break;
                }
            } else if (last) {
#pragma unroll 1
                for (int q0 = 0; q0 < u.ncontrib; q0 += 2) {
                    const bool two = q0 + 1 < u.ncontrib;
                    const int64_t s0 = half_slot(P, partial_slot(P.sched, u.tile, q0));
                    const int64_t s1 = two ? half_slot(P, partial_slot(P.sched, u.tile, q0 + 1)) : s0;
                    float4 p0[W / 4], p1[W / 4];
#pragma unroll
                    for (int j = 0; j < W / 4; ++j) {
                        p0[j] = __ldcg(partial_quad<BN>(P.partials, s0, c, j, r));
                        p1[j] = __ldcg(partial_quad<BN>(P.partials, s1, c, j, r));
                    }
#pragma unroll
                    for (int j = 0; j < W / 4; ++j) {
                        v[4 * j] += p0[j].x;
                        v[4 * j + 1] += p0[j].y;
                        v[4 * j + 2] += p0[j].z;
                        v[4 * j + 3] += p0[j].w;
                    }
                    if (two) {
#pragma unroll
                        for (int j = 0; j < W / 4; ++j) {
                            v[4 * j] += p1[j].x;
                            v[4 * j + 1] += p1[j].y;
                            v[4 * j + 2] += p1[j].z;
                            v[4 * j + 3] += p1[j].w;
                        }
                    }
                }
            }
            finish_chunk(u, c, v, last);
        }
    }
    // drain: C slabs still in flight, then every store
    if (lane == 0) {
        for (uint32_t p = gpos; p < ppos; ++p) wait_bar_drain(&cbar[p % ncb], (p / ncb) & 1u, g);
        bulk_wait_group_all();
    }
    __syncwarp();
}

// The epilogue of a kernel whose epilogue warps are the four starting at
// thread `lead` (a multiple of 128 plus, in the two-role kernels, 64).
template <int BN>
__device__ __forceinline__ void epilogue(const GemmKernelParams& P, const CUtensorMap* tmC, const CUtensorMap* tmD,
                                         uint32_t tmem_base, uint64_t* tfull, uint64_t* tempty, uint8_t* esmem,
                                         uint64_t* cbar, volatile uint32_t* bcast, const FixupSmem& fx,
                                         const Guard& g, int lead) {
    if constexpr (BN >= 32) {
        if (P.epi.tma) {
            epilogue_tma<BN>(P, tmC, tmD, tmem_base, tfull, tempty, esmem, cbar, bcast, fx, g, lead);
            return;
        }
    }
    epilogue_role<BN>(P, tmem_base, tfull, tempty, reinterpret_cast<float*>(esmem), bcast, fx, g, lead);
}

}  // namespace qg
