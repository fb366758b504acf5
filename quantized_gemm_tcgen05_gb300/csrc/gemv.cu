// Small-M streaming kernel (see gemv.h).
//
// Work split: a warp owns a group of R = 4 rows of B (4 output columns n) and
// one of `kslices` contiguous slices of their K range; its lanes stride the
// slice in 16-byte chunks, so every load instruction of a warp reads 512
// contiguous bytes of a row.  A CTA of 8 warps covers 8 / kslices row
// groups; the per-warp partial sums meet in shared memory and are added in
// slice order, so results are bitwise run-to-run deterministic.  The grid is
// at most one wave of resident CTAs and walks the row groups with a stride.
//
// Per element: b^ = b (16-bit B, no scale), RN_A(b * v) (16-bit B with V) or
// RN_A((q - z) * v) (int4 B, z = 0 without zero points; unscaled: q), each
// product exact in fp32 and rounded once to A's type; then acc += a * b^ in
// fp32 (exact product, fp32 sum).
#include <atomic>

#include "gemv.h"
#include "umma_dq_gemm.cuh"

namespace qg {

namespace {

constexpr int GEMV_R = 4;        // rows of B per warp
constexpr int GEMV_WARPS = 8;    // warps per CTA

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Eight 16-bit values (one 16-byte chunk) as fp32.
template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        if constexpr (BF16) {
            f[2 * t] = lo_bf16(w[t]);
            f[2 * t + 1] = hi_bf16(w[t]);
        } else {
            const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&w[t]));
            f[2 * t] = h.x;
            f[2 * t + 1] = h.y;
        }
    }
}

// RN to A's type of two exact fp32 values, back as fp32.
template <bool BF16>
__device__ __forceinline__ void round2(float& a, float& b) {
    if constexpr (BF16) {
        const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
        const uint32_t u = *reinterpret_cast<const uint32_t*>(&r);
        a = lo_bf16(u);
        b = hi_bf16(u);
    } else {
        const float2 r = __half22float2(__floats2half2_rn(a, b));
        a = r.x;
        b = r.y;
    }
}

// Group of the 8-value block i8 along K: i8 / (gb / 8), by a multiply exact
// for i8 < 2^24.
__device__ __forceinline__ int64_t group_of(uint64_t gmagic, int64_t i8) {
    return (int64_t)(((uint64_t)i8 * gmagic) >> 40);
}

__device__ __forceinline__ float scale_at(const GemvParams& p, uint64_t gmagic, int64_t n, int64_t i8) {
    const uint16_t bits = reinterpret_cast<const uint16_t*>(p.V)[group_of(gmagic, i8) * p.ldv + n];
    return p.v_bf16 ? __uint_as_float((uint32_t)bits << 16) : __half2float(__ushort_as_half(bits));
}

// Zero point of column n for block i8: the low nibble of its byte, two's
// complement; 0 without zero points.
__device__ __forceinline__ int zero_at(const GemvParams& p, uint64_t gmagic, int64_t n, int64_t i8) {
    if (!p.Z) return 0;
    const uint8_t b = reinterpret_cast<const uint8_t*>(p.Z)[group_of(gmagic, i8) * p.ldz + n];
    return (int)((uint32_t)b << 28) >> 28;
}

// A group scale and zero point prepared for dequant8: for bf16 results the
// split pair (vhi2, vlo2) and the offset pair of the packed path, else the
// fp32 value and the magic-number bias 2^23 + 8 + z.
struct Scale {
    uint32_t vhi2, vlo2, off2;
    float v, zoff;
};

template <bool BF16>
__device__ __forceinline__ Scale prep_scale(float v, bool scaled, int z = 0) {
    Scale s{0x3F803F80u, 0u, int4_off2(z), scaled ? v : 1.0f, 8388616.0f + (float)z};  // unscaled: v = 1
    if (BF16 && scaled) split_scale_bf16(v, s.vhi2, s.vlo2);
    return s;
}

// Eight int4 values (one 32-bit word: k = 2t in bits 4t..4t+3 of byte t, odd k
// in the high nibble) times their scale, each rounded once to A's type.
template <bool BF16>
__device__ __forceinline__ void dequant8(uint32_t w, const Scale& sc, float* f) {
    if constexpr (BF16) {
        const uint32_t vhi2 = sc.vhi2, vlo2 = sc.vlo2;
        const uint32_t w4 = w >> 4;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t pr = int4_pair_bf16(__byte_perm(w, w4, (uint32_t)t * 0x11u | (uint32_t)(4 + t) * 0x1100u),
                                               vhi2, vlo2, sc.off2);
            f[2 * t] = lo_bf16(pr);
            f[2 * t + 1] = hi_bf16(pr);
        }
    } else {
        // biased nibble u = q + 8 becomes the float 2^23 + u, so
        // q - z = f - (2^23 + 8 + z), exactly
        const uint32_t x = w ^ 0x88888888u;
        const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
        const float s = sc.v, zo = sc.zoff;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            f[2 * t] = (__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7650u | t)) - zo) * s;
            f[2 * t + 1] = (__uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7650u | t)) - zo) * s;
            round2<false>(f[2 * t], f[2 * t + 1]);
        }
    }
}

// M = 1 runs four CTAs per SM (at most 64 registers, one chunk per row in
// flight); larger M two.  Measured on GB300, bf16 N 4096 K 14336 at M = 1:
// 20.7 us with four (all row blocks in one round), 22.1 us with two.
template <int MT, int U, bool BF16, bool INT4>
__global__ void __launch_bounds__(GEMV_WARPS * 32, MT == 1 ? 4 : 2) gemv_kernel(const GemvParams p, uint64_t gmagic) {
    constexpr int R = GEMV_R;
    __shared__ float red[GEMV_WARPS][MT][R];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.kslices;
    const int groups_per_cta = GEMV_WARPS / S;
    const int gi = warp / S, s = warp % S;
    const int M = (int)p.M;
    const int64_t nchunk = INT4 ? p.K / 32 : p.K / 8;
    const int64_t cps = (nchunk + S - 1) / S;
    const int64_t cbeg = s * cps;
    const int64_t cend = cbeg + cps < nchunk ? cbeg + cps : nchunk;
    const int64_t row_bytes = INT4 ? p.ldb / 2 : p.ldb * 2;
    const int64_t ngroups = (p.N + R - 1) / R;
    // every CTA of the grid is resident (one wave), so the next kernel may
    // start its set-up now; it waits for this grid before touching memory
    griddep_launch_dependents();
    // meanwhile warm L2 with this warp's first weight chunks (a hint only: L2
    // is where memory is coherent, so a write by the previous kernel still
    // reaches the loads below)
    {
        const int64_t grp = (int64_t)blockIdx.x * groups_per_cta + gi;
        if (grp < ngroups) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = grp * R + r < p.N ? grp * R + r : p.N - 1;
                const uint8_t* base = reinterpret_cast<const uint8_t*>(p.B) + row * row_bytes;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t c = cbeg + lane + 32 * u;
                    if (c < cend) asm volatile("prefetch.global.L2 [%0];" ::"l"(base + c * 16));
                }
            }
        }
    }
    griddep_wait();
    const uint16_t* A = reinterpret_cast<const uint16_t*>(p.A);
    const bool scaled = p.V != nullptr;

    for (int64_t gbase = (int64_t)blockIdx.x * groups_per_cta; gbase < ngroups;
         gbase += (int64_t)gridDim.x * groups_per_cta) {
        const int64_t grp = gbase + gi;
        float acc[MT][R];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) acc[m][r] = 0.0f;
        if (grp < ngroups) {
            const uint4* brow[R];
            int64_t nr[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                // rows past N re-read the last row; their sums are never stored
                nr[r] = grp * R + r < p.N ? grp * R + r : p.N - 1;
                brow[r] = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.B) + nr[r] * row_bytes);
            }
            for (int64_t c = cbeg + lane; c < cend; c += 32 * U) {
                uint4 bv[U][R];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        if (c + 32 * u < cend) bv[u][r] = __ldcs(brow[r] + c + 32 * u);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t cu = c + 32 * u;
                    if (cu >= cend) break;
                    constexpr int WORDS = INT4 ? 4 : 1;  // 8-value blocks per chunk
                    // int4 groups of 32 or more: one scale per row for the whole chunk
                    Scale vc[R];
                    if (INT4 && scaled && p.gb >= 32) {
#pragma unroll
                        for (int r = 0; r < R; ++r)
                            vc[r] = prep_scale<BF16>(scale_at(p, gmagic, nr[r], cu * 4), true,
                                                     zero_at(p, gmagic, nr[r], cu * 4));
                    }
#pragma unroll
                    for (int j = 0; j < WORDS; ++j) {
                        const int64_t i8 = INT4 ? cu * 4 + j : cu;  // 8-value block index along K
                        float b[R][8];
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            if constexpr (INT4) {
                                const Scale sc =
                                    !scaled ? prep_scale<BF16>(1.0f, false)
                                            : (p.gb >= 32 ? vc[r]
                                                          : prep_scale<BF16>(scale_at(p, gmagic, nr[r], i8), true,
                                                                             zero_at(p, gmagic, nr[r], i8)));
                                const uint32_t w = j == 0 ? bv[u][r].x : (j == 1 ? bv[u][r].y : (j == 2 ? bv[u][r].z : bv[u][r].w));
                                dequant8<BF16>(w, sc, b[r]);
                            } else {
                                const float v = scaled ? scale_at(p, gmagic, nr[r], i8) : 1.0f;
                                unpack8<BF16>(bv[u][r], b[r]);
                                if (scaled) {
#pragma unroll
                                    for (int t = 0; t < 8; t += 2) {
                                        b[r][t] *= v;
                                        b[r][t + 1] *= v;
                                        round2<BF16>(b[r][t], b[r][t + 1]);
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            if (m >= M) break;
                            float a[8];
                            unpack8<BF16>(__ldg(reinterpret_cast<const uint4*>(A + m * p.lda) + i8), a);
#pragma unroll
                            for (int r = 0; r < R; ++r)
#pragma unroll
                                for (int t = 0; t < 8; ++t) acc[m][r] = fmaf(a[t], b[r][t], acc[m][r]);
                        }
                    }
                }
            }
        }
        // lane sums in a fixed butterfly order, then the slices in order
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float v = acc[m][r];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0) red[warp][m][r] = v;
            }
        __syncthreads();
        const int t = threadIdx.x;
        if (t < groups_per_cta * MT * R) {
            const int g2 = t / (MT * R), m = (t / R) % MT, r = t % R;
            const int64_t n = (gbase + g2) * R + r;
            if (m < M && n < p.N) {
                float sum = 0.0f;
                for (int k = 0; k < S; ++k) sum += red[g2 * S + k][m][r];
                float cv = 0.0f;
                if (p.beta != 0.0f) {
                    const int64_t ci = (int64_t)m * p.ldc + n;
                    cv = p.d_type == DT_F32 ? reinterpret_cast<const float*>(p.C)[ci]
                                            : (p.d_type == DT_BF16
                                                   ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.C)[ci])
                                                   : __half2float(reinterpret_cast<const __half*>(p.C)[ci]));
                }
                float d = fmaf(p.alpha, sum, p.beta * cv);
                if (p.epi_flags) {
                    // the fused steps of the tensor-core epilogue, same order
                    if (p.epi_flags & EPI_BIAS) d += ld_elem(p.bias, p.bias_type, n);
                    if (p.epi_flags & EPI_RELU) d = d < 0.0f ? 0.0f : d;
                    if (p.epi_flags & EPI_GELU) d = 0.5f * d * (1.0f + erff(d * 0.70710678118654752f));
                }
                const int64_t di = (int64_t)m * p.ldd + n;
                if (p.d_type == DT_S8)
                    reinterpret_cast<int8_t*>(p.D)[di] = (int8_t)quant_s8(d, p.qscale[m], p.qzp);
                else if (p.d_type == DT_F32)
                    reinterpret_cast<float*>(p.D)[di] = d;
                else if (p.d_type == DT_BF16)
                    reinterpret_cast<__nv_bfloat16*>(p.D)[di] = __float2bfloat16_rn(d);
                else
                    reinterpret_cast<__half*>(p.D)[di] = __float2half_rn(d);
            }
        }
        __syncthreads();  // red[] is reused by the next row block
    }
}

template <int MT, int U, bool BF16, bool INT4>
cudaError_t launch_t(const GemvParams& p, int sm_count, cudaStream_t st) {
    // resident CTAs per SM, once per device
    static std::atomic<int> occ_cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int occ = occ_cache[dev & 63].load();
    if (occ <= 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_kernel<MT, U, BF16, INT4>, GEMV_WARPS * 32, 0);
        if (e != cudaSuccess) return e;
        if (occ <= 0) return cudaErrorInvalidConfiguration;
        occ_cache[dev & 63].store(occ);
    }
    const int64_t ngroups = (p.N + GEMV_R - 1) / GEMV_R;
    const int64_t blocks = (ngroups + GEMV_WARPS / p.kslices - 1) / (GEMV_WARPS / p.kslices);
    const int64_t cap = (int64_t)occ * sm_count;
    const int grid = (int)(blocks < cap ? blocks : cap);
    uint64_t gmagic = 0;
    if (p.V) {
        const uint64_t d = (uint64_t)(p.gb / 8);
        gmagic = ((1ull << 40) + d - 1) / d;  // ceil(2^40 / d)
    }
    return launch_pdl(gemv_kernel<MT, U, BF16, INT4>, grid, GEMV_WARPS * 32, 0, st, p, gmagic);
}

template <bool BF16, bool INT4>
cudaError_t launch_m(const GemvParams& p, int sm_count, cudaStream_t st) {
    if (p.M <= 1) return launch_t<1, 1, BF16, INT4>(p, sm_count, st);
    if (p.M <= 2) return launch_t<2, 2, BF16, INT4>(p, sm_count, st);
    if (p.M <= 4) return launch_t<4, 1, BF16, INT4>(p, sm_count, st);
    return launch_t<8, 1, BF16, INT4>(p, sm_count, st);
}

}  // namespace

int gemv_kslices(int64_t N, int64_t K, int b_int4, int64_t want_warps) {
    const int64_t nchunk = b_int4 ? K / 32 : K / 8;
    const int64_t groups = (N + GEMV_R - 1) / GEMV_R;
    int s = 1;
    // more slices while the GPU is short of warps and every lane keeps a chunk
    while (s < GEMV_WARPS && groups * s < want_warps && nchunk / (2 * s) >= 32) s *= 2;
    return s;
}

cudaError_t launch_gemv(const GemvParams& p, int sm_count, cudaStream_t st) {
    const int s = p.kslices;
    if (p.M < 1 || p.M > GEMV_MAX_M || p.N < 1 || p.K < 8 || !(s == 1 || s == 2 || s == 4 || s == 8))
        return cudaErrorInvalidValue;
    if (p.b_int4 ? (p.K % 32 != 0 || p.ldb % 32 != 0) : (p.K % 8 != 0 || p.ldb % 8 != 0)) return cudaErrorInvalidValue;
    if (p.lda % 8 != 0 || (reinterpret_cast<uintptr_t>(p.A) & 15) || (reinterpret_cast<uintptr_t>(p.B) & 15))
        return cudaErrorInvalidValue;
    // the group-index multiply is exact for 8-value block indices below 2^24 and gb / 8 below 2^16
    if (p.V && (p.gb < 8 || p.gb % 8 != 0 || p.gb >= (1 << 19) || p.K / 8 >= (1 << 24))) return cudaErrorInvalidValue;
    if (p.a_bf16)
        return p.b_int4 ? launch_m<true, true>(p, sm_count, st) : launch_m<true, false>(p, sm_count, st);
    return p.b_int4 ? launch_m<false, true>(p, sm_count, st) : launch_m<false, false>(p, sm_count, st);
}

}  // namespace qg
