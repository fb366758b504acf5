// Parameter blocks handed from the host dispatcher to the kernels.  Plain
// structs of integers and pointers, passed by value as kernel parameters.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "work_sched.h"

namespace qg {

enum DType : int32_t { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2, DT_S4 = 3, DT_S8 = 4, DT_E4M3 = 5, DT_E5M2 = 6 };

// Where a bounded wait gave up (recorded in the device status word).
enum WaitSite : uint32_t {
    SITE_PRODUCER_EMPTY = 1,
    SITE_MMA_FULL = 2,
    SITE_MMA_TMEM_EMPTY = 3,
    SITE_EPI_TMEM_FULL = 4,
    SITE_DRAIN = 5,
    SITE_DQ_RAW = 6,
    SITE_DQ_EMPTY = 7,
    SITE_MMA_OPERAND = 8,
    SITE_SELFTEST = 9,
};

// Where a device-side bounds check failed (checked builds only, see
// QG_DEVICE_CHECKS in common.cuh): recorded in the same status words, with
// bit 1 of the first word set.
enum CheckSite : uint32_t {
    CHECK_UNIT = 16,     // a unit's tile coordinates or K range outside the problem
    CHECK_PARTIAL = 17,  // a partial slot outside the workspace's partials
    CHECK_COUNTER = 18,  // a tile counter outside the workspace's barriers
    CHECK_ELEMENT = 19,  // an element of C or D outside its extent
};

// Epilogue: D = fma(alpha, acc, beta * C) rounded to D's type.
struct EpiParams {
    void* D;
    const void* C;     // NULL when beta == 0 (never read then)
    int64_t ldd, ldc;  // elements
    int64_t d_bstride, c_bstride;  // elements between batches (0 for grouped)
    int64_t M, N;      // output rows / columns (per batch)
    float alpha, beta;
    int32_t d_type;    // DT_F32 / DT_F16 / DT_BF16 (C has the same type), or DT_S8 (quantised, no C)
    int32_t swap;      // 0: tile rows are D rows; 1: tile rows are D columns
    int32_t vec_ok;    // C/D bases and ld allow 16-byte vector access
    int32_t tma;       // C/D move through shared memory with TMA (tmC / tmD)
    int32_t ncb;       // shared-memory C/D buffers per epilogue warp (TMA path)
    int32_t flags;     // EPI_BIAS | EPI_RELU | EPI_GELU (the ABI's GEMM_EPILOGUE_*)
    int32_t bias_type; // DT_F32 / DT_F16 / DT_BF16
    const void* bias;  // N values, one per output column (EPI_BIAS)
    const float* qscale;  // d_type DT_S8: M scales, one per output row
    int32_t qzp;          // d_type DT_S8: zero point
    int64_t d_extent, c_extent;  // elements of D / C the call may touch (bounds of the checked build)
    uint32_t* status;            // device status words (the checked build records failed checks there)
};

// Fused epilogue steps after x = alpha * acc + beta * c: + bias[column], then
// ReLU or GELU (DeepGEMM kernel-set blog, section 6.1).
enum EpiFlags : int32_t { EPI_BIAS = 1, EPI_RELU = 2, EPI_GELU = 4 };

// Group-wise scaling / int4 dequantisation of one shared-memory operand
// before the tensor core reads it (the role of the scale operands U/V that
// advance at K-group boundaries).  The operand's value at (row r, k) becomes
// RN(x[r][k] * scale[k / group][r]) in the MMA input type, with x the int4
// nibble or the stored 16-bit value.  The scale rows a K-step needs are
// copied into the stage by TMA together with the operand tiles.
struct OperandXform {
    int32_t has_scale;   // scale rows arrive with every stage (TMA), else unscaled
    int32_t has_zero;    // int4 operand: zero-point rows (one byte per value) arrive too
    int32_t scale_type;  // DT_F16 / DT_BF16
    int32_t group;       // group size along K: a multiple of 64, or a divisor of 64 (>= 8)
    int32_t sc_rows;     // scale rows per 64-wide K-step: max(1, 64 / group)
    int32_t int4;        // operand is packed int4 (raw tile rows of 32 bytes)
    int32_t active;      // any transform at all
};

struct DqParams {
    OperandXform x, y;   // X: UMMA M side (128-row tiles), Y: UMMA N side
    int64_t K;
    int32_t out_bf16;    // rounded operand type: 1 bf16, 0 f16
};

struct GemmKernelParams {
    SchedParams sched;
    EpiParams epi;
    DqParams dq;
    uint32_t idesc;       // tcgen05.mma instruction descriptor
    int32_t x3d, y3d;     // the X / Y tensor maps take a batch coordinate
    int32_t stages;       // shared-memory ring depth
    float* partials;      // fp32 partial tiles (split-K / stream-K)
    int32_t* counters;    // per-tile arrival counters (self-resetting)
    uint32_t* status;     // device status words [4]
    uint64_t timeout_ns;  // bound on every wait
    int32_t pair;         // CTA-pair kernel: units are 256-row tiles shared by the two CTAs of a cluster
    int32_t ks;           // K-steps per stage (>1: X/Y maps index K chunks of one K-step)
    int32_t kstep;        // elements per K-step: one 128-byte swizzle row (64 16-bit, 128 8-bit values)
    int32_t mma_f8;       // operands are 8-bit floats: tcgen05.mma.kind::f8f6f4
    uint64_t partials_bytes;  // workspace sizes (bounds of the checked build)
    uint64_t counters_bytes;
};

// Instruction descriptor of tcgen05.mma.kind::f16: fp32 accumulator (bits
// 4-5 = 1), A/B format (bits 7-9 / 10-12: 0 = f16, 1 = bf16), both operands
// K-major (bits 15, 16 = 0), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
QG_HD uint32_t make_idesc_f16(int ab_is_bf16, int m, int n) {
    uint32_t fmt = ab_is_bf16 ? 1u : 0u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4: the same fields, with
// the A/B formats E4M3 = 0 and E5M2 = 1.
QG_HD uint32_t make_idesc_f8(int a_e5m2, int b_e5m2, int m, int n) {
    return (1u << 4) | ((uint32_t)(a_e5m2 ? 1 : 0) << 7) | ((uint32_t)(b_e5m2 ? 1 : 0) << 10) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Tile widths (UMMA N) instantiated for each kernel.
#define QG_FOR_EACH_DENSE_BN(X) X(16) X(32) X(64) X(128) X(192) X(224) X(256)
#define QG_FOR_EACH_DQ_BN(X) X(16) X(32) X(64) X(128) X(256)
#define QG_FOR_EACH_PAIR_BN(X) X(128) X(224) X(256)

// Entry points implemented in the .cu files.
// The four tensor maps of one launch: X and Y operands, C and D (the last two
// are used only when EpiParams::tma is set).
struct GemmMaps {
    CUtensorMap x, y, c, d;
    CUtensorMap xs, ys;  // scale rows of X / Y (transforming kernel only)
    CUtensorMap z;       // zero-point rows of the int4 operand (transforming kernel only)
};

// Per-width launchers (explicitly instantiated in umma_gemm_bn*.cu and
// umma_dq_gemm_bn*.cu).
template <int BN>
cudaError_t launch_umma_bn(const GemmMaps& m, const GemmKernelParams& p, int grid, cudaStream_t st);
template <int BN>
int umma_stages_bn(int ks);
template <int BN>
cudaError_t launch_dq_bn(const GemmMaps& m, const GemmKernelParams& p, int grid, cudaStream_t st);
template <int BN>
int dq_stages_bn();
template <int BN>
cudaError_t launch_pair_bn(const GemmMaps& m, const GemmKernelParams& p, int grid, cudaStream_t st);
template <int BN>
int pair_stages_bn(int ks);
template <int BN>
int pair_max_clusters_bn();

cudaError_t launch_umma_gemm(int bn, const GemmMaps& maps, const GemmKernelParams& p, int grid, cudaStream_t st);
cudaError_t launch_umma_dq_gemm(int bn, const GemmMaps& maps, const GemmKernelParams& p, int grid,
                                cudaStream_t st);
cudaError_t launch_scale_c(const EpiParams& e, int64_t batches, cudaStream_t st);
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t timeout_ns, cudaStream_t st);
int umma_max_stages(int bn, int ks);
cudaError_t launch_umma_pair_gemm(int bn, const GemmMaps& maps, const GemmKernelParams& p, int grid, cudaStream_t st);
int umma_pair_max_stages(int bn, int ks);
int umma_pair_max_clusters(int bn);
int umma_dq_max_stages(int bn);
cudaError_t device_status_ptr(uint32_t** out);

}  // namespace qg
