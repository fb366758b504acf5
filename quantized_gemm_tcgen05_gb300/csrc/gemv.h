// Small-M path of D = alpha * (A @ B^) + beta * C (decode shapes, M <= 8):
// a streaming matrix-vector kernel on the CUDA cores.  With M this small the
// product is bound by reading B from HBM, so the tensor core buys nothing;
// each warp streams rows of B with coalesced 16-byte loads, forms B^ the same
// way the tensor-core path does (int4 nibble or 16-bit value times its group
// scale, exact in fp32, rounded once to A's type), and accumulates the exact
// products a * b^ in fp32 ("InternLM Lmdeploy Gemm Interface", section
// Signature, for the operation; "InternLM Lmdeploy MainloopSm80V2", section
// Description, for the U/V group scales).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace qg {

constexpr int GEMV_MAX_M = 8;

struct GemvParams {
    const void* A;   // M x K, K contiguous (lda elements)
    const void* B;   // N rows of K values, K contiguous: 16-bit (ldb elements) or packed int4 (ldb nibbles)
    const void* V;   // [K / gb][ldv] 16-bit group scales of B, or null
    const void* Z;   // int4 B with V: [K / gb][ldz] zero points (low nibble of each byte), or null
    const void* C;   // M x N (ldc), read only when beta != 0
    void* D;         // M x N (ldd)
    int64_t lda, ldb, ldv, ldz, ldc, ldd;
    int64_t M, N, K;
    float alpha, beta;
    int32_t a_bf16;  // A (and 16-bit B) is bf16, else fp16
    int32_t b_int4;  // B is packed int4 (two's-complement nibbles, k = 2t in bits 3:0 of byte t)
    int32_t v_bf16;  // V is bf16, else fp16
    int32_t gb;      // group size of V along K
    int32_t d_type;  // DT_F32 / DT_F16 / DT_BF16
    int32_t kslices; // warps that split one row group's K range (1, 2, 4 or 8)
    int32_t epi_flags;  // EPI_BIAS | EPI_RELU | EPI_GELU, applied after alpha / beta
    int32_t bias_type;  // DT_F32 / DT_F16 / DT_BF16
    const void* bias;   // N values, one per output column
    const float* qscale;  // d_type DT_S8: M scales, one per output row
    int32_t qzp;          // d_type DT_S8: zero point
};

// Launch for M <= GEMV_MAX_M.  Returns cudaErrorInvalidValue for shapes the
// kernel does not take (the dispatcher never offers those).
cudaError_t launch_gemv(const GemvParams& p, int sm_count, cudaStream_t st);

// K slices per row group that give at least `want_warps` warps of work.
int gemv_kslices(int64_t N, int64_t K, int b_int4, int64_t want_warps);

}  // namespace qg
