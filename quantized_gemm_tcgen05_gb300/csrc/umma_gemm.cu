// Entry points of the dense tcgen05 GEMM (dispatch over the tile widths
// instantiated in umma_gemm_bn*.cu), plus the small helper kernels: D = beta*C
// for K == 0 and the bounded-wait self-test.
#include "common.cuh"

namespace qg {

__device__ uint32_t g_device_status[4];

// D = beta * C (or 0), then the fused bias / activation, for K == 0, where
// no accumulator exists.
__global__ void scale_c_kernel(EpiParams e, int64_t batches) {
    const int64_t total = batches * e.M * e.N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / (e.M * e.N), rem = i % (e.M * e.N);
        const int64_t m = rem / e.N, n = rem % e.N;
        const float c = e.beta != 0.0f ? ld_elem(e.C, e.d_type, b * e.c_bstride + m * e.ldc + n) : 0.0f;
        const float x = e.beta != 0.0f ? e.beta * c : 0.0f;
        store_out(e, b * e.d_bstride + m * e.ldd + n, e.flags ? epi_finish(e, x, bias_at(e, n)) : x, m);
    }
}

// Self-test of the bounded wait: waits on an mbarrier that nothing arrives
// on, so the wait must run out, record SITE_SELFTEST and return.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const Guard g{status, timeout_ns, &abort_flag};
        if (!wait_bar(&bar, 0, g, SITE_SELFTEST)) atomicExch(&status[1], SITE_SELFTEST);
        mbar_arrive(&bar);  // complete the phase so nothing is left pending
    }
}

cudaError_t launch_umma_gemm(int bn, const GemmMaps& m, const GemmKernelParams& p, int grid, cudaStream_t st) {
    switch (bn) {
#define QG_CASE(B) \
    case B: return launch_umma_bn<B>(m, p, grid, st);
        QG_FOR_EACH_DENSE_BN(QG_CASE)
#undef QG_CASE
        default: return cudaErrorInvalidValue;
    }
}

int umma_max_stages(int bn, int ks) {
    switch (bn) {
#define QG_CASE(B) \
    case B: return umma_stages_bn<B>(ks);
        QG_FOR_EACH_DENSE_BN(QG_CASE)
#undef QG_CASE
        default: return 0;
    }
}

cudaError_t launch_umma_pair_gemm(int bn, const GemmMaps& m, const GemmKernelParams& p, int grid, cudaStream_t st) {
    switch (bn) {
#define QG_CASE(B) \
    case B: return launch_pair_bn<B>(m, p, grid, st);
        QG_FOR_EACH_PAIR_BN(QG_CASE)
#undef QG_CASE
        default: return cudaErrorInvalidValue;
    }
}

int umma_pair_max_stages(int bn, int ks) {
    switch (bn) {
#define QG_CASE(B) \
    case B: return pair_stages_bn<B>(ks);
        QG_FOR_EACH_PAIR_BN(QG_CASE)
#undef QG_CASE
        default: return 0;
    }
}

int umma_pair_max_clusters(int bn) {
    switch (bn) {
#define QG_CASE(B) \
    case B: return pair_max_clusters_bn<B>();
        QG_FOR_EACH_PAIR_BN(QG_CASE)
#undef QG_CASE
        default: return 0;
    }
}

cudaError_t launch_scale_c(const EpiParams& e, int64_t batches, cudaStream_t st) {
    int64_t total = batches * e.M * e.N;
    int grid = (int)((total + 255) / 256);
    if (grid > 4096) grid = 4096;
    if (grid < 1) grid = 1;
    scale_c_kernel<<<grid, 256, 0, st>>>(e, batches);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t timeout_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

cudaError_t device_status_ptr(uint32_t** out) {
    return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_device_status);
}

}  // namespace qg
