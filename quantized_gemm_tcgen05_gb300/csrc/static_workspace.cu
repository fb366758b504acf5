// gemm_run_noalloc: gemm_run for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a plug-in inside a host
// framework whose caching allocator owns every byte of the device and hands
// out no scratch, or code on a latency-critical path where an allocation
// would synchronise the device.  gemm_run needs no allocation either, but its
// split-K / stream-K schedules need a caller-provided workspace.  This entry
// point supplies that workspace from a fixed array in the library's own
// device memory instead, so the caller passes only inputs and outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "gemm.h"
#include "handle_internal.h"

namespace {

constexpr size_t kNoallocBarriers = GEMM_NOALLOC_BARRIERS_SIZE;  // 16384 per-tile arrival counters
constexpr size_t kNoallocPartials = GEMM_NOALLOC_PARTIALS_SIZE;  // 8 MB of fp32 partial tiles
static_assert(kNoallocBarriers == (64u << 10) && kNoallocPartials == (8u << 20),
              "the documented limits of gemm_run_noalloc");

// Every GPU that loads the library holds this array until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBarriers + kNoallocPartials];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on `dev` (host code cannot use the symbol's own
// name: on the host it is only a stand-in).  Looked up once per device, with
// that device current.
int scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        int prev = -1;
        if (cudaGetDevice(&prev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (prev != dev) cudaSetDevice(prev);
        if (e != cudaSuccess || !ptr) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GEMM_OK;
}

}  // namespace

extern "C" int gemm_run_noalloc(gemm_handle_t h, const gemm_op_t* op, float alpha, const void* A,
                                const gemm_layout_t* Adesc, const void* U, const gemm_layout_t* Udesc, const void* B,
                                const gemm_layout_t* Bdesc, const void* V, const gemm_layout_t* Vdesc, float beta,
                                const void* C, const gemm_layout_t* Cdesc, void* D, const gemm_layout_t* Ddesc,
                                gemm_stream_t stream) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    void* base = nullptr;
    int rc = scratch_address(qg::handle_device(h), &base);
    if (rc) return rc;
    // the counters must start at zero; a previous call may have been cut short
    if (cudaMemsetAsync(base, 0, kNoallocBarriers, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    gemm_workspace_t ws;
    ws.barriers = base;
    ws.barriers_size = kNoallocBarriers;
    ws.partials = static_cast<unsigned char*>(base) + kNoallocBarriers;
    ws.partials_size = kNoallocPartials;
    return gemm_run(h, op, alpha, A, Adesc, U, Udesc, B, Bdesc, V, Vdesc, beta, C, Cdesc, D, Ddesc, &ws, stream);
}
