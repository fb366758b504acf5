// The C ABI (include/gemm.h): handle, operand validation, tensor-map
// construction, dispatch through the cache / heuristic / measurer, kernel
// launch, cache export/import.  Host code only; every arithmetic step of the
// GEMM runs in the CUDA kernels.
#include "gemm.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <new>
#include <string>
#include <vector>

#include "dispatch.h"
#include "gemv.h"
#include "handle_internal.h"
#include "kparams.h"

using namespace qg;

#ifdef QG_DEVICE_CHECKS
static constexpr bool kDeviceChecksHost = true;
#else
static constexpr bool kDeviceChecksHost = false;
#endif

struct gemm_handle {
    int device = 0;
    int sm_count = 0;
    int cc = 0;
    std::string name;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    uint32_t* status = nullptr;  // device status words
    std::map<Key, Choice> cache;
    std::string last_choice = "none";
    bool log = false;
    int force_splitk = 0;
    uint64_t timeout_ns = 2000000000ull;
    // Host-path caches: tensor maps by their encode arguments (direct-mapped)
    // and recently validated device pointers (ring).  They keep a repeated
    // gemm_run call to a few microseconds of host work.
    struct MapEntry {
        uint64_t key[16];
        CUtensorMap map;
        bool valid;
    };
    MapEntry maps[128] = {};
    int pair_clusters = -1;  // clusters of two the CTA-pair kernel can keep resident (queried once)
    const void* dev_ptrs[64] = {};
    int dev_ptr_next = 0;
};

namespace {

bool is16(int32_t t) { return t == GEMM_F16 || t == GEMM_BF16; }
bool is_f8(int32_t t) { return t == GEMM_E4M3 || t == GEMM_E5M2; }
// Bytes per element of a tensor-core input (16-bit or 8-bit float).
int64_t in_bytes(int32_t t) { return is_f8(t) ? 1 : 2; }
// Tensor-map element type of a tensor-core input.
CUtensorMapDataType in_map_type(int32_t t) {
    if (is_f8(t)) return CU_TENSOR_MAP_DATA_TYPE_UINT8;  // raw bytes: TMA only moves them
    return t == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}
bool is_float_out(int32_t t) { return t == GEMM_F32 || t == GEMM_F16 || t == GEMM_BF16; }
static_assert(GEMM_F32 == DT_F32 && GEMM_F16 == DT_F16 && GEMM_BF16 == DT_BF16 && GEMM_S4 == DT_S4 &&
                  GEMM_S8 == DT_S8 && GEMM_E4M3 == DT_E4M3 && GEMM_E5M2 == DT_E5M2,
              "the C ABI's dtype codes are the kernels' codes");
static_assert(GEMM_EPILOGUE_BIAS == EPI_BIAS && GEMM_EPILOGUE_RELU == EPI_RELU && GEMM_EPILOGUE_GELU == EPI_GELU,
              "the C ABI's epilogue flags are the kernels' flags");


bool device_pointer_uncached(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Validate one operand layout against the expected shape and order.
bool device_pointer(gemm_handle* h, const void* p) {
    for (const void* q : h->dev_ptrs)
        if (q == p) return true;
    if (!device_pointer_uncached(p)) return false;
    h->dev_ptrs[h->dev_ptr_next] = p;
    h->dev_ptr_next = (h->dev_ptr_next + 1) % 64;
    return true;
}

// cuTensorMapEncodeTiled through the handle's cache (same arguments, same map).
CUresult encode_cached(gemm_handle* h, CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank, const void* ptr,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       CUtensorMapSwizzle swz) {
    uint64_t key[16] = {0};
    key[0] = (uint64_t)dt | ((uint64_t)rank << 8) | ((uint64_t)swz << 16);
    key[1] = reinterpret_cast<uintptr_t>(ptr);
    for (cuuint32_t i = 0; i < rank && i < 5; ++i) {
        key[2 + i] = dims[i];
        key[7 + i] = box[i];
        if (i + 1 < rank) key[12 + i] = strides[i];
    }
    uint64_t hsh = 1469598103934665603ull;
    for (uint64_t k : key) hsh = (hsh ^ k) * 1099511628211ull;
    gemm_handle::MapEntry& e = h->maps[hsh % 128];
    if (e.valid && memcmp(e.key, key, sizeof key) == 0) {
        *m = e.map;
        return CUDA_SUCCESS;
    }
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = h->encode(m, dt, rank, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
        memcpy(e.key, key, sizeof key);
        e.map = *m;
        e.valid = true;
    }
    return r;
}

int check_layout(const gemm_layout_t* d, int32_t order, int64_t rows, int64_t cols) {
    if (!d) return GEMM_ERR_INVALID_ARG;
    if (d->order != order) return GEMM_ERR_UNSUPPORTED;
    if (d->rows != rows || d->cols != cols || d->num < 1) return GEMM_ERR_INVALID_ARG;
    const int64_t inner = order == GEMM_ROW_MAJOR ? cols : rows;
    if (d->ld < (inner > 0 ? inner : 1)) return GEMM_ERR_INVALID_ARG;
    if (d->num > 1 && d->batch_stride < 0) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int qg::handle_device(gemm_handle_t h) { return h ? h->device : -1; }

namespace {

// Elements of D (or C) a call may touch: batches x rows, the last row N long.
int64_t out_extent(int64_t M, int64_t N, int64_t ld, int32_t batches, int64_t bstride) {
    if (M <= 0 || N <= 0) return 0;
    return (int64_t)(batches > 1 ? batches - 1 : 0) * bstride + (M - 1) * ld + N;
}

// The checked build's self-test knob: GEMM_CHECK_SHRINK_WORKSPACE=1 tells the
// kernels a quarter of the partials buffer the caller passed (the buffer
// itself is whole, so the accesses the check then skips stay inside it).
uint64_t checked_partials_bytes(uint64_t bytes) {
#ifdef QG_DEVICE_CHECKS
    const char* e = getenv("GEMM_CHECK_SHRINK_WORKSPACE");
    if (e && e[0] == '1') return bytes / 4;
#endif
    return bytes;
}

}  // namespace

extern "C" {

const char* gemm_status_string(int s) {
    switch (s) {
        case GEMM_OK: return "ok";
        case GEMM_ERR_INVALID_ARG: return "invalid argument";
        case GEMM_ERR_UNSUPPORTED: return "unsupported operand combination or device";
        case GEMM_ERR_WORKSPACE: return "workspace missing or too small";
        case GEMM_ERR_CUDA: return "CUDA error";
        case GEMM_ERR_NO_KERNEL: return "no kernel accepts the problem";
        case GEMM_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
        case GEMM_ERR_BAD_CACHE: return "malformed or foreign dispatch cache";
        case GEMM_ERR_DEVICE_CHECK: return "a device-side bounds check failed (checked build)";
        default: return "unknown status";
    }
}

int gemm_create(gemm_handle_t* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_UNSUPPORTED;  // kernels are built for sm_103a
    gemm_handle* h = new (std::nothrow) gemm_handle;
    if (!h) return GEMM_ERR_CUDA;
    h->device = dev;
    h->sm_count = prop.multiProcessorCount;
    h->cc = prop.major * 10 + prop.minor;
    h->name = prop.name;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        delete h;
        return GEMM_ERR_CUDA;
    }
    h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    if (device_status_ptr(&h->status) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return GEMM_ERR_CUDA;
    }
    const char* lg = getenv("GEMM_LOG");
    h->log = lg && lg[0] && lg[0] != '0';
    const char* fs = getenv("GEMM_FORCE_SPLITK");
    if (fs) h->force_splitk = atoi(fs);
    const char* to = getenv("GEMM_WAIT_TIMEOUT_MS");
    if (to && atoll(to) > 0) h->timeout_ns = (uint64_t)atoll(to) * 1000000ull;
    *out = h;
    return GEMM_OK;
}

int gemm_destroy(gemm_handle_t h) {
    delete h;
    return GEMM_OK;
}

}  // extern "C"

namespace {

// Tensor map over a [batches][rows][K] operand stored with K contiguous; a
// box is one K-step (128 bytes) of box_rows rows.
int make_map(gemm_handle* h, CUtensorMap* m, const void* ptr, int32_t type, int64_t K, int64_t rows, int64_t ld,
             int32_t batches, int64_t bstride, int32_t box_rows) {
    const CUtensorMapDataType dt = in_map_type(type);
    const int64_t es = in_bytes(type);
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)batches};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * es), (cuuint64_t)(bstride * es)};
    cuuint32_t box[3] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows, 1};
    const cuuint32_t rank = batches > 1 ? 3 : 2;
    CUresult r = encode_cached(h, m, dt, rank, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Tensor map over a K-major operand viewed as [K-steps][rows][one K-step of
// 128 bytes]: a box of several K-steps x box_rows rows lands as that many
// SWIZZLE_128B tiles, one copy for several K-steps.  Only for K a multiple of
// the K-step (the inner dimension must not run past a row).
int make_map_kchunk(gemm_handle* h, CUtensorMap* m, const void* ptr, int32_t type, int64_t K, int64_t rows, int64_t ld,
                    int32_t box_rows, int32_t chunks) {
    const CUtensorMapDataType dt = in_map_type(type);
    const int64_t es = in_bytes(type), kstep = 128 / es;
    cuuint64_t dims[3] = {(cuuint64_t)kstep, (cuuint64_t)rows, (cuuint64_t)(K / kstep)};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * es), 128};
    cuuint32_t box[3] = {(cuuint32_t)kstep, (cuuint32_t)box_rows, (cuuint32_t)chunks};
    CUresult r = encode_cached(h, m, dt, 3, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// The same K-chunk view over a [batches][rows][K] operand (grouped experts):
// [batches][K-steps][rows][one K-step], one expert per box.
int make_map_kchunk4(gemm_handle* h, CUtensorMap* m, const void* ptr, int32_t type, int64_t K, int64_t rows,
                     int64_t ld, int32_t batches, int64_t bstride, int32_t box_rows, int32_t chunks) {
    const CUtensorMapDataType dt = in_map_type(type);
    const int64_t es = in_bytes(type), kstep = 128 / es;
    cuuint64_t dims[4] = {(cuuint64_t)kstep, (cuuint64_t)rows, (cuuint64_t)(K / kstep), (cuuint64_t)batches};
    cuuint64_t strides[3] = {(cuuint64_t)(ld * es), 128, (cuuint64_t)(bstride * es)};
    cuuint32_t box[4] = {(cuuint32_t)kstep, (cuuint32_t)box_rows, (cuuint32_t)chunks, 1};
    CUresult r = encode_cached(h, m, dt, 4, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Tensor map over packed int4 rows: [batches][rows][K/2 bytes], box 32 bytes
// x rows, no swizzle (the dequantising warps rewrite the tile into the
// swizzled layout the tensor core reads).
int make_map_s4(gemm_handle* h, CUtensorMap* m, const void* ptr, int64_t K, int64_t rows, int64_t ld_nibbles,
                int32_t box_rows, int32_t batches = 1, int64_t bstride_nibbles = 0) {
    cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)rows, (cuuint64_t)batches};
    cuuint64_t strides[2] = {(cuuint64_t)(ld_nibbles / 2), (cuuint64_t)(bstride_nibbles / 2)};
    cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
    CUresult r = encode_cached(h, m, CU_TENSOR_MAP_DATA_TYPE_UINT8, batches > 1 ? 3 : 2, ptr, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Tensor map over a [batches][M][N] row-major C or D with 32 x 32 boxes in
// the swizzled layout the TMA epilogue reads and writes (64-byte rows for
// 16-bit types, 128-byte rows for fp32).
int make_map_cd(gemm_handle* h, CUtensorMap* m, const void* ptr, int32_t type, int64_t M, int64_t N, int64_t ld,
                int32_t batches, int64_t bstride) {
    const int64_t es = type == GEMM_F32 ? 4 : 2;
    CUtensorMapDataType dt = type == GEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                              : (type == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)batches};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * es), (cuuint64_t)(bstride * es)};
    cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t rank = batches > 1 ? 3 : 2;
    CUresult r = encode_cached(h, m, dt, rank, ptr, dims, strides, box,
                               es == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Tensor map over a [batches][groups][cols] row-major scale matrix (U or V;
// one per expert for grouped problems): each K-step copies box_rows group
// rows x box_cols columns into its stage.
int make_map_scale(gemm_handle* h, CUtensorMap* m, const void* ptr, int32_t type, int64_t groups, int64_t cols,
                   int64_t ld, int32_t box_cols, int32_t box_rows, int32_t batches = 1, int64_t bstride = 0) {
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)groups, (cuuint64_t)batches};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(bstride * 2)};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    CUtensorMapDataType dt = type == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = encode_cached(h, m, dt, batches > 1 ? 3 : 2, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Tensor map over the [batches][groups][cols] byte matrix of int4 zero points,
// boxed like the scale rows.
int make_map_zero(gemm_handle* h, CUtensorMap* m, const void* ptr, int64_t groups, int64_t cols, int64_t ld,
                  int32_t box_cols, int32_t box_rows, int32_t batches, int64_t bstride) {
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)groups, (cuuint64_t)batches};
    cuuint64_t strides[2] = {(cuuint64_t)ld, (cuuint64_t)bstride};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    CUresult r = encode_cached(h, m, CU_TENSOR_MAP_DATA_TYPE_UINT8, batches > 1 ? 3 : 2, ptr, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Programs a choice can use: SMs, or for the CTA pair twice the resident clusters.
int capacity(gemm_handle* h, const Choice& c) {
    if (!c.pair) return h->sm_count;
    if (h->pair_clusters < 0) {
        const int n = umma_pair_max_clusters(256);
        h->pair_clusters = n > 0 ? n : 0;
    }
    const int cap = 2 * h->pair_clusters;
    return cap < h->sm_count ? cap : h->sm_count;
}

// K-steps the CTA-pair kernel copies per TMA box: two when K is a multiple of
// 64 and the problem is not batched, else one (GEMM_PAIR_KS=1|2|3 overrides
// the two).
int pair_kchunks(const Problem& p) {
    static const int want = [] {
        const char* e = getenv("GEMM_PAIR_KS");
        const int v = e ? atoi(e) : 2;
        return v >= 1 && v <= 3 ? v : 2;
    }();
    if (want < 2 || p.K % kstep_of(p) != 0 || p.batches != 1 || p.K < kstep_of(p)) return 1;
    return want;
}

// K-steps the single-CTA kernel copies per TMA box: up to GEMM_KS (default 2,
// at most 3) when K is a multiple of 64, the problem is not batched and three
// stages of that many K-steps still fit; else one.
int single_kchunks(const Problem& p, const Choice& c) {
    static const int want = [] {
        const char* e = getenv("GEMM_KS");
        const int v = e ? atoi(e) : 2;
        return v >= 1 && v <= 3 ? v : 2;
    }();
    if (p.K % kstep_of(p) != 0 || p.batches != 1 || p.K < kstep_of(p) || p.family != FAM_DENSE) return 1;
    for (int ks = want; ks > 1; --ks)
        if (umma_max_stages(c.bn, ks) >= 3) return ks;
    return 1;
}

// The small-M streaming kernel: no workspace, no tensor maps.
int launch_gemv_choice(gemm_handle* h, const Problem& p, cudaStream_t st) {
    GemvParams g;
    memset(&g, 0, sizeof g);
    g.A = p.A;
    g.B = p.B;
    g.V = p.V;
    g.Z = p.Z;
    g.ldz = p.ldz;
    g.C = p.beta != 0.0f ? p.C : nullptr;
    g.D = p.D;
    g.lda = p.lda;
    g.ldb = p.ldb;
    g.ldv = p.ldv;
    g.ldc = p.ldc;
    g.ldd = p.ldd;
    g.M = p.M;
    g.N = p.N;
    g.K = p.K;
    g.alpha = p.alpha;
    g.beta = p.beta;
    g.a_bf16 = p.a_type == GEMM_BF16;
    g.b_int4 = p.b_type == GEMM_S4;
    g.v_bf16 = p.v_type == GEMM_BF16;
    g.gb = p.V ? p.gb : 0;
    g.d_type = p.d_type;
    g.epi_flags = p.epi_flags;
    g.bias = p.bias;
    g.bias_type = p.bias_type;
    g.qscale = p.qscale;
    g.qzp = p.qzp;
    // enough warps for the weight stream: about 24 per SM (GEMM_GEMV_KSLICES
    // = 1, 2, 4 or 8 overrides the split, for tuning)
    g.kslices = gemv_kslices(p.N, p.K, g.b_int4, (int64_t)h->sm_count * 24);
    if (const char* ks = getenv("GEMM_GEMV_KSLICES")) {
        const int v = atoi(ks);
        if (v == 1 || v == 2 || v == 4 || v == 8) g.kslices = v;
    }
    const cudaError_t e = launch_gemv(g, h->sm_count, st);
    if (e == cudaErrorInvalidValue) return GEMM_ERR_NO_KERNEL;
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

int launch_choice(gemm_handle* h, const Problem& p, const Choice& c, const gemm_workspace_t* ws, cudaStream_t st) {
    if (c.gemv) return launch_gemv_choice(h, p, st);
    GemmKernelParams kp;
    memset(&kp, 0, sizeof kp);
    if (c.pair && capacity(h, c) < 2) return GEMM_ERR_NO_KERNEL;
    kp.sched = make_sched(p, c, capacity(h, c));
    const size_t need_p = partials_bytes_needed(kp.sched, c.bn, c.pair);
    const size_t need_c = counters_bytes_needed(kp.sched, c.pair);
    if (need_p || need_c) {
        if (!ws || !ws->partials || !ws->barriers || ws->partials_size < need_p || ws->barriers_size < need_c)
            return GEMM_ERR_WORKSPACE;
        if (!aligned16(ws->partials) || (reinterpret_cast<uintptr_t>(ws->barriers) & 3u)) return GEMM_ERR_INVALID_ARG;
        kp.partials = static_cast<float*>(ws->partials);
        kp.counters = static_cast<int32_t*>(ws->barriers);
        kp.partials_bytes = checked_partials_bytes(ws->partials_size);
        kp.counters_bytes = ws->barriers_size;
    }
    EpiParams& e = kp.epi;
    e.D = p.D;
    e.C = p.beta != 0.0f ? p.C : nullptr;
    e.ldd = p.ldd;
    e.ldc = p.ldc;
    e.d_bstride = is_grouped(p) ? 0 : p.d_bs;
    e.c_bstride = is_grouped(p) ? 0 : p.c_bs;
    e.d_extent = out_extent(p.M, p.N, p.ldd, is_grouped(p) ? 1 : p.batches, p.d_bs);
    e.c_extent = e.C ? out_extent(p.M, p.N, p.ldc, is_grouped(p) ? 1 : p.batches, p.c_bs) : 0;
    e.status = h->status;
    e.M = p.M;
    e.N = p.N;
    e.alpha = p.alpha;
    e.beta = p.beta;
    e.d_type = p.d_type;
    e.flags = p.epi_flags;
    e.bias = p.bias;
    e.bias_type = p.bias_type;
    e.qscale = p.qscale;
    e.qzp = p.qzp;
    e.swap = c.swap;
    const int64_t eb = p.d_type == GEMM_F32 ? 4 : (p.d_type == GEMM_S8 ? 1 : 2);
    e.vec_ok = aligned16(p.D) && (p.ldd * eb) % 16 == 0 &&
               (e.C == nullptr || (aligned16(p.C) && (p.ldc * eb) % 16 == 0)) &&
               (p.batches == 1 || ((p.d_bs * eb) % 16 == 0 && (e.C == nullptr || (p.c_bs * eb) % 16 == 0)));
    kp.mma_f8 = is_f8(p.a_type);
    kp.kstep = kstep_of(p);
    kp.idesc = kp.mma_f8 ? make_idesc_f8(p.a_type == GEMM_E5M2, p.b_type == GEMM_E5M2, 128, c.bn)
                         : make_idesc_f16(p.a_type == GEMM_BF16, 128, c.bn);
    kp.status = h->status;
    kp.timeout_ns = h->timeout_ns;

    GemmMaps maps;
    memset(&maps, 0, sizeof maps);
    CUtensorMap& tx = maps.x;
    CUtensorMap& ty = maps.y;
    int rc;
    const bool dq = is_dq(p);
    const bool s4 = p.b_type == GEMM_S4;
    if (p.family == FAM_GROUPED_DQ) {
        // experts' int4 or 16-bit B, one slice per expert (the Y operand's
        // third coordinate); A (the token rows) is one 2-D operand
        rc = make_map(h, &tx, p.A, p.a_type, p.K, p.M, p.lda, 1, 0, 128);
        if (rc == GEMM_OK)
            rc = s4 ? make_map_s4(h, &ty, p.B, p.K, p.N, p.ldb, c.bn, p.num_experts, p.b_bs)
                    : make_map(h, &ty, p.B, p.b_type, p.K, p.N, p.ldb, p.num_experts, p.b_bs, c.bn);
        kp.x3d = 0;
        kp.y3d = p.num_experts > 1;
    } else if (p.family == FAM_GROUPED && c.pair && pair_kchunks(p) > 1) {
        // 256-row expert blocks on CTA pairs: each CTA its 128 token rows and
        // half of the expert's Y tile, several K-steps per copy
        const int ks = pair_kchunks(p);
        rc = make_map_kchunk(h, &tx, p.A, p.a_type, p.K, p.M, p.lda, 128, ks);
        if (rc == GEMM_OK)
            rc = make_map_kchunk4(h, &ty, p.B, p.b_type, p.K, p.N, p.ldb, p.num_experts, p.b_bs, c.bn / 2, ks);
        kp.x3d = 0;
        kp.y3d = 1;
        kp.ks = ks;
    } else if (p.family == FAM_GROUPED) {
        rc = make_map(h, &tx, p.A, p.a_type, p.K, p.M, p.lda, 1, 0, 128);
        if (rc == GEMM_OK)
            rc = make_map(h, &ty, p.B, p.b_type, p.K, p.N, p.ldb, p.num_experts, p.b_bs, c.pair ? c.bn / 2 : c.bn);
        kp.x3d = 0;
        kp.y3d = 1;
    } else if (!c.pair && !dq && single_kchunks(p, c) > 1) {
        // several K-steps per copy: X is B (rows N) when swapped, else A
        const void* X = c.swap ? p.B : p.A;
        const void* Y = c.swap ? p.A : p.B;
        const int ks = single_kchunks(p, c);
        rc = make_map_kchunk(h, &tx, X, p.a_type, p.K, c.swap ? p.N : p.M, c.swap ? p.ldb : p.lda, 128, ks);
        if (rc == GEMM_OK)
            rc = make_map_kchunk(h, &ty, Y, p.a_type, p.K, c.swap ? p.M : p.N, c.swap ? p.lda : p.ldb, c.bn, ks);
        kp.x3d = kp.y3d = 0;
        kp.ks = ks;
    } else if (c.swap) {
        rc = s4 ? make_map_s4(h, &tx, p.B, p.K, p.N, p.ldb, 128) : make_map(h, &tx, p.B, p.b_type, p.K, p.N, p.ldb, 1, 0, 128);
        if (rc == GEMM_OK) rc = make_map(h, &ty, p.A, p.a_type, p.K, p.M, p.lda, 1, 0, c.bn);
        kp.x3d = kp.y3d = 0;
    } else if (c.pair && pair_kchunks(p) > 1) {
        // the CTA pair loads half of the Y tile in each CTA, several K-steps per copy
        const int ks = pair_kchunks(p);
        rc = make_map_kchunk(h, &tx, p.A, p.a_type, p.K, p.M, p.lda, 128, ks);
        if (rc == GEMM_OK) rc = make_map_kchunk(h, &ty, p.B, p.b_type, p.K, p.N, p.ldb, c.bn / 2, ks);
        kp.x3d = kp.y3d = 0;
        kp.ks = ks;
    } else {
        rc = make_map(h, &tx, p.A, p.a_type, p.K, p.M, p.lda, p.batches, p.a_bs, 128);
        // the CTA pair loads half of the Y tile in each CTA
        const int32_t y_box = c.pair ? c.bn / 2 : c.bn;
        if (rc == GEMM_OK)
            rc = s4 ? make_map_s4(h, &ty, p.B, p.K, p.N, p.ldb, c.bn)
                    : make_map(h, &ty, p.B, p.b_type, p.K, p.N, p.ldb, p.batches, p.b_bs, y_box);
        kp.x3d = kp.y3d = p.batches > 1;
    }
    if (rc != GEMM_OK) return rc;
    // TMA epilogue: C / D through shared memory when their layout allows it
    {
        const int64_t es = p.d_type == GEMM_F32 ? 4 : 2;
        auto ok16 = [&](const void* ptr, int64_t ld, int64_t bs) {
            return aligned16(ptr) && (ld * es) % 16 == 0 && (p.batches == 1 || (bs * es) % 16 == 0);
        };
        const char* et = getenv("GEMM_EPI_TMA");
        const bool allowed = !(et && et[0] == '0');
        e.tma = allowed && !c.swap && !is_grouped(p) && c.bn >= 32 && p.d_type != GEMM_S8 &&
                ok16(p.D, p.ldd, p.d_bs) &&
                (e.C == nullptr || ok16(p.C, p.ldc, p.c_bs)) && !(c.pair && es == 4);
        if (e.tma) {
            // buffers per epilogue warp: 32 KB of epilogue shared memory split
            // over 4 warps
            e.ncb = es == 2 ? 4 : 2;
            rc = make_map_cd(h, &maps.d, p.D, p.d_type, p.M, p.N, p.ldd, p.batches, p.d_bs);
            if (rc == GEMM_OK && e.C) rc = make_map_cd(h, &maps.c, p.C, p.d_type, p.M, p.N, p.ldc, p.batches, p.c_bs);
            if (rc != GEMM_OK) return rc;
        }
    }
    if (dq) {
        DqParams& d = kp.dq;
        d.K = p.K;
        d.out_bf16 = p.a_type == GEMM_BF16;
        auto xform = [](const void* scale, int32_t type, int32_t group, int32_t int4) {
            OperandXform o;
            o.has_scale = scale != nullptr;
            o.has_zero = 0;
            o.scale_type = type;
            o.group = scale ? group : 64;
            o.sc_rows = scale ? (group >= 64 ? 1 : 64 / group) : 0;
            o.int4 = int4;
            o.active = scale != nullptr || int4;
            return o;
        };
        const OperandXform a_side = xform(p.U, p.u_type, p.ga, 0);
        OperandXform b_side = xform(p.V, p.v_type, p.gb, s4 ? 1 : 0);
        b_side.has_zero = p.Z != nullptr;
        d.x = c.swap ? b_side : a_side;
        d.y = c.swap ? a_side : b_side;
        // scale rows: X side tiles are 128 rows, Y side tiles are BN rows
        const void* xs_ptr = c.swap ? p.V : p.U;
        const void* ys_ptr = c.swap ? p.U : p.V;
        if (xs_ptr) {
            const bool v = c.swap;
            // 136 columns: the copy starts at the 8-aligned column below the
            // tile's first row (token blocks of grouped problems start anywhere)
            rc = make_map_scale(h, &maps.xs, xs_ptr, v ? p.v_type : p.u_type, p.K / (v ? p.gb : p.ga), v ? p.N : p.M,
                                v ? p.ldv : p.ldu, 136, d.x.sc_rows);
            if (rc != GEMM_OK) return rc;
        }
        if (ys_ptr) {
            const bool v = !c.swap;
            const int32_t nb = v && kp.y3d ? p.num_experts : 1;  // grouped: V per expert
            rc = make_map_scale(h, &maps.ys, ys_ptr, v ? p.v_type : p.u_type, p.K / (v ? p.gb : p.ga), v ? p.N : p.M,
                                v ? p.ldv : p.ldu, c.bn, d.y.sc_rows, nb, v ? p.v_bs : 0);
            if (rc != GEMM_OK) return rc;
        }
        if (p.Z) {  // zero points of the int4 B, on whichever side B is
            const int32_t nb = !c.swap && kp.y3d ? p.num_experts : 1;
            rc = make_map_zero(h, &maps.z, p.Z, p.K / p.gb, p.N, p.ldz, c.swap ? 128 : c.bn,
                               c.swap ? d.x.sc_rows : d.y.sc_rows, nb, p.z_bs);
            if (rc != GEMM_OK) return rc;
        }
        kp.stages = umma_dq_max_stages(c.bn);
        if (kp.stages < 2) return GEMM_ERR_NO_KERNEL;
        if (const char* fs = getenv("GEMM_STAGES")) {  // ring depth override for tuning sweeps
            const int want = atoi(fs);
            if (want >= 2 && want < kp.stages) kp.stages = want;
        }
        cudaError_t ce = launch_umma_dq_gemm(c.bn, maps, kp, kp.sched.programs, st);
        return ce == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }
    if (kp.ks == 0) kp.ks = 1;
    kp.stages = c.pair ? umma_pair_max_stages(c.bn, kp.ks) : umma_max_stages(c.bn, kp.ks);
    if (kp.stages < 2) return GEMM_ERR_NO_KERNEL;
    if (const char* fs = getenv("GEMM_STAGES")) {  // ring depth override for tuning sweeps
        const int want = atoi(fs);
        if (want >= 2 && want < kp.stages) kp.stages = want;
    }
    if (c.pair) {
        kp.pair = 1;
        kp.idesc = kp.mma_f8 ? make_idesc_f8(p.a_type == GEMM_E5M2, p.b_type == GEMM_E5M2, 256, c.bn)
                             : make_idesc_f16(p.a_type == GEMM_BF16, 256, c.bn);
        cudaError_t ce = launch_umma_pair_gemm(c.bn, maps, kp, 2 * kp.sched.programs, st);
        return ce == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }
    cudaError_t ce = launch_umma_gemm(c.bn, maps, kp, kp.sched.programs, st);
    return ce == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

bool workspace_fits(gemm_handle* h, const Problem& p, const Choice& c, const gemm_workspace_t* ws) {
    if (c.gemv) return true;
    SchedParams s = make_sched(p, c, capacity(h, c));
    const size_t need_p = partials_bytes_needed(s, c.bn, c.pair), need_c = counters_bytes_needed(s, c.pair);
    if (!need_p && !need_c) return true;
    return ws && ws->partials && ws->barriers && ws->partials_size >= need_p && ws->barriers_size >= need_c;
}

// Time one candidate on the stream: one warm-up, then the median of 3.
float measure(gemm_handle* h, const Problem& p, const Choice& c, const gemm_workspace_t* ws, cudaStream_t st) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return -1.0f;
    if (cudaEventCreate(&b) != cudaSuccess) {
        cudaEventDestroy(a);
        return -1.0f;
    }
    float best[3] = {-1, -1, -1};
    bool ok = launch_choice(h, p, c, ws, st) == GEMM_OK;
    for (int i = 0; ok && i < 3; ++i) {
        cudaEventRecord(a, st);
        ok = launch_choice(h, p, c, ws, st) == GEMM_OK;
        cudaEventRecord(b, st);
        if (ok && cudaEventSynchronize(b) == cudaSuccess) cudaEventElapsedTime(&best[i], a, b);
        else ok = false;
    }
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (!ok) {
        cudaGetLastError();
        return -1.0f;
    }
    std::sort(best, best + 3);
    return best[1] * 1000.0f;
}

// GEMM_FORCE_KERNEL="<family>_bn<N>[_swap]/<dp|streamk|splitk<S>>" (the
// names gemm_last_choice prints) pins the kernel, for tests and sweeps.
bool forced_kernel(const Problem& p, Choice* out) {
    const char* f = getenv("GEMM_FORCE_KERNEL");
    if (!f || !*f) return false;
    if (strcmp(f, "gemv") == 0) {
        if (!gemv_eligible(p)) return false;
        *out = Choice();
        out->bn = 128;
        out->gemv = 1;
        return true;
    }
    const char* bn = strstr(f, "bn");
    const char* slash = strchr(f, '/');
    if (!bn || !slash) return false;
    Choice c;
    c.bn = atoi(bn + 2);
    c.swap = strstr(f, "_swap") != nullptr && strstr(f, "_swap") < slash;
    c.pair = strncmp(f, "umma2_", 6) == 0;
    if (strncmp(slash + 1, "dp", 2) == 0) {
        c.sched = SCHED_DP;
    } else if (strncmp(slash + 1, "streamk", 7) == 0) {
        c.sched = SCHED_STREAMK;
    } else if (strncmp(slash + 1, "splitk", 6) == 0) {
        c.sched = SCHED_SPLITK;
        c.splits = atoi(slash + 7);
    } else {
        return false;
    }
    if (!(c.bn == 16 || c.bn == 32 || c.bn == 64 || c.bn == 128 || c.bn == 192 || c.bn == 224 || c.bn == 256))
        return false;
    if (is_dq(p) && (c.bn == 192 || c.bn == 224)) return false;
    if (c.swap && (is_grouped(p) || p.batches != 1)) return false;
    if (c.pair && ((p.family != FAM_DENSE && p.family != FAM_GROUPED) || c.swap || c.sched == SCHED_SPLITK ||
                   !(c.bn == 128 || c.bn == 224 || c.bn == 256)))
        return false;
    if (is_grouped(p)) c.sched = SCHED_DP;
    *out = c;
    return true;
}

// The last step of an automatic choice, shared by gemm_run and the host-only
// gemm_heuristic_choice: grouped problems run data-parallel; a split whose
// partials do not fit the workspace first tries half-width tiles, then (when
// the schedule was not forced) runs unsplit.  Returns false when a forced
// schedule does not fit.
template <typename Fits>
bool settle_schedule(const Problem& p, Choice* c, bool forced, const Fits& fits) {
    if (is_grouped(p)) c->sched = SCHED_DP;
    if (!fits(*c) && c->sched != SCHED_DP && !c->swap && c->bn > 128) {
        Choice narrower = *c;  // half-width tiles halve the partial-tile footprint
        narrower.bn = 128;
        if (fits(narrower)) *c = narrower;
    }
    if (!fits(*c)) {
        if (forced) return false;
        c->sched = SCHED_DP;  // automatic choices fall back to no split
    }
    return true;
}

int dispatch_and_run(gemm_handle* h, const gemm_op_t* op, Problem& p, const gemm_workspace_t* ws, cudaStream_t st) {
    if (p.M == 0 || p.N == 0) {
        h->last_choice = "empty";
        return GEMM_OK;
    }
    if (p.K == 0) {  // no products: D = beta * C
        EpiParams e;
        memset(&e, 0, sizeof e);
        e.D = p.D;
        e.C = p.beta != 0.0f ? p.C : nullptr;
        e.ldd = p.ldd;
        e.ldc = p.ldc;
        e.d_bstride = p.d_bs;
        e.c_bstride = p.c_bs;
        e.M = p.M;
        e.N = p.N;
        e.alpha = p.alpha;
        e.beta = p.beta;
        e.d_type = p.d_type;
        e.flags = p.epi_flags;
        e.bias = p.bias;
        e.bias_type = p.bias_type;
        e.qscale = p.qscale;
        e.qzp = p.qzp;
        e.d_extent = out_extent(p.M, p.N, p.ldd, p.batches, p.d_bs);
        e.c_extent = e.C ? out_extent(p.M, p.N, p.ldc, p.batches, p.c_bs) : 0;
        e.status = h->status;
        h->last_choice = "scale_c";
        return launch_scale_c(e, p.batches, st) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }
    Choice c;
    bool have = forced_kernel(p, &c);
    if (have && !workspace_fits(h, p, c, ws)) return GEMM_ERR_WORKSPACE;
    const int forced_split = op->splitk > 1 ? op->splitk : h->force_splitk;
    const bool forced = forced_split > 1 || op->splitk == 1 || op->streamk != 0;
    const Key key = make_key(p);
    if (!have && !forced && op->dispatch != GEMM_DISPATCH_MEASURE) {
        auto it = h->cache.find(key);
        if (it != h->cache.end()) {
            c = it->second;
            have = workspace_fits(h, p, c, ws);
        }
    }
    // measuring synchronises the stream, which a stream capture forbids: a
    // measuring call on a capturing stream uses the cache or the heuristic
    bool measure_ok = op->dispatch == GEMM_DISPATCH_MEASURE;
    if (measure_ok) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
            cudaGetLastError();
            measure_ok = false;
        } else if (cs != cudaStreamCaptureStatusNone) {
            measure_ok = false;
        }
    }
    if (!have && !forced && op->dispatch == GEMM_DISPATCH_MEASURE && !measure_ok) {
        auto it = h->cache.find(key);
        if (it != h->cache.end()) {
            c = it->second;
            have = workspace_fits(h, p, c, ws);
        }
    }
    if (!have && !forced && measure_ok) {
        auto it = h->cache.find(key);
        if (it != h->cache.end() && workspace_fits(h, p, it->second, ws)) {
            c = it->second;
            have = true;
        } else if (!(p.beta != 0.0f && p.C == p.D)) {  // timing must not destroy an in-place C
            float best = -1.0f;
            for (const Choice& cand : candidates(p, h->sm_count)) {
                if (!workspace_fits(h, p, cand, ws)) continue;
                float us = measure(h, p, cand, ws, st);
                if (h->log) fprintf(stderr, "qgemm: measured %s: %.2f us\n", choice_name(p, cand).c_str(), us);
                if (us > 0 && (best < 0 || us < best)) {
                    best = us;
                    c = cand;
                    c.us = us;
                    have = true;
                }
            }
            if (have) h->cache[key] = c;
        }
    }
    if (!have) {
        c = heuristic(p, h->sm_count, ws && ws->partials ? ws->partials_size : 0, !forced);
        if (forced_split > 1) {
            c.sched = SCHED_SPLITK;
            c.splits = forced_split;
        } else if (op->streamk == 1) {
            c.sched = SCHED_STREAMK;
        } else if (op->splitk == 1 || op->streamk == -1) {
            if (c.sched != SCHED_DP && (op->splitk == 1 || c.sched == SCHED_STREAMK)) c.sched = SCHED_DP;
        }
        if (!settle_schedule(p, &c, forced, [&](const Choice& x) { return workspace_fits(h, p, x, ws); }))
            return GEMM_ERR_WORKSPACE;
    }
    h->last_choice = choice_name(p, c);
    if (h->log)
        fprintf(stderr, "qgemm: M=%lld N=%lld K=%lld batches=%d -> %s\n", (long long)p.M, (long long)p.N,
                (long long)p.K, p.batches, h->last_choice.c_str());
    int rc = launch_choice(h, p, c, ws, st);
    if (rc == GEMM_ERR_CUDA) cudaGetLastError();
    return rc;
}

// Shared validation of gemm_run / gemm_run_grouped.
int build_problem(gemm_handle* h, const gemm_op_t* op, float alpha, const void* A, const gemm_layout_t* Adesc,
                  const void* U, const gemm_layout_t* Udesc, const void* B, const gemm_layout_t* Bdesc,
                  const void* V, const gemm_layout_t* Vdesc, float beta, const void* C, const gemm_layout_t* Cdesc,
                  void* D, const gemm_layout_t* Ddesc, bool grouped, Problem* out) {
    if (!h || !op || !Adesc || !Bdesc || !Ddesc) return GEMM_ERR_INVALID_ARG;
    // fused epilogue: known flags only, ReLU and GELU exclusive, a bias of a
    // float type aligned to its element when the bias flag is set
    if (op->epilogue & ~(GEMM_EPILOGUE_BIAS | GEMM_EPILOGUE_RELU | GEMM_EPILOGUE_GELU)) return GEMM_ERR_INVALID_ARG;
    if ((op->epilogue & GEMM_EPILOGUE_RELU) && (op->epilogue & GEMM_EPILOGUE_GELU)) return GEMM_ERR_INVALID_ARG;
    if (op->epilogue & GEMM_EPILOGUE_BIAS) {
        if (!op->bias) return GEMM_ERR_INVALID_ARG;
        if (op->bias_type != GEMM_F32 && op->bias_type != GEMM_F16 && op->bias_type != GEMM_BF16)
            return GEMM_ERR_UNSUPPORTED;
        const uintptr_t align = op->bias_type == GEMM_F32 ? 4 : 2;
        if (reinterpret_cast<uintptr_t>(op->bias) % align) return GEMM_ERR_INVALID_ARG;
        if (!device_pointer(h, op->bias)) return GEMM_ERR_INVALID_ARG;
    }
    if (op->dispatch < GEMM_DISPATCH_DEFAULT || op->dispatch > GEMM_DISPATCH_REUSE) return GEMM_ERR_INVALID_ARG;
    if (op->splitk < 0 || op->streamk < -1 || op->streamk > 1) return GEMM_ERR_INVALID_ARG;
    if (op->splitk > 1 && op->streamk == 1) return GEMM_ERR_INVALID_ARG;
    Problem p;
    memset(&p, 0, sizeof p);
    p.M = Adesc->rows;
    p.K = Adesc->cols;
    p.N = Bdesc->cols;
    if (p.M < 0 || p.N < 0 || p.K < 0) return GEMM_ERR_INVALID_ARG;
    if (p.M > INT32_MAX || p.N > INT32_MAX || p.K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    p.a_type = Adesc->type;
    p.b_type = Bdesc->type;
    p.d_type = Ddesc->type;
    // A and B: both f16, both bf16, both E4M3 or both E5M2; or 16-bit A with int4 B
    if (!is16(p.a_type) && !is_f8(p.a_type)) return GEMM_ERR_UNSUPPORTED;
    if (!(p.b_type == p.a_type || (p.b_type == GEMM_S4 && is16(p.a_type)))) return GEMM_ERR_UNSUPPORTED;
    p.kstep = (int32_t)(128 / in_bytes(p.a_type));
    if (!is_float_out(p.d_type) && p.d_type != GEMM_S8) return GEMM_ERR_UNSUPPORTED;
    int rc;
    if ((rc = check_layout(Adesc, GEMM_ROW_MAJOR, p.M, p.K))) return rc;
    if ((rc = check_layout(Bdesc, GEMM_COL_MAJOR, p.K, p.N))) return rc;
    if ((rc = check_layout(Ddesc, GEMM_ROW_MAJOR, p.M, p.N))) return rc;
    p.alpha = alpha;
    p.beta = beta;
    p.epi_flags = op->epilogue;
    if (p.d_type == GEMM_S8) {
        // output quantisation: per-row fp32 scales on the device; C is not read
        if (beta != 0.0f || Ddesc->num != 1) return GEMM_ERR_UNSUPPORTED;
        if (!op->out_scale || (reinterpret_cast<uintptr_t>(op->out_scale) & 3)) return GEMM_ERR_INVALID_ARG;
        if (p.M > 0 && !device_pointer(h, op->out_scale)) return GEMM_ERR_INVALID_ARG;
        p.qscale = op->out_scale;
        p.qzp = op->out_zero_point;
    }
    p.bias = (op->epilogue & GEMM_EPILOGUE_BIAS) ? op->bias : nullptr;
    p.bias_type = op->bias_type;
    p.A = A;
    p.lda = Adesc->ld;
    p.a_bs = Adesc->batch_stride;
    p.B = B;
    p.ldb = Bdesc->ld;
    p.b_bs = Bdesc->batch_stride;
    p.D = D;
    p.ldd = Ddesc->ld;
    p.d_bs = Ddesc->batch_stride;
    p.batches = Adesc->num;
    if (beta != 0.0f) {
        if (!C || !Cdesc) return GEMM_ERR_INVALID_ARG;
        if ((rc = check_layout(Cdesc, GEMM_ROW_MAJOR, p.M, p.N))) return rc;
        if (Cdesc->type != p.d_type) return GEMM_ERR_UNSUPPORTED;
        if (!grouped && Cdesc->num != p.batches) return GEMM_ERR_INVALID_ARG;
        p.C = C;
        p.ldc = Cdesc->ld;
        p.c_bs = Cdesc->batch_stride;
    }
    // scale operands: NULL means unscaled
    if (U) {
        if (!Udesc || op->quant_a_group <= 0) return GEMM_ERR_INVALID_ARG;
        p.ga = op->quant_a_group;
        if (p.ga < 8 || p.K % p.ga || (p.ga % 64 && 64 % p.ga)) return GEMM_ERR_INVALID_ARG;
        if (!is16(Udesc->type)) return GEMM_ERR_UNSUPPORTED;
        if ((rc = check_layout(Udesc, GEMM_ROW_MAJOR, p.K / p.ga, p.M))) return rc;
        if (Udesc->num != 1) return GEMM_ERR_UNSUPPORTED;
        if (!aligned16(U) || (Udesc->ld * 2) % 16) return GEMM_ERR_INVALID_ARG;  // copied by TMA
        p.U = U;
        p.ldu = Udesc->ld;
        p.u_type = Udesc->type;
    }
    if (V) {
        if (!Vdesc || op->quant_b_group <= 0) return GEMM_ERR_INVALID_ARG;
        p.gb = op->quant_b_group;
        if (p.gb < 8 || p.K % p.gb || (p.gb % 64 && 64 % p.gb)) return GEMM_ERR_INVALID_ARG;
        if (!is16(Vdesc->type)) return GEMM_ERR_UNSUPPORTED;
        if ((rc = check_layout(Vdesc, GEMM_ROW_MAJOR, p.K / p.gb, p.N))) return rc;
        // grouped problems: one V per expert (as many as B has matrices)
        if (Vdesc->num != (grouped ? Bdesc->num : 1)) return grouped ? GEMM_ERR_INVALID_ARG : GEMM_ERR_UNSUPPORTED;
        if (!aligned16(V) || (Vdesc->ld * 2) % 16) return GEMM_ERR_INVALID_ARG;  // copied by TMA
        if (Vdesc->num > 1 && (Vdesc->batch_stride < (p.K / p.gb) * Vdesc->ld || (Vdesc->batch_stride * 2) % 16))
            return GEMM_ERR_INVALID_ARG;
        p.V = V;
        p.ldv = Vdesc->ld;
        p.v_bs = Vdesc->num > 1 ? Vdesc->batch_stride : 0;
        p.v_type = Vdesc->type;
    }
    if (op->b_zero) {
        // zero points of an int4 B with V: (K/gb) x N bytes per expert, copied by TMA
        if (!p.V || p.b_type != GEMM_S4) return GEMM_ERR_INVALID_ARG;
        if (!aligned16(op->b_zero) || op->b_zero_ld < p.N || op->b_zero_ld % 16) return GEMM_ERR_INVALID_ARG;
        const int64_t nz = grouped ? Bdesc->num : 1;
        if (nz > 1 && (op->b_zero_batch_stride < (p.K / p.gb) * op->b_zero_ld || op->b_zero_batch_stride % 16))
            return GEMM_ERR_INVALID_ARG;
        if (p.N > 0 && p.K > 0 && !device_pointer(h, op->b_zero)) return GEMM_ERR_INVALID_ARG;
        p.Z = op->b_zero;
        p.ldz = op->b_zero_ld;
        p.z_bs = nz > 1 ? op->b_zero_batch_stride : 0;
    }
    p.family = (p.U || p.V || p.b_type == GEMM_S4) ? FAM_DQ : FAM_DENSE;
    if (is_f8(p.a_type) && p.family != FAM_DENSE) return GEMM_ERR_UNSUPPORTED;  // no U/V on 8-bit operands
    if (grouped) {
        if (Adesc->num != 1 || Ddesc->num != 1) return GEMM_ERR_INVALID_ARG;
        p.family = p.family == FAM_DQ ? FAM_GROUPED_DQ : FAM_GROUPED;
        p.batches = 1;
    } else {
        if (Bdesc->num != p.batches || Ddesc->num != p.batches) return GEMM_ERR_INVALID_ARG;
        if (p.batches > 1 && (p.U || p.V || p.b_type == GEMM_S4)) return GEMM_ERR_UNSUPPORTED;
        if (p.batches > 1) {
            if (p.a_bs < p.M * p.lda || p.b_bs < p.N * p.ldb || p.d_bs < p.M * p.ldd) return GEMM_ERR_INVALID_ARG;
            if (p.C && p.c_bs < 0) return GEMM_ERR_INVALID_ARG;
        }
    }
    if (p.M == 0 || p.N == 0) {
        *out = p;
        return GEMM_OK;
    }
    if (!D || (p.K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
    if (p.K > 0) {
        // operands read by the tensor-memory accelerator
        if (!aligned16(A) || !aligned16(B)) return GEMM_ERR_INVALID_ARG;
        const int64_t es = in_bytes(p.a_type);
        if ((p.lda * es) % 16 || (p.a_bs * es) % 16) return GEMM_ERR_INVALID_ARG;
        if (p.b_type == GEMM_S4) {
            if (p.K % 2 || p.ldb % 32 || p.b_bs % 32) return GEMM_ERR_INVALID_ARG;
        } else if ((p.ldb * es) % 16 || (p.b_bs * es) % 16) {
            return GEMM_ERR_INVALID_ARG;
        }
        if (!device_pointer(h, A) || !device_pointer(h, B)) return GEMM_ERR_INVALID_ARG;
    }
    if (!device_pointer(h, D)) return GEMM_ERR_INVALID_ARG;
    if (p.C && !device_pointer(h, p.C)) return GEMM_ERR_INVALID_ARG;
    *out = p;
    return GEMM_OK;
}

int bind_device(gemm_handle* h) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (cur != h->device && cudaSetDevice(h->device) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm_run(gemm_handle_t h, const gemm_op_t* op, float alpha, const void* A, const gemm_layout_t* Adesc,
             const void* U, const gemm_layout_t* Udesc, const void* B, const gemm_layout_t* Bdesc, const void* V,
             const gemm_layout_t* Vdesc, float beta, const void* C, const gemm_layout_t* Cdesc, void* D,
             const gemm_layout_t* Ddesc, const gemm_workspace_t* workspace, gemm_stream_t stream) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    int rc = bind_device(h);
    if (rc) return rc;
    Problem p;
    rc = build_problem(h, op, alpha, A, Adesc, U, Udesc, B, Bdesc, V, Vdesc, beta, C, Cdesc, D, Ddesc, false, &p);
    if (rc) return rc;
    return dispatch_and_run(h, op, p, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int gemm_run_grouped(gemm_handle_t h, const gemm_op_t* op, float alpha, const void* A, const gemm_layout_t* Adesc,
                     const void* U, const gemm_layout_t* Udesc, const void* B, const gemm_layout_t* Bdesc,
                     const void* V, const gemm_layout_t* Vdesc, float beta, const void* C,
                     const gemm_layout_t* Cdesc, void* D, const gemm_layout_t* Ddesc,
                     const int32_t* expert_offsets_dev, int32_t num_experts, const gemm_workspace_t* workspace,
                     gemm_stream_t stream) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    int rc = bind_device(h);
    if (rc) return rc;
    if (num_experts < 1 || num_experts > 4096 || !expert_offsets_dev || !Bdesc || Bdesc->num != num_experts)
        return GEMM_ERR_INVALID_ARG;
    if (num_experts > 1 && Bdesc->batch_stride < Bdesc->cols * Bdesc->ld) return GEMM_ERR_INVALID_ARG;
    Problem p;
    rc = build_problem(h, op, alpha, A, Adesc, U, Udesc, B, Bdesc, V, Vdesc, beta, C, Cdesc, D, Ddesc, true, &p);
    if (rc) return rc;
    if (!device_pointer(h, expert_offsets_dev) || (reinterpret_cast<uintptr_t>(expert_offsets_dev) & 3u))
        return GEMM_ERR_INVALID_ARG;
    p.offsets = expert_offsets_dev;
    p.num_experts = num_experts;
    return dispatch_and_run(h, op, p, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int gemm_export(gemm_handle_t h, void* buf, size_t cap, size_t* written) {
    if (!h || !written) return GEMM_ERR_INVALID_ARG;
    const std::string s = cache_serialize(h->cache, h->name, h->sm_count, h->cc);
    *written = s.size();
    if (!buf) return GEMM_OK;
    if (cap < s.size()) return GEMM_ERR_INVALID_ARG;
    memcpy(buf, s.data(), s.size());
    return GEMM_OK;
}

int gemm_import(gemm_handle_t h, const void* buf, size_t size) {
    if (!h || (!buf && size)) return GEMM_ERR_INVALID_ARG;
    std::string s(static_cast<const char*>(buf), size);
    std::map<Key, Choice> merged = h->cache;
    if (!cache_parse(s, h->name, h->sm_count, h->cc, &merged)) return GEMM_ERR_BAD_CACHE;
    h->cache.swap(merged);
    return GEMM_OK;
}

int gemm_get_tuning_seq(gemm_handle_t h, int32_t* out, int32_t cap, int32_t* n) {
    if (!h || !n || cap < 0) return GEMM_ERR_INVALID_ARG;
    const auto& seq = tuning_seq();
    *n = (int32_t)seq.size();
    if (out)
        for (int32_t i = 0; i < cap && i < (int32_t)seq.size(); ++i) out[i] = seq[i];
    return GEMM_OK;
}

int gemm_cache_size(gemm_handle_t h, int32_t* n) {
    if (!h || !n) return GEMM_ERR_INVALID_ARG;
    *n = (int32_t)h->cache.size();
    return GEMM_OK;
}

int gemm_checked_build(void) { return kDeviceChecksHost ? 1 : 0; }

int gemm_device_status(gemm_handle_t h, gemm_stream_t stream) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    int rc = bind_device(h);
    if (rc) return rc;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    uint32_t st[4] = {0, 0, 0, 0};
    if (cudaMemcpy(st, h->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (st[0] == 0) return GEMM_OK;
    if (h->log)
        fprintf(stderr, "qgemm: device %s (site %u, block %u, count %u)\n",
                (st[0] & 2u) ? "bounds check failed" : "wait gave up", st[1], st[2], st[3]);
    if (cudaMemset(h->status, 0, sizeof st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return (st[0] & 2u) ? GEMM_ERR_DEVICE_CHECK : GEMM_ERR_DEVICE_TIMEOUT;
}

int gemm_selftest_wait_timeout(gemm_handle_t h, uint64_t timeout_ns, gemm_stream_t stream) {
    if (!h || timeout_ns == 0 || timeout_ns > 10000000000ull) return GEMM_ERR_INVALID_ARG;
    int rc = bind_device(h);
    if (rc) return rc;
    if (launch_wait_selftest(h->status, timeout_ns, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return gemm_device_status(h, stream);
}

const char* gemm_last_choice(gemm_handle_t h) { return h ? h->last_choice.c_str() : "none"; }

int gemm_plan_streamk(int64_t m, int64_t n, int64_t k, int32_t block_m, int32_t block_n, int32_t block_k,
                      int32_t total_sm, int64_t out[7]) {
    if (!out || m < 0 || n < 0 || k < 0 || block_m <= 0 || block_n <= 0 || block_k <= 0 || total_sm <= 0)
        return GEMM_ERR_INVALID_ARG;
    StreamKPlan p = streamk_plan(m, n, k, block_m, block_n, block_k, total_sm);
    out[0] = p.iters_per_tile;
    out[1] = p.total_tiles;
    out[2] = p.streamk_tiles;
    out[3] = p.blocking_tiles;
    out[4] = p.full_tiles;
    out[5] = p.partial_tiles;
    out[6] = p.sm_partition_factor;
    return GEMM_OK;
}

int gemm_heuristic_choice(int64_t m, int64_t n, int64_t k, int32_t a_type, int32_t b_type, int32_t d_type,
                          int32_t quant_a_group, int32_t quant_b_group, int32_t num_experts, int32_t sm_count,
                          size_t partials_size, char* out, size_t cap) {
    if (!out || cap == 0 || m < 1 || n < 1 || k < 1 || sm_count < 1 || num_experts < 0) return GEMM_ERR_INVALID_ARG;
    if ((!is16(a_type) && !is_f8(a_type)) || !(b_type == a_type || (b_type == GEMM_S4 && is16(a_type))))
        return GEMM_ERR_INVALID_ARG;
    if (!is_float_out(d_type) && d_type != GEMM_S8) return GEMM_ERR_INVALID_ARG;
    Problem p;
    memset(&p, 0, sizeof p);
    p.M = m;
    p.N = n;
    p.K = k;
    p.a_type = a_type;
    p.b_type = b_type;
    p.d_type = d_type;
    p.kstep = (int32_t)(128 / in_bytes(a_type));
    p.batches = 1;
    if (is_f8(a_type) && (quant_a_group > 0 || quant_b_group > 0)) return GEMM_ERR_INVALID_ARG;
    // the heuristic only asks whether scales are present: a marker stands in
    static const int32_t marker = 0;
    if (quant_a_group > 0) {
        p.U = &marker;
        p.ga = quant_a_group;
    }
    if (quant_b_group > 0) {
        p.V = &marker;
        p.gb = quant_b_group;
    }
    p.family = (p.U || p.V || b_type == GEMM_S4) ? FAM_DQ : FAM_DENSE;
    if (num_experts > 0) {
        p.family = p.family == FAM_DQ ? FAM_GROUPED_DQ : FAM_GROUPED;
        p.num_experts = num_experts;
    }
    Choice c = heuristic(p, sm_count, partials_size);
    // the automatic fallbacks of dispatch_and_run, against a workspace of
    // partials_size bytes of partials and a barrier buffer of the usual size
    // (on this path every program count is sm_count)
    settle_schedule(p, &c, false, [&](const Choice& x) {
        if (x.gemv) return true;
        const SchedParams sp = make_sched(p, x, sm_count);
        return partials_bytes_needed(sp, x.bn, x.pair) <= partials_size &&
               counters_bytes_needed(sp, x.pair) <= GEMM_BARRIERS_SIZE;
    });
    const std::string name = choice_name(p, c);
    if (name.size() + 1 > cap) return GEMM_ERR_INVALID_ARG;
    memcpy(out, name.c_str(), name.size() + 1);
    return GEMM_OK;
}

int gemm_grouped_block(const int32_t* sizes, int32_t num_experts, int32_t block_m, int64_t block,
                       int64_t out[3]) {
    if (!sizes || !out || num_experts < 1 || block_m <= 0 || block < 0) return GEMM_ERR_INVALID_ARG;
    std::vector<int32_t> off(num_experts + 1, 0);
    for (int32_t e = 0; e < num_experts; ++e) {
        if (sizes[e] < 0) return GEMM_ERR_INVALID_ARG;
        off[e + 1] = off[e] + sizes[e];
    }
    int32_t ex, rows;
    int64_t m0;
    grouped_block(off.data(), num_experts, block_m, block, &ex, &m0, &rows);
    out[0] = ex;
    out[1] = m0;
    out[2] = rows;
    return GEMM_OK;
}

}  // extern "C"
