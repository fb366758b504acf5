/*
 * gemm.h -- C ABI of the GB300 (sm_103a) quantized GEMM library.
 *
 * The library computes
 *
 *     D = alpha * (A-hat @ B-hat) + beta * C
 *
 * with fp16/bf16 operands and fp32 accumulation, where A-hat / B-hat are the
 * operands after optional group-wise scaling by U / V (the "quantization scale
 * operands" that advance at K-group boundaries) and B may be int4.  This is the
 * interface of "InternLM Lmdeploy Gemm Interface" (sections Description,
 * Signature, I/O Contract, Usage Examples): one handle per device that owns a
 * kernel registry, a dispatch cache, a problem analyser and a measurer; a Run
 * call taking every operand with a layout; Export/Import of the dispatch
 * cache; GetTuningSeq.
 *
 * Conventions for every function below:
 *  - The return value is a gemm_status_t; 0 (GEMM_OK) means success.  Nothing
 *    aborts, throws or exits across this ABI.
 *  - All pointers are owned by the caller.  The library never allocates device
 *    memory inside gemm_run / gemm_run_grouped; scratch comes from the caller's
 *    workspace.
 *  - Calls that take a stream are asynchronous on that stream (a CUDA stream
 *    handle; NULL is the legacy default stream).  Errors found on the host are
 *    returned before anything is enqueued.
 *  - A handle is bound to the CUDA device that was current when it was
 *    created.  It is not thread-safe: do not run and import concurrently on one
 *    handle.
 */
#ifndef QGEMM_GEMM_H_
#define QGEMM_GEMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ----------------------------------------------------------- */
typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,    /* null required pointer, bad size/ld, misalignment,
                                    K not a multiple of a group size, ...          */
    GEMM_ERR_UNSUPPORTED = 2,    /* dtype/order combination or device not served   */
    GEMM_ERR_WORKSPACE = 3,      /* partials or barrier buffer too small / missing  */
    GEMM_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed               */
    GEMM_ERR_NO_KERNEL = 5,      /* no registered kernel accepts the problem        */
    GEMM_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up on a bounded wait             */
    GEMM_ERR_BAD_CACHE = 7,      /* import blob malformed, wrong version or device  */
    GEMM_ERR_DEVICE_CHECK = 8    /* a device-side bounds check failed (checked build) */
} gemm_status_t;

/* ---- operand description ------------------------------------------------------ */
typedef enum {
    GEMM_F32 = 0, GEMM_F16 = 1, GEMM_BF16 = 2,
    GEMM_S4 = 3,                /* two's-complement nibbles, two per byte        */
    GEMM_S8 = 4,                /* int8 (quantised D)                           */
    GEMM_E4M3 = 5, GEMM_E5M2 = 6 /* 8-bit floats (1-4-3 bias 7, no infinity; 1-5-2 bias 15) */
} gemm_dtype_t;
typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_order_t;

/*
 * MatrixLayout.  A logical rows x cols matrix:
 *   row-major: element (r, c) at r*ld + c;  col-major: at c*ld + r.
 * ld and batch_stride count elements (for GEMM_S4, 4-bit elements, so a
 * col-major int4 B with ld = K has K/2 bytes per column).  num > 1 describes
 * num matrices batch_stride elements apart (batched GEMM, or the experts of a
 * grouped GEMM).
 *
 * Operands served (anything else returns GEMM_ERR_UNSUPPORTED):
 *   A : M x K, row-major, f16/bf16/e4m3/e5m2        (K contiguous)
 *   B : K x N, col-major, same type as A, or S4 with a 16-bit A (K contiguous)
 *   U : (K/ga) x M, row-major, f16/bf16            scale of A per (row, K-group)
 *   V : (K/gb) x N, row-major, f16/bf16            scale of B per (K-group, column)
 *   C : M x N, row-major, same type as D
 *   D : M x N, row-major, f32/f16/bf16
 * 8-bit float operands (the FP8 inputs of the DeepGEMM kernel-set blog,
 * sections 1.2 and 6.3) take no U/V: a per-tensor scale goes into alpha.
 * A, B, U and V base addresses must be 16-byte aligned and their ld a
 * multiple of 16 bytes (they are read by the tensor-memory accelerator); C
 * and D may have any ld >= N and element alignment (16-byte aligned ones are
 * moved through shared memory by TMA, others element by element).
 */
typedef struct {
    int32_t type;          /* gemm_dtype_t  */
    int32_t order;         /* gemm_order_t  */
    int64_t rows, cols;
    int64_t ld;
    int32_t num;           /* >= 1 */
    int64_t batch_stride;  /* elements; used when num > 1 */
} gemm_layout_t;

/* Dispatch policies for gemm_op_t.dispatch. */
enum {
    GEMM_DISPATCH_DEFAULT = 0, /* cache hit, else the heuristic                   */
    GEMM_DISPATCH_MEASURE = 1, /* on a miss, time the candidates on the stream
                                  (synchronises it) and store the winner; on a
                                  stream that is being captured nothing is
                                  timed: the cache, else the heuristic         */
    GEMM_DISPATCH_REUSE = 2    /* cache only (no measuring), else the heuristic   */
};

/*
 * Epilogue flags for gemm_op_t.epilogue: the fused bias + activation of the
 * DeepGEMM kernel-set blog, section 6.1 (bias, then ReLU or GELU, applied in
 * the epilogue that writes D).  With x = alpha * acc + beta * c (fp32):
 *   GEMM_EPILOGUE_BIAS  x += bias[j] (one value per output column j, shared by
 *                       every row, batch and expert);
 *   GEMM_EPILOGUE_RELU  x = x < 0 ? 0 : x (NaN stays NaN);
 *   GEMM_EPILOGUE_GELU  x = x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), the exact
 *                       (erf) form;
 * then D = RN_D(x).  RELU and GELU exclude each other; 0 is the plain
 * alpha/beta/cast epilogue.
 */
enum {
    GEMM_EPILOGUE_DEFAULT = 0,
    GEMM_EPILOGUE_BIAS = 1,
    GEMM_EPILOGUE_RELU = 2,
    GEMM_EPILOGUE_GELU = 4
};

/*
 * Output quantisation (DeepGEMM kernel-set blog, section 6.2): a D of type
 * GEMM_S8 receives y = round(x * out_scale[i] + zp) for row i, where x is the
 * fp32 value the epilogue would otherwise round to D (after alpha/beta and the
 * fused bias / activation).  The product-plus-offset is one fp32 fma, the
 * rounding is to nearest-even and the result saturates to [-128, 127] (NaN
 * gives 0).  It
 * needs beta == 0 (C is not read) and one batch; grouped problems index the
 * scales by D's row (token).
 */

/*
 * Operation: "dispatch policy, epilogue, quantization config" (Gemm Interface,
 * I/O Contract).
 */
typedef struct {
    int32_t dispatch;      /* GEMM_DISPATCH_*                                        */
    int32_t epilogue;      /* GEMM_EPILOGUE_* flags (0: alpha/beta/cast)              */
    int32_t quant_a_group; /* 0: no U; else U's group size along K: 8, 16, 32 or a multiple of 64 */
    int32_t quant_b_group; /* 0: no V; else V's group size along K: 8, 16, 32 or a multiple of 64 */
    int32_t splitk;        /* 0: automatic; 1: unsplit; S > 1: force S K-slices       */
    int32_t streamk;       /* 0: automatic; 1: force stream-K; -1: never stream-K     */
    const void* bias;      /* GEMM_EPILOGUE_BIAS: N contiguous values on the device,
                              aligned to their element size, owned by the caller;
                              ignored otherwise                                       */
    int32_t bias_type;     /* GEMM_F32 / GEMM_F16 / GEMM_BF16                         */
    int32_t out_zero_point;/* GEMM_S8 D: the zero point zp                           */
    const float* out_scale;/* GEMM_S8 D: M fp32 scales on the device, one per row of D
                              (per token); ignored for other D types                  */
    /* Asymmetric int4 B (zero points advance at K-group boundaries with V, as
     * the scale operands of "InternLM Lmdeploy Gemm MainloopSm80V2", section
     * Description, do): B-hat[k][j] = RN_A((q[k][j] - z[k/gb][j]) * V[k/gb][j]).
     * z is a 4-bit two's-complement zero point in [-8, 7] stored one per byte
     * (the byte's low nibble; its high nibble is ignored), in a (K/gb) x N
     * row-major byte matrix on the device.  NULL means symmetric (z = 0).
     * Needs an int4 B with V; b_zero 16-byte aligned, b_zero_ld (bytes between
     * rows, >= N) a multiple of 16; grouped problems give one matrix per expert,
     * b_zero_batch_stride bytes apart (a multiple of 16).                     */
    const void* b_zero;
    int64_t b_zero_ld;
    int64_t b_zero_batch_stride;
} gemm_op_t;

/*
 * Workspace (Gemm Interface, Description: kBarriersSize for split-K barriers
 * and kPartialsSize for partial results).  barriers: one int32 arrival counter
 * per output tile; it must be zeroed once by the caller (cudaMemsetAsync) and
 * the library leaves it zeroed after every call.  partials: fp32 partial tiles.
 * Either may be NULL for calls that do not split K; calls that do need them
 * return GEMM_ERR_WORKSPACE when they are missing or too small.  Concurrent
 * calls (other streams) must not share a workspace.
 */
typedef struct {
    void* barriers;
    size_t barriers_size;
    void* partials;
    size_t partials_size;
} gemm_workspace_t;

#define GEMM_BARRIERS_SIZE ((size_t)1 << 20) /* kBarriersSize: 1 MB  */
#define GEMM_PARTIALS_SIZE ((size_t)32 << 20) /* kPartialsSize: 32 MB */

typedef struct gemm_handle* gemm_handle_t;
typedef struct CUstream_st* gemm_stream_t; /* identical to cudaStream_t */

/* Gemm() / ~Gemm(): bind to the current device (compute capability 10.3),
 * build the kernel registry.  UNSUPPORTED on another device, CUDA when no
 * device is usable. */
int gemm_create(gemm_handle_t* out);
int gemm_destroy(gemm_handle_t h);

/*
 * Gemm::Run.  D = alpha * (A-hat @ B-hat) + beta * C.
 * With fp16/bf16 or E4M3/E5M2 operands every product is exact in fp32.
 *   A-hat[i][k] = A[i][k], or RN_A(A[i][k] * U[k/ga][i]) with U;
 *   B-hat[k][j] = B[k][j], or RN_B(B[k][j] * V[k/gb][j]) with V;
 *   int4 B: B-hat[k][j] = RN_A(q[k][j] * V[k/gb][j]) (q without V), where q
 *   is the two's-complement nibble: column j holds k = 2t in bits 3:0 and
 *   k = 2t+1 in bits 7:4 of byte t.
 * Accumulation is fp32; the epilogue forms fma(alpha, acc, beta*c) in fp32 and
 * rounds once (nearest-even) to D's type.  C is not read when beta == 0 and
 * may then be NULL (Usage Examples passes nullptr with beta 0).  U/V NULL
 * means unscaled.  num > 1 on A, B, C, D runs a batched GEMM.
 * M, N or K of 0 is allowed (K == 0 gives D = beta*C).
 */
int gemm_run(gemm_handle_t h, const gemm_op_t* op, float alpha,
             const void* A, const gemm_layout_t* Adesc,
             const void* U, const gemm_layout_t* Udesc,
             const void* B, const gemm_layout_t* Bdesc,
             const void* V, const gemm_layout_t* Vdesc,
             float beta,
             const void* C, const gemm_layout_t* Cdesc,
             void* D, const gemm_layout_t* Ddesc,
             const gemm_workspace_t* workspace, gemm_stream_t stream);

/*
 * gemm_run without a workspace argument, for callers that cannot allocate
 * device memory: for example a plug-in inside a host framework whose caching
 * allocator owns all device memory and hands out no scratch, or code on a
 * latency-critical path where an allocation would synchronise the device.
 * The pages have no counterpart to this entry point.
 *   - Scratch for split-K / stream-K comes from a fixed array in the library's
 *     own device memory: 64 KB of tile counters and 8 MB of fp32 partials
 *     (GEMM_NOALLOC_BARRIERS_SIZE / GEMM_NOALLOC_PARTIALS_SIZE).  Every GPU
 *     that loads the library holds it until the process exits.
 *   - A problem whose chosen or forced schedule needs more scratch than that is
 *     rejected with GEMM_ERR_WORKSPACE (automatic choices fall back to an
 *     unsplit schedule instead).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Each call clears the counters on `stream` (cudaMemsetAsync) and then
 *     behaves as gemm_run.  It calls no cudaMalloc / cudaFree.
 *   - All calls share the one array: calls that may overlap on the GPU (other
 *     streams, other threads) race and must be serialised by the caller.
 */
#define GEMM_NOALLOC_BARRIERS_SIZE ((size_t)64 << 10)
#define GEMM_NOALLOC_PARTIALS_SIZE ((size_t)8 << 20)
int gemm_run_noalloc(gemm_handle_t h, const gemm_op_t* op, float alpha,
                     const void* A, const gemm_layout_t* Adesc,
                     const void* U, const gemm_layout_t* Udesc,
                     const void* B, const gemm_layout_t* Bdesc,
                     const void* V, const gemm_layout_t* Vdesc,
                     float beta,
                     const void* C, const gemm_layout_t* Cdesc,
                     void* D, const gemm_layout_t* Ddesc,
                     gemm_stream_t stream);

/*
 * Grouped (MoE) GEMM, after the grouped GEMM of the TileLang tutorial
 * "gemm_variants.py" (section gemm_grouped): the rows of A are sorted by
 * expert, expert e owning rows expert_offsets[e] .. expert_offsets[e+1]-1, and
 * D[those rows] = alpha * A[those rows] @ B_e + beta * C[those rows].
 *   A : (sum m_e) x K row-major;  B : num = num_experts matrices K x N,
 *   col-major, batch_stride apart;  C, D : (sum m_e) x N row-major.
 *   expert_offsets_dev: DEVICE int32[num_experts + 1], prefix sums starting at
 *   0 and ending at Adesc->rows; read on the device only (no host sync).
 *   Experts with zero rows are allowed.
 *   U (optional): (K/ga) x (sum m_e) row-major, one scale per token row and
 *   K-group, num = 1.  V (optional, and the zero points of gemm_op_t):
 *   num = num_experts matrices (K/gb) x N, batch_stride apart, one per expert
 *   (a W4A16 mixture of experts with an int4 B).
 */
int gemm_run_grouped(gemm_handle_t h, const gemm_op_t* op, float alpha,
                     const void* A, const gemm_layout_t* Adesc,
                     const void* U, const gemm_layout_t* Udesc,
                     const void* B, const gemm_layout_t* Bdesc,
                     const void* V, const gemm_layout_t* Vdesc,
                     float beta,
                     const void* C, const gemm_layout_t* Cdesc,
                     void* D, const gemm_layout_t* Ddesc,
                     const int32_t* expert_offsets_dev, int32_t num_experts,
                     const gemm_workspace_t* workspace, gemm_stream_t stream);

/*
 * Gemm::Export / Gemm::Import of the dispatch cache.  Export with buf == NULL
 * (or cap too small) stores the needed size in *written and returns GEMM_OK
 * (respectively GEMM_ERR_INVALID_ARG).  Import merges the entries of a blob
 * made by Export on a device with the same name and SM count; any other blob
 * (including one of an older format version: this library writes version 3)
 * returns GEMM_ERR_BAD_CACHE and leaves the cache unchanged.
 */
int gemm_export(gemm_handle_t h, void* buf, size_t cap, size_t* written);
int gemm_import(gemm_handle_t h, const void* buf, size_t size);

/* Gemm::GetTuningSeq: the ascending M values (batch sizes) the dispatch cache
 * is keyed on; a problem uses the smallest entry >= M.  *n receives the
 * length; at most cap values are written to out (out may be NULL). */
int gemm_get_tuning_seq(gemm_handle_t h, int32_t* out, int32_t cap, int32_t* n);

/* Number of cache entries (for tests and tooling). */
int gemm_cache_size(gemm_handle_t h, int32_t* n);

/* Text of a status code (static storage). */
const char* gemm_status_string(int status);

/*
 * Device-side status: synchronises `stream`, then returns GEMM_OK,
 * GEMM_ERR_DEVICE_TIMEOUT if any kernel of this library on this device gave
 * up on a bounded wait since the last call, or GEMM_ERR_DEVICE_CHECK if (in
 * the checked build) a device-side bounds check failed; it clears the record.
 * The kernels never trap: a wait that runs out, or an access a check refuses,
 * is recorded here, the access is skipped and D is left undefined.
 */
int gemm_device_status(gemm_handle_t h, gemm_stream_t stream);

/*
 * 1 when this library is the checked debug build (compiled with
 * QG_DEVICE_CHECKS, libqgemm_checked.so), else 0.  In that build every work
 * unit's tile coordinates, K range, partial slots and tile counter are checked
 * against the problem and the workspace sizes, and every element the register
 * epilogue reads or writes against C's / D's extent, before the access; a
 * failed check is reported by gemm_device_status.  The checks stand in for a
 * memory checker on machines where none can run.
 */
int gemm_checked_build(void);

/*
 * Self-test of the device-side failure detection: launches one tiny kernel
 * whose single thread waits on an mbarrier that nothing ever completes, with
 * a bound of timeout_ns (1 ns .. 10 s).  The wait runs out, the kernel records
 * it and returns, and this call returns the result of gemm_device_status --
 * GEMM_ERR_DEVICE_TIMEOUT when the mechanism works.  Nothing faults or traps.
 */
int gemm_selftest_wait_timeout(gemm_handle_t h, uint64_t timeout_ns, gemm_stream_t stream);

/* The kernel chosen for the last gemm_run / gemm_run_grouped on this handle,
 * as a short text ("umma_bn256/dp", "umma_bn16_swap/streamk", ...). */
const char* gemm_last_choice(gemm_handle_t h);

/*
 * Host-only planners, exposed so their integers can be checked bit-exactly.
 *
 * gemm_plan_streamk: the stream-K sizing of the TileLang tutorial
 * "gemm_variants.py" (section streamk_plan) for an m x n x k problem cut into
 * block_m x block_n x block_k steps over total_sm programs.  out[7] receives
 * iters_per_tile, total_tiles, streamk_tiles, blocking_tiles, full_tiles,
 * partial_tiles, sm_partition_factor.
 */
int gemm_plan_streamk(int64_t m, int64_t n, int64_t k, int32_t block_m, int32_t block_n,
                      int32_t block_k, int32_t total_sm, int64_t out[7]);

/*
 * Host-only diagnostic: the name (as gemm_last_choice prints it) of the kernel
 * and schedule the heuristic picks, with no cache entry and no forced
 * schedule, for a problem of this shape and these types on a device with
 * sm_count SMs and partials_size bytes of workspace partials.  quant_a_group /
 * quant_b_group > 0 mean U / V scales; num_experts > 0 describes a grouped
 * problem with m rows in total.  Needs no GPU.  Writes a NUL-terminated name
 * of at most cap bytes to out; returns GEMM_ERR_INVALID_ARG for bad arguments
 * or a too small buffer.
 */
int gemm_heuristic_choice(int64_t m, int64_t n, int64_t k, int32_t a_type, int32_t b_type, int32_t d_type,
                          int32_t quant_a_group, int32_t quant_b_group, int32_t num_experts, int32_t sm_count,
                          size_t partials_size, char* out, size_t cap);

/* gemm_grouped_block: the grouped tile map (same page, section gemm_grouped)
 * for padded M-block `block` of experts with `sizes[0..E-1]` rows:
 * out[0] = expert, out[1] = first row, out[2] = rows (0 past the last block).
 * This is the code the device runs. */
int gemm_grouped_block(const int32_t* sizes, int32_t num_experts, int32_t block_m, int64_t block,
                       int64_t out[3]);

#ifdef __cplusplus
}
#endif
#endif /* QGEMM_GEMM_H_ */
