"""Python binding of the GB300 GEMM library (libqgemm.so).

Argument marshalling only: every function here forwards to the C ABI of
``include/gemm.h`` under the same name; every step of the GEMM runs in the
library's CUDA kernels.  PyTorch is used for device memory and streams in the
convenience helpers at the bottom (``layout_of``, ``Workspace``, ``run``).

Loading fails loudly (``LibraryNotBuilt``) when the shared library is missing:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqgemm.so")
# the checked debug build (device-side bounds checks); loaded instead of the
# regular library when GEMM_DEVICE_CHECKS=1 is set in the environment
CHECKED_LIB_PATH = os.path.join(_PKG, "libqgemm_checked.so")

# ---- enums (gemm.h) -----------------------------------------------------------
GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_WORKSPACE = 3
GEMM_ERR_CUDA = 4
GEMM_ERR_NO_KERNEL = 5
GEMM_ERR_DEVICE_TIMEOUT = 6
GEMM_ERR_BAD_CACHE = 7
GEMM_ERR_DEVICE_CHECK = 8

GEMM_F32, GEMM_F16, GEMM_BF16, GEMM_S4, GEMM_S8, GEMM_E4M3, GEMM_E5M2 = 0, 1, 2, 3, 4, 5, 6
GEMM_ROW_MAJOR, GEMM_COL_MAJOR = 0, 1
GEMM_DISPATCH_DEFAULT, GEMM_DISPATCH_MEASURE, GEMM_DISPATCH_REUSE = 0, 1, 2
GEMM_EPILOGUE_DEFAULT, GEMM_EPILOGUE_BIAS, GEMM_EPILOGUE_RELU, GEMM_EPILOGUE_GELU = 0, 1, 2, 4
GEMM_BARRIERS_SIZE = 1 << 20
GEMM_PARTIALS_SIZE = 32 << 20
GEMM_NOALLOC_BARRIERS_SIZE = 64 << 10
GEMM_NOALLOC_PARTIALS_SIZE = 8 << 20

# Every exported symbol of gemm.h.
SYMBOLS = (
    "gemm_create", "gemm_destroy", "gemm_run", "gemm_run_grouped", "gemm_export", "gemm_import",
    "gemm_get_tuning_seq", "gemm_cache_size", "gemm_status_string", "gemm_device_status",
    "gemm_selftest_wait_timeout", "gemm_last_choice", "gemm_plan_streamk", "gemm_grouped_block",
    "gemm_run_noalloc", "gemm_heuristic_choice", "gemm_checked_build",
)


class LibraryNotBuilt(ImportError):
    pass


class GemmError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {gemm_status_string(code)} ({code})" if what else gemm_status_string(code))


class gemm_layout_t(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int32), ("order", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ld", ctypes.c_int64), ("num", ctypes.c_int32),
                ("batch_stride", ctypes.c_int64)]


class gemm_op_t(ctypes.Structure):
    _fields_ = [("dispatch", ctypes.c_int32), ("epilogue", ctypes.c_int32), ("quant_a_group", ctypes.c_int32),
                ("quant_b_group", ctypes.c_int32), ("splitk", ctypes.c_int32), ("streamk", ctypes.c_int32),
                ("bias", ctypes.c_void_p), ("bias_type", ctypes.c_int32), ("out_zero_point", ctypes.c_int32),
                ("out_scale", ctypes.c_void_p), ("b_zero", ctypes.c_void_p), ("b_zero_ld", ctypes.c_int64),
                ("b_zero_batch_stride", ctypes.c_int64)]


class gemm_workspace_t(ctypes.Structure):
    _fields_ = [("barriers", ctypes.c_void_p), ("barriers_size", ctypes.c_size_t),
                ("partials", ctypes.c_void_p), ("partials_size", ctypes.c_size_t)]


_lib = None


def lib():
    """The loaded shared library (raises LibraryNotBuilt if absent)."""
    global _lib
    if _lib is not None:
        return _lib
    path = CHECKED_LIB_PATH if os.environ.get("GEMM_DEVICE_CHECKS") == "1" else LIB_PATH
    if not os.path.exists(path):
        raise LibraryNotBuilt(f"{path} is missing; run __graft_entry__.build() or "
                              "python quantized_gemm_tcgen05_gb300/_build.py"
                              + (" --checks" if path == CHECKED_LIB_PATH else ""))
    L = ctypes.CDLL(path)
    P, I32, I64, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    LP = ctypes.POINTER(gemm_layout_t)
    sig = {
        "gemm_create": (ctypes.c_int, [ctypes.POINTER(P)]),
        "gemm_destroy": (ctypes.c_int, [P]),
        "gemm_run": (ctypes.c_int, [P, ctypes.POINTER(gemm_op_t), F, P, LP, P, LP, P, LP, P, LP, F, P, LP, P, LP,
                                    ctypes.POINTER(gemm_workspace_t), P]),
        "gemm_run_noalloc": (ctypes.c_int, [P, ctypes.POINTER(gemm_op_t), F, P, LP, P, LP, P, LP, P, LP, F, P, LP, P,
                                            LP, P]),
        "gemm_run_grouped": (ctypes.c_int, [P, ctypes.POINTER(gemm_op_t), F, P, LP, P, LP, P, LP, P, LP, F, P, LP,
                                            P, LP, P, I32, ctypes.POINTER(gemm_workspace_t), P]),
        "gemm_export": (ctypes.c_int, [P, P, SZ, ctypes.POINTER(SZ)]),
        "gemm_import": (ctypes.c_int, [P, P, SZ]),
        "gemm_get_tuning_seq": (ctypes.c_int, [P, ctypes.POINTER(I32), I32, ctypes.POINTER(I32)]),
        "gemm_cache_size": (ctypes.c_int, [P, ctypes.POINTER(I32)]),
        "gemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "gemm_device_status": (ctypes.c_int, [P, P]),
        "gemm_selftest_wait_timeout": (ctypes.c_int, [P, ctypes.c_uint64, P]),
        "gemm_last_choice": (ctypes.c_char_p, [P]),
        "gemm_plan_streamk": (ctypes.c_int, [I64, I64, I64, I32, I32, I32, I32, ctypes.POINTER(I64)]),
        "gemm_grouped_block": (ctypes.c_int, [ctypes.POINTER(I32), I32, I32, I64, ctypes.POINTER(I64)]),
        "gemm_heuristic_choice": (ctypes.c_int, [I64, I64, I64, I32, I32, I32, I32, I32, I32, I32, ctypes.c_size_t,
                                                 ctypes.c_char_p, ctypes.c_size_t]),
        "gemm_checked_build": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _lib = L
    return L


# ---- thin forwards, same names as the C ABI ----------------------------------------

def gemm_status_string(code: int) -> str:
    try:
        return lib().gemm_status_string(int(code)).decode()
    except LibraryNotBuilt:
        return f"status {code}"


def gemm_create():
    h = ctypes.c_void_p()
    rc = lib().gemm_create(ctypes.byref(h))
    if rc:
        raise GemmError(rc, "gemm_create")
    return h


def gemm_destroy(h):
    return lib().gemm_destroy(h)


def _lp(x):
    return None if x is None else ctypes.byref(x)


def gemm_run(h, op, alpha, A, Adesc, U, Udesc, B, Bdesc, V, Vdesc, beta, C, Cdesc, D, Ddesc, workspace, stream):
    """Returns the status code (0 = OK).  Pointers are ints (device addresses)."""
    return lib().gemm_run(h, ctypes.byref(op), float(alpha), A, _lp(Adesc), U, _lp(Udesc), B, _lp(Bdesc), V,
                          _lp(Vdesc), float(beta), C, _lp(Cdesc), D, _lp(Ddesc), _lp(workspace), stream)


def gemm_run_noalloc(h, op, alpha, A, Adesc, U, Udesc, B, Bdesc, V, Vdesc, beta, C, Cdesc, D, Ddesc, stream):
    """gemm_run whose split-K / stream-K scratch is the library's own fixed
    device array (no workspace argument, no allocation)."""
    return lib().gemm_run_noalloc(h, ctypes.byref(op), float(alpha), A, _lp(Adesc), U, _lp(Udesc), B, _lp(Bdesc), V,
                                  _lp(Vdesc), float(beta), C, _lp(Cdesc), D, _lp(Ddesc), stream)


def gemm_run_grouped(h, op, alpha, A, Adesc, U, Udesc, B, Bdesc, V, Vdesc, beta, C, Cdesc, D, Ddesc,
                     expert_offsets_dev, num_experts, workspace, stream):
    return lib().gemm_run_grouped(h, ctypes.byref(op), float(alpha), A, _lp(Adesc), U, _lp(Udesc), B, _lp(Bdesc),
                                  V, _lp(Vdesc), float(beta), C, _lp(Cdesc), D, _lp(Ddesc), expert_offsets_dev,
                                  int(num_experts), _lp(workspace), stream)


def gemm_export(h) -> bytes:
    n = ctypes.c_size_t()
    rc = lib().gemm_export(h, None, 0, ctypes.byref(n))
    if rc:
        raise GemmError(rc, "gemm_export")
    buf = ctypes.create_string_buffer(max(n.value, 1))
    rc = lib().gemm_export(h, buf, n.value, ctypes.byref(n))
    if rc:
        raise GemmError(rc, "gemm_export")
    return buf.raw[:n.value]


def gemm_import(h, blob: bytes) -> int:
    return lib().gemm_import(h, blob, len(blob))


def gemm_get_tuning_seq(h):
    n = ctypes.c_int32()
    rc = lib().gemm_get_tuning_seq(h, None, 0, ctypes.byref(n))
    if rc:
        raise GemmError(rc, "gemm_get_tuning_seq")
    out = (ctypes.c_int32 * n.value)()
    lib().gemm_get_tuning_seq(h, out, n.value, ctypes.byref(n))
    return list(out)


def gemm_cache_size(h) -> int:
    n = ctypes.c_int32()
    rc = lib().gemm_cache_size(h, ctypes.byref(n))
    if rc:
        raise GemmError(rc, "gemm_cache_size")
    return n.value


def gemm_device_status(h, stream=None) -> int:
    return lib().gemm_device_status(h, stream)


def gemm_selftest_wait_timeout(h, timeout_ns, stream=None) -> int:
    return lib().gemm_selftest_wait_timeout(h, int(timeout_ns), stream)


def gemm_last_choice(h) -> str:
    return lib().gemm_last_choice(h).decode()


def gemm_plan_streamk(m, n, k, block_m, block_n, block_k, total_sm):
    out = (ctypes.c_int64 * 7)()
    rc = lib().gemm_plan_streamk(m, n, k, block_m, block_n, block_k, total_sm, out)
    if rc:
        raise GemmError(rc, "gemm_plan_streamk")
    keys = ("iters_per_tile", "total_tiles", "streamk_tiles", "blocking_tiles", "full_tiles", "partial_tiles",
            "sm_partition_factor")
    return dict(zip(keys, list(out)))


def gemm_heuristic_choice(m, n, k, a_type, b_type, d_type, quant_a_group=0, quant_b_group=0, num_experts=0,
                          sm_count=152, partials_size=GEMM_PARTIALS_SIZE):
    """The kernel / schedule name the heuristic picks for this problem (host only)."""
    buf = ctypes.create_string_buffer(96)
    rc = lib().gemm_heuristic_choice(m, n, k, a_type, b_type, d_type, quant_a_group, quant_b_group, num_experts,
                                     sm_count, partials_size, buf, len(buf))
    if rc:
        raise GemmError(rc, "gemm_heuristic_choice")
    return buf.value.decode()


def gemm_grouped_block(sizes, block_m, block):
    arr = (ctypes.c_int32 * len(sizes))(*[int(s) for s in sizes])
    out = (ctypes.c_int64 * 3)()
    rc = lib().gemm_grouped_block(arr, len(sizes), block_m, block, out)
    if rc:
        raise GemmError(rc, "gemm_grouped_block")
    return tuple(out)


# ---- torch convenience (memory and streams only) ------------------------------------

def _dtype_code(t):
    import torch
    return {torch.float32: GEMM_F32, torch.float16: GEMM_F16, torch.bfloat16: GEMM_BF16, torch.int8: GEMM_S8,
            torch.float8_e4m3fn: GEMM_E4M3, torch.float8_e5m2: GEMM_E5M2}[t]


def layout(type_, order, rows, cols, ld, num=1, batch_stride=0):
    return gemm_layout_t(type_, order, rows, cols, ld, num, batch_stride)


def row_major(t, type_=None):
    """Layout of a [rows, cols] or [num, rows, cols] row-major tensor."""
    type_ = _dtype_code(t.dtype) if type_ is None else type_
    if t.dim() == 3:
        return layout(type_, GEMM_ROW_MAJOR, t.shape[1], t.shape[2], max(t.stride(1), t.shape[2], 1), t.shape[0],
                      t.stride(0))
    return layout(type_, GEMM_ROW_MAJOR, t.shape[0], t.shape[1], max(t.stride(0), t.shape[1], 1))


def col_major_from_nk(t, k=None, type_=None):
    """Layout of B given as a [N, K] (or [num, N, K]) tensor with K contiguous,
    i.e. a col-major K x N matrix.  For packed int4 pass type_=GEMM_S4 and the
    uint8 [N, K/2] tensor; k then is K."""
    type_ = _dtype_code(t.dtype) if type_ is None else type_
    mult = 2 if type_ == GEMM_S4 else 1
    kk = t.shape[-1] * mult if k is None else k
    if t.dim() == 3:
        return layout(type_, GEMM_COL_MAJOR, kk, t.shape[1], max(t.stride(1) * mult, kk, 1), t.shape[0],
                      t.stride(0) * mult)
    return layout(type_, GEMM_COL_MAJOR, kk, t.shape[0], max(t.stride(0) * mult, kk, 1))


class Workspace:
    """Caller-owned workspace: 1 MB of zeroed barriers and 32 MB of partials."""

    def __init__(self, device="cuda", barriers_size=GEMM_BARRIERS_SIZE, partials_size=GEMM_PARTIALS_SIZE):
        import torch
        self.barriers = torch.zeros(barriers_size, dtype=torch.uint8, device=device)
        self.partials = torch.empty(partials_size, dtype=torch.uint8, device=device)
        self.c = gemm_workspace_t(self.barriers.data_ptr(), barriers_size, self.partials.data_ptr(), partials_size)


def current_stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def ptr(t):
    return None if t is None else t.data_ptr()
