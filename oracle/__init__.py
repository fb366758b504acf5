"""CPU oracle for the GEMM library -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The GPU library never does, and nothing here is
shared with it: the floating-point definition lives in ``gemm_oracle.c``
(plain fp64 triple loop, OpenMP over rows); the integer schedules below are
restated from the pages in plain Python.

Sources, by page and section:
  * D = alpha*(A@B) + beta*C with U/V scale operands, C unused when beta == 0:
    "InternLM Lmdeploy Gemm Interface", Description / Signature / Usage Examples.
  * Scale operands advance at K-group boundaries: "InternLM Lmdeploy Gemm
    MainloopSm80V2", Description.
  * FP8 (E4M3 / E5M2) operands: DeepGEMM kernel-set blog, sections 1.2 and
    6.3 (quantised INT8/FP8 inputs; the FP8 path as the extension that pays
    off most on new hardware).
  * split-K, stream-K plan, grouped (MoE) tile map and batched flattening:
    TileLang tutorial "gemm_variants.py", sections gemm_splitk, gemm_streamk,
    streamk_plan, gemm_grouped, gemm_batched.

Every function here is pinned by tests under ``tests/`` against something
other than itself (numpy float64 matmul, brute force, closed forms, worked
examples); see the test module docstrings.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

F32, F16, BF16, S4, S8, E4M3, E5M2 = 0, 1, 2, 3, 4, 5, 6
FP8 = (E4M3, E5M2)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle in place (gcc, OpenMP).  Returns the .so path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Gemm(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("a_type", ctypes.c_int), ("A", ctypes.c_void_p), ("lda", ctypes.c_int64),
        ("b_type", ctypes.c_int), ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64),
        ("u_type", ctypes.c_int), ("U", ctypes.c_void_p), ("ldu", ctypes.c_int64), ("ga", ctypes.c_int64),
        ("v_type", ctypes.c_int), ("V", ctypes.c_void_p), ("ldv", ctypes.c_int64), ("gb", ctypes.c_int64),
        ("c_type", ctypes.c_int), ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
        ("alpha", ctypes.c_double), ("beta", ctypes.c_double),
        ("epilogue", ctypes.c_int), ("bias_type", ctypes.c_int), ("bias", ctypes.c_void_p),
        ("Z", ctypes.c_void_p), ("ldz", ctypes.c_int64),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.oracle_decode.restype = ctypes.c_double
            L.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
            L.oracle_encode_rn.restype = ctypes.c_uint32
            L.oracle_encode_rn.argtypes = [ctypes.c_int, ctypes.c_double]
            L.oracle_ulp.restype = ctypes.c_double
            L.oracle_ulp.argtypes = [ctypes.c_int, ctypes.c_double]
            L.oracle_int4_at.restype = ctypes.c_int
            L.oracle_int4_at.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
            L.oracle_zero_at.restype = ctypes.c_int
            L.oracle_zero_at.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
            L.oracle_gemm.restype = ctypes.c_int
            L.oracle_gemm.argtypes = [ctypes.POINTER(_Gemm), ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_gemm_entries.restype = ctypes.c_int
            L.oracle_gemm_entries.argtypes = [ctypes.POINTER(_Gemm), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


# ---- scalar formats --------------------------------------------------------

def decode(dtype: int, bits) -> np.ndarray:
    """Exact value of stored fp16/bf16/fp32 or E4M3/E5M2 bit patterns, as float64."""
    L = lib()
    flat = np.asarray(bits).reshape(-1)
    out = np.fromiter((L.oracle_decode(dtype, int(b)) for b in flat), dtype=np.float64, count=flat.size)
    return out.reshape(np.shape(bits))


def encode_rn(dtype: int, values) -> np.ndarray:
    """Round float64 values to fp16/bf16 (RN-even); returns bit patterns."""
    L = lib()
    flat = np.asarray(values, dtype=np.float64).reshape(-1)
    out = np.fromiter((L.oracle_encode_rn(dtype, float(v)) for v in flat), dtype=np.uint32, count=flat.size)
    return out.reshape(np.shape(values))


def ulp(dtype: int, values) -> np.ndarray:
    L = lib()
    flat = np.asarray(values, dtype=np.float64).reshape(-1)
    out = np.fromiter((L.oracle_ulp(dtype, float(v)) for v in flat), dtype=np.float64, count=flat.size)
    return out.reshape(np.shape(values))


def int4_at(packed: np.ndarray, n: int, k: int) -> int:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    return int(lib().oracle_int4_at(p.ctypes.data, p.shape[1], n, k))


def zero_at(Z: np.ndarray, g: int, n: int) -> int:
    """Zero point of K-group g, column n: the low nibble of byte Z[g][n], two's
    complement."""
    z = np.ascontiguousarray(Z, dtype=np.int8)
    return int(lib().oracle_zero_at(z.ctypes.data, z.shape[1], g, n))


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Signed nibbles of a packed N x (K/2) byte matrix as an N x K int array:
    byte t holds k = 2t in bits 3:0 and k = 2t+1 in bits 7:4."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0xF).astype(np.int64)
    hi = (p >> 4).astype(np.int64)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return np.where(out >= 8, out - 16, out)


# ---- the GEMM ----------------------------------------------------------------

def _arr(x, dt):
    return None if x is None else np.ascontiguousarray(x, dtype=dt)


def _desc(p, keep):
    """Build the C problem struct from a synth.Problem-like object."""
    g = _Gemm()
    g.M, g.N, g.K = p.M, p.N, p.K
    A = _arr(p.A, np.uint8 if p.a_type in FP8 else np.uint16)
    keep.append(A)
    g.a_type, g.A, g.lda = p.a_type, A.ctypes.data, p.K
    if p.b_type == S4:
        B = _arr(p.B, np.uint8)
        g.ldb = p.K // 2
    elif p.b_type in FP8:
        B = _arr(p.B, np.uint8)
        g.ldb = p.K
    else:
        B = _arr(p.B, np.uint16)
        g.ldb = p.K
    keep.append(B)
    g.b_type, g.B = p.b_type, B.ctypes.data
    if getattr(p, "U", None) is not None:
        U = _arr(p.U, np.float32 if p.u_type == F32 else np.uint16).view(
            np.uint32 if p.u_type == F32 else np.uint16)
        keep.append(U)
        g.u_type, g.U, g.ldu, g.ga = p.u_type, U.ctypes.data, p.M, p.ga
    if getattr(p, "V", None) is not None:
        V = _arr(p.V, np.float32 if p.v_type == F32 else np.uint16).view(
            np.uint32 if p.v_type == F32 else np.uint16)
        keep.append(V)
        g.v_type, g.V, g.ldv, g.gb = p.v_type, V.ctypes.data, p.N, p.gb
    if getattr(p, "Z", None) is not None:
        Z = _arr(p.Z, np.int8)
        keep.append(Z)
        g.Z, g.ldz = Z.ctypes.data, p.N
    g.alpha, g.beta = float(p.alpha), float(p.beta)
    g.epilogue = int(getattr(p, "epilogue", 0) or 0)
    if g.epilogue & 1:
        bias = np.ascontiguousarray(p.bias)
        bias = bias.view(np.uint32) if p.bias_type == F32 else bias.astype(np.uint16, copy=False)
        keep.append(bias)
        g.bias_type, g.bias = p.bias_type, bias.ctypes.data
    if p.beta != 0.0:
        C = np.ascontiguousarray(p.C)
        C = C.view(np.uint32) if p.c_type == F32 else C.astype(np.uint16, copy=False)
        keep.append(C)
        g.c_type, g.C, g.ldc = p.c_type, C.ctypes.data, p.N
    return g


def gemm(p):
    """(ref, bound) for a whole problem, both M x N float64."""
    keep = []
    g = _desc(p, keep)
    ref = np.empty((p.M, p.N), dtype=np.float64)
    bound = np.empty((p.M, p.N), dtype=np.float64)
    rc = lib().oracle_gemm(ctypes.byref(g), ref.ctypes.data, bound.ctypes.data)
    if rc:
        raise RuntimeError(f"oracle_gemm failed ({rc})")
    return ref, bound


def gemm_entries(p, ii, jj):
    """(ref, bound) at the listed (ii[t], jj[t]) entries only."""
    keep = []
    g = _desc(p, keep)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    ref = np.empty(ii.size, dtype=np.float64)
    bound = np.empty(ii.size, dtype=np.float64)
    rc = lib().oracle_gemm_entries(ctypes.byref(g), ii.ctypes.data, jj.ctypes.data, ii.size,
                                   ref.ctypes.data, bound.ctypes.data)
    if rc:
        raise RuntimeError(f"oracle_gemm_entries failed ({rc})")
    return ref, bound


def quantize_s8(x, scale, zp):
    """Output quantisation (DeepGEMM kernel-set blog, section 6.2): the int8 code
    round(x * scale_i + zp) of every value of row i, to nearest-even, saturated
    to [-128, 127], NaN giving 0.  x: [M, N] values before rounding (float64),
    scale: [M] per-row (per-token) scales."""
    t = np.asarray(x, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[:, None] + float(zp)
    q = np.clip(np.rint(t), -128, 127)
    return np.where(np.isnan(t), 0.0, q)


class _Slice:
    """One expert's rows of a grouped problem, viewed as a dense problem."""

    def __init__(self, gp, e, rows=None):
        lo, hi = int(gp.offsets[e]), int(gp.offsets[e + 1])
        idx = np.arange(lo, hi) if rows is None else lo + np.asarray(rows, dtype=np.int64)
        self.M = len(idx)
        self.N, self.K = gp.N, gp.K
        self.a_type = gp.a_type
        self.b_type = gp.b_type if getattr(gp, "b_type", None) is not None else gp.a_type
        self.A = gp.A[idx]
        self.B = gp.B[e]
        # per-expert V (and zero points); U holds one scale per token row
        self.V = gp.V[e] if getattr(gp, "V", None) is not None else None
        self.v_type, self.gb = getattr(gp, "v_type", None), getattr(gp, "gb", 0)
        self.Z = gp.Z[e] if getattr(gp, "Z", None) is not None else None
        self.U = np.ascontiguousarray(gp.U[:, idx]) if getattr(gp, "U", None) is not None else None
        self.u_type, self.ga = getattr(gp, "u_type", None), getattr(gp, "ga", 0)
        self.alpha, self.beta = gp.alpha, gp.beta
        self.C = None
        self.c_type = None
        self.epilogue = getattr(gp, "epilogue", 0)
        self.bias, self.bias_type = getattr(gp, "bias", None), getattr(gp, "bias_type", None)


def grouped(gp):
    """Grouped GEMM as the loop of per-expert GEMMs it is defined to be:
    rows offsets[e]..offsets[e+1] of A times expert e's B (dequantised with
    expert e's V and zero points, A's rows scaled by their U columns).
    Returns (ref, bound) of shape [sum m_e, N]."""
    T = int(gp.offsets[-1])
    ref = np.empty((T, gp.N), dtype=np.float64)
    bound = np.empty((T, gp.N), dtype=np.float64)
    for e in range(len(gp.counts)):
        lo, hi = int(gp.offsets[e]), int(gp.offsets[e + 1])
        if hi > lo:
            r, b = gemm(_Slice(gp, e))
            ref[lo:hi], bound[lo:hi] = r, b
    return ref, bound


def grouped_entries(gp, ii, jj):
    """Sampled entries of a grouped result: row ii[t] belongs to the expert
    whose offset range holds it."""
    ii = np.asarray(ii, dtype=np.int64)
    jj = np.asarray(jj, dtype=np.int64)
    ref = np.empty(ii.size)
    bound = np.empty(ii.size)
    experts = np.searchsorted(gp.offsets, ii, side="right") - 1
    for e in np.unique(experts):
        sel = np.nonzero(experts == e)[0]
        sl = _Slice(gp, int(e))
        r, b = gemm_entries(sl, ii[sel] - int(gp.offsets[e]), jj[sel])
        ref[sel], bound[sel] = r, b
    return ref, bound


# ---- integer schedules (TileLang "gemm_variants.py") ---------------------------

def streamk_plan(m, n, k, block_m, block_n, block_k, total_sm):
    """The stream-K sizing of the tutorial's ``streamk_plan`` section: tiles
    that do not fill a last whole wave (plus one more wave when more than one
    wave of whole tiles remains) are shared out by iteration; the rest are
    handed out whole."""
    num_block_m = -(-m // block_m)
    num_block_n = -(-n // block_n)
    iters_per_tile = -(-k // block_k)
    total_tiles = num_block_m * num_block_n
    streamk_tiles = total_tiles % total_sm
    if total_tiles - streamk_tiles > total_sm:
        streamk_tiles += total_sm
    blocking_tiles = total_tiles - streamk_tiles
    streamk_iters = streamk_tiles * iters_per_tile
    return {
        "iters_per_tile": iters_per_tile,
        "total_tiles": total_tiles,
        "streamk_tiles": streamk_tiles,
        "blocking_tiles": blocking_tiles,
        "full_tiles": streamk_iters // total_sm,
        "partial_tiles": streamk_iters % total_sm,
        "sm_partition_factor": max(blocking_tiles // total_sm, 1),
    }


def streamk_program_work(plan, pid, programs):
    """The (tile, k_begin, k_end) segments program ``pid`` runs, in order.

    Stream-K phase: the program's iteration range starts at
    pid*full + min(pid, partial) and ends where program pid+1's begins; it is
    cut at tile boundaries.  Blocking phase: tile pid + streamk_tiles +
    p*programs for p < sm_partition_factor, skipped when it is past the last
    tile (the plan sets the factor to 1 even when no blocking tile exists)."""
    ipt = plan["iters_per_tile"]
    full, part = plan["full_tiles"], plan["partial_tiles"]
    start = pid * full + min(pid, part)
    last = (pid + 1) * full + min(pid + 1, part)
    out = []
    it = start
    while it < last:
        end = min(it + (ipt - it % ipt), last)
        out.append((it // ipt, it % ipt, it % ipt + (end - it)))
        it = end
    for p in range(plan["sm_partition_factor"]):
        t = pid + plan["streamk_tiles"] + p * programs
        if t < plan["total_tiles"]:
            out.append((t, 0, ipt))
    return out


def splitk_ranges(k_iters, splits):
    """Split-K slices in whole K-steps: chunk = ceil(k_iters / splits); the
    number of slices is clipped so none is empty; the last may be shorter."""
    if k_iters <= 0:
        return [(0, 0)]
    splits = max(1, min(splits, k_iters))
    chunk = -(-k_iters // splits)
    n = -(-k_iters // chunk)
    return [(s * chunk, min(k_iters, (s + 1) * chunk)) for s in range(n)]


def grouped_tile_map(sizes, block_m):
    """Per padded M-block of a grouped GEMM: (expert, m_start, actual_rows).

    padded_off[e] = sum_{j<e} ceil(m_j / bM) * bM; block b belongs to the
    largest e with padded_off[e] <= b*bM (a linear scan that keeps the last
    match); m_start = b*bM - padded_off[e] + off[e];
    rows = max(0, min(bM, m_e + padded_off[e] - b*bM))."""
    sizes = [int(s) for s in sizes]
    off, padded = [], []
    o = po = 0
    for s in sizes:
        off.append(o)
        padded.append(po)
        o += s
        po += -(-s // block_m) * block_m
    total_blocks = sum(-(-s // block_m) for s in sizes)
    out = []
    for b in range(total_blocks):
        ms = b * block_m
        e = 0
        for i in range(len(sizes)):
            if ms >= padded[i]:
                e = i
        m_start = ms - padded[e] + off[e]
        rows = max(0, min(block_m, sizes[e] + padded[e] - ms))
        out.append((e, m_start, rows))
    return out


def batched_block(cid, m_num, n_num):
    """Flattened batched grid index -> (batch, m-block, n-block)."""
    bid = cid // (m_num * n_num)
    rem = cid % (m_num * n_num)
    return bid, rem // n_num, rem % n_num
