"""Shared helpers for the GPU parity tests: move synth problems to the device,
call the library through its C ABI, and compare with the oracle under the
acceptance rule

    |D - ref| <= 1e-5 * S + 1e-6                 (fp32 D)
    |D - ref| <= 1e-5 * S + 1e-6 + ulp_D(ref)    (fp16 / bf16 D)

where S = |alpha| * sum_k |a_ik * b_kj| + |beta * c_ij| is returned by the
oracle alongside ref.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import quantized_gemm_tcgen05_gb300 as qg
import oracle
import synth

TORCH_DT = {synth.F32: torch.float32, synth.F16: torch.float16, synth.BF16: torch.bfloat16, synth.S8: torch.int8,
            synth.E4M3: torch.float8_e4m3fn, synth.E5M2: torch.float8_e5m2}


def dev_bits(bits, dtype):
    """numpy storage bits -> device tensor of the storage dtype."""
    if dtype == synth.F32:
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.float32)).cuda()
    if dtype == synth.S4:
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).cuda()
    if dtype in (synth.E4M3, synth.E5M2):
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).view(TORCH_DT[dtype]).cuda()
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(TORCH_DT[dtype]).cuda()


def padded_rows(bits, dtype):
    """A 2-D scale matrix on the device with its row stride rounded up to 8
    elements; returns (tensor, ld)."""
    rows, cols = bits.shape
    ld = -(-cols // 8) * 8
    t = torch.zeros(rows, ld, dtype=TORCH_DT[dtype], device="cuda")
    t[:, :cols] = dev_bits(bits, dtype)
    return t, ld


def zero_rows(Z):
    """int8 zero points [.., rows, cols] on the device with the row stride
    rounded up to 16 bytes; returns (tensor, ld, batch stride in bytes)."""
    Z = np.ascontiguousarray(Z, dtype=np.int8)
    lead, (rows, cols) = Z.shape[:-2], Z.shape[-2:]
    ld = -(-cols // 16) * 16
    t = torch.zeros(*lead, rows, ld, dtype=torch.int8, device="cuda")
    t[..., :cols] = torch.from_numpy(Z).cuda()
    return t, ld, rows * ld


def tolerance(ref, bound, d_type):
    tol = 1e-5 * bound + 1e-6
    if d_type != synth.F32:
        tol = tol + oracle.ulp(d_type, ref)
    return tol


def assert_quant(d, ref, bound, scale, zp, what=""):
    """An int8 D against the oracle's pre-rounding values: each code must lie
    between the codes of ref*scale+zp moved by the fp32 value's tolerance (and
    the fma's rounding) either way; where no rounding boundary lies within
    that band this is the single exact code."""
    d = np.asarray(d, dtype=np.float64)
    s = np.asarray(scale, dtype=np.float64)[:, None]
    band = tolerance(ref, bound, synth.F32) * np.abs(s) + 1e-4
    lo = oracle.quantize_s8(ref - band / np.abs(s) * np.sign(s), scale, zp)
    hi = oracle.quantize_s8(ref + band / np.abs(s) * np.sign(s), scale, zp)
    lo, hi = np.minimum(lo, hi), np.maximum(lo, hi)
    bad = (d < lo) | (d > hi)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        exact = oracle.quantize_s8(ref, scale, zp)
        msg = ", ".join(f"{tuple(i)}: got {d[tuple(i)]:.0f} want {exact[tuple(i)]:.0f} [{lo[tuple(i)]:.0f}, {hi[tuple(i)]:.0f}]"
                        for i in idx)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} int8 codes out of range; {msg}")
    return int((lo != hi).sum())


def assert_close(d, ref, bound, d_type, what=""):
    d = np.asarray(d, dtype=np.float64)
    tol = tolerance(ref, bound, d_type)
    err = np.abs(d - ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = ", ".join(f"{tuple(i)}: got {d[tuple(i)]!r} ref {ref[tuple(i)]!r} tol {tol[tuple(i)]:.3g}"
                        for i in idx)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; {msg}")


class Lib:
    """A handle plus a workspace on the current device."""

    def __init__(self):
        self.h = qg.gemm_create()
        self.ws = qg.Workspace()

    def close(self):
        qg.gemm_destroy(self.h)


def op(dispatch=0, splitk=0, streamk=0, ga=0, gb=0):
    return qg.gemm_op_t(dispatch, 0, ga, gb, splitk, streamk)


def run_problem(lib, p, o=None, D=None, C=None, stream=None, workspace=True):
    """Run a synth.Problem through gemm_run.  Returns (status, D tensor)."""
    o = o or op(ga=p.ga if p.U is not None else 0, gb=p.gb if p.V is not None else 0)
    A = dev_bits(p.A, p.a_type)
    B = dev_bits(p.B, p.b_type)
    Ad = qg.row_major(A)
    Bd = qg.col_major_from_nk(B, k=p.K, type_=p.b_type)
    if D is None:
        fill = 101 if p.d_type == synth.S8 else float("nan")  # a code the tests' scales never produce
        D = torch.full((p.M, p.N), fill, dtype=TORCH_DT[p.d_type], device="cuda")
    Dd = qg.row_major(D)
    Cd = None
    if p.beta != 0.0 and C is None:
        C = dev_bits(p.C, p.c_type)
    if C is not None:
        Cd = qg.row_major(C)
    U = Ud = V = Vd = None
    if p.U is not None:  # scale rows padded to a multiple of 8 elements (16 bytes)
        U, ldu = padded_rows(p.U, p.u_type)
        Ud = qg.layout(p.u_type, qg.GEMM_ROW_MAJOR, p.K // p.ga, p.M, ldu)
    if p.V is not None:
        V, ldv = padded_rows(p.V, p.v_type)
        Vd = qg.layout(p.v_type, qg.GEMM_ROW_MAJOR, p.K // p.gb, p.N, ldv)
    bias = _attach_epilogue(p, o)
    Z = None
    if getattr(p, "Z", None) is not None:
        Z, o.b_zero_ld, _ = zero_rows(p.Z)
        o.b_zero = qg.ptr(Z)
    qs = None
    if p.d_type == synth.S8:
        qs = torch.from_numpy(np.ascontiguousarray(p.q_scale, dtype=np.float32)).cuda()
        o.out_scale, o.out_zero_point = qg.ptr(qs), p.q_zp
    st = stream if stream is not None else qg.current_stream()
    rc = qg.gemm_run(lib.h, o, p.alpha, qg.ptr(A), Ad, qg.ptr(U), Ud, qg.ptr(B), Bd, qg.ptr(V), Vd, p.beta,
                     qg.ptr(C), Cd, qg.ptr(D), Dd, lib.ws.c if workspace else None, st)
    torch.cuda.synchronize()
    del bias, qs
    return rc, D


def _attach_epilogue(p, o):
    """Copy the problem's fused-epilogue flags and bias (if any) into the op.
    Returns the device bias tensor, which must outlive the call."""
    flags = getattr(p, "epilogue", 0) or 0
    if not flags:
        return None
    o.epilogue = flags
    if not flags & qg.GEMM_EPILOGUE_BIAS:
        return None
    bias = dev_bits(p.bias, p.bias_type)
    o.bias, o.bias_type = qg.ptr(bias), p.bias_type
    return bias


def grouped_to_device(gp):
    b_type = getattr(gp, "b_type", None)
    b_type = gp.a_type if b_type is None else b_type
    A = dev_bits(gp.A, gp.a_type)
    B = dev_bits(gp.B, b_type)
    off = torch.from_numpy(gp.offsets.astype(np.int32)).cuda()
    return A, B, off


def run_grouped(lib, gp, o=None, A=None, B=None, off=None):
    """Run a synth.GroupedProblem through gemm_run_grouped (with its per-token
    U, per-expert V and zero points when it has them).  Returns (status, D)."""
    if A is None:
        A, B, off = grouped_to_device(gp)
    T = int(gp.offsets[-1])
    E = len(gp.counts)
    fill = 101 if gp.d_type == synth.S8 else float("nan")
    D = torch.full((T, gp.N), fill, dtype=TORCH_DT[gp.d_type], device="cuda")
    o = o or op(ga=getattr(gp, "ga", 0) if getattr(gp, "U", None) is not None else 0,
                gb=getattr(gp, "gb", 0) if getattr(gp, "V", None) is not None else 0)
    b_type = getattr(gp, "b_type", None)
    Bd = qg.col_major_from_nk(B, k=gp.K, type_=gp.a_type if b_type is None else b_type)
    U = Ud = V = Vd = Z = None
    if getattr(gp, "U", None) is not None:
        U, ldu = padded_rows(gp.U, gp.u_type)
        Ud = qg.layout(gp.u_type, qg.GEMM_ROW_MAJOR, gp.K // gp.ga, T, ldu)
    if getattr(gp, "V", None) is not None:
        groups = gp.K // gp.gb
        ldv = -(-gp.N // 8) * 8
        V = torch.zeros(E, groups, ldv, dtype=TORCH_DT[gp.v_type], device="cuda")
        V[..., :gp.N] = dev_bits(gp.V, gp.v_type)
        Vd = qg.layout(gp.v_type, qg.GEMM_ROW_MAJOR, groups, gp.N, ldv, E, groups * ldv)
    if getattr(gp, "Z", None) is not None:
        Z, o.b_zero_ld, o.b_zero_batch_stride = zero_rows(gp.Z)
        o.b_zero = qg.ptr(Z)
    bias = _attach_epilogue(gp, o)
    qs = None
    if gp.d_type == synth.S8:
        qs = torch.from_numpy(np.ascontiguousarray(gp.q_scale, dtype=np.float32)).cuda()
        o.out_scale, o.out_zero_point = qg.ptr(qs), gp.q_zp
    rc = qg.gemm_run_grouped(lib.h, o, gp.alpha, qg.ptr(A), qg.row_major(A), qg.ptr(U), Ud, qg.ptr(B), Bd, qg.ptr(V),
                             Vd, gp.beta, None, None, qg.ptr(D), qg.row_major(D), qg.ptr(off), E, lib.ws.c,
                             qg.current_stream())
    torch.cuda.synchronize()
    del bias, qs, U, V, Z
    return rc, D


def sample_indices(M, N, n, seed):
    """Sampled (i, j) positions covering corners, tile edges and random interior."""
    rng = np.random.default_rng(seed)
    fixed_i = [0, M - 1, min(127, M - 1), min(128, M - 1), M // 2]
    fixed_j = [0, N - 1, min(255, N - 1), min(256, N - 1), N // 2]
    ii = np.concatenate([np.repeat(fixed_i, len(fixed_j)), rng.integers(0, M, n)])
    jj = np.concatenate([np.tile(fixed_j, len(fixed_i)), rng.integers(0, N, n)])
    return ii, jj
