"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers and rounds them once to the storage
type (fp16 / bf16 with round-to-nearest-even, int4 packed two per byte).  It
holds none of the GEMM arithmetic, so both the CUDA path and the CPU oracle
can consume its output without sharing any of the method's code.

Every array is returned as raw storage bits in numpy (uint16 for 16-bit
floats, uint8 for packed int4 and for 8-bit floats, float32 for fp32), laid
out exactly as the library expects them:

* A   : M x K, row-major (K contiguous)
* B   : "col-major K x N", i.e. stored N x K with K contiguous
* Bq  : int4 weights stored N x (K/2) bytes; byte t of row n holds k = 2t in
        bits 3:0 and k = 2t+1 in bits 7:4 (two's-complement nibbles)
* V   : per (K-group, column) scales, [K/g][N], N contiguous
* U   : per (K-group, row) scales,    [K/g][M], M contiguous
* C/D : M x N, row-major

The workloads follow the five configurations the GEMM is benchmarked on
(dense fp16 256^3, dense bf16 4096^3, decode-shaped bf16, W4A16, grouped MoE).
Seeds are 1000 + the configuration number (1..5).
"""
from __future__ import annotations

import dataclasses
import numpy as np

F32, F16, BF16, S4, S8, E4M3, E5M2 = 0, 1, 2, 3, 4, 5, 6
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16", S4: "s4", S8: "s8", E4M3: "e4m3", E5M2: "e5m2"}


def _round_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 values once (RN-even) to fp16/bf16 storage bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == F16:
        return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    if dtype == BF16:
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype in (E4M3, E5M2):
        # 8-bit floats: RN-even; the workloads' values stay far inside the
        # finite range (|x| <= 448 for E4M3), so nothing saturates
        f8 = torch.float8_e4m3fn if dtype == E4M3 else torch.float8_e5m2
        return t.to(f8).view(torch.uint8).numpy().copy()
    raise ValueError(f"cannot round to dtype {dtype}")


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Pack signed integers in [-8, 7], shape (N, K) with K even, two per byte.

    Byte t of row n holds k = 2t in the low nibble and k = 2t + 1 in the high
    nibble, two's complement.  This is storage layout only.
    """
    q = np.asarray(q, dtype=np.int64)
    if q.shape[-1] % 2:
        raise ValueError("K must be even to pack int4")
    if q.min(initial=0) < -8 or q.max(initial=0) > 7:
        raise ValueError("int4 values must lie in [-8, 7]")
    u = (q & 0xF).astype(np.uint8)
    return np.ascontiguousarray(u[..., 0::2] | (u[..., 1::2] << 4))


@dataclasses.dataclass
class Problem:
    """One GEMM instance: raw operand bits plus the scalars."""

    M: int
    N: int
    K: int
    a_type: int
    b_type: int
    d_type: int
    A: np.ndarray
    B: np.ndarray
    alpha: float = 1.0
    beta: float = 0.0
    c_type: int | None = None
    C: np.ndarray | None = None
    V: np.ndarray | None = None      # [K/gb][N]
    v_type: int | None = None
    gb: int = 0
    Z: np.ndarray | None = None      # int4 B with V: [K/gb][N] int8 zero points in [-8, 7]
    U: np.ndarray | None = None      # [K/ga][M]
    u_type: int | None = None
    ga: int = 0
    name: str = ""
    epilogue: int = 0                # fused epilogue flags: 1 bias, 2 ReLU, 4 GELU
    bias: np.ndarray | None = None   # [N] storage bits (float32 values for F32)
    bias_type: int | None = None
    q_scale: np.ndarray | None = None  # int8 D: [M] float32 per-row scales
    q_zp: int = 0                      # int8 D: zero point


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def dense(M, N, K, *, seed, a_type=BF16, d_type=BF16, dist="normal", scale=1.0,
          alpha=1.0, beta=0.0, c_dist_scale=1.0, name="") -> Problem:
    """Dense problem.  dist 'uniform' draws U[-1,1]; 'normal' draws N(0, scale^2)."""
    g = _rng(seed)
    if dist == "uniform":
        a = g.uniform(-1.0, 1.0, size=(M, K)).astype(np.float32)
        b = g.uniform(-1.0, 1.0, size=(N, K)).astype(np.float32)
    elif dist == "normal":
        a = (g.standard_normal(size=(M, K), dtype=np.float32) * np.float32(scale))
        b = (g.standard_normal(size=(N, K), dtype=np.float32) * np.float32(scale))
    else:
        raise ValueError(dist)
    p = Problem(M, N, K, a_type, a_type, d_type, _round_bits(a, a_type), _round_bits(b, a_type),
                alpha=alpha, beta=beta, name=name)
    if beta != 0.0:
        c = g.standard_normal(size=(M, N), dtype=np.float32) * np.float32(c_dist_scale)
        p.c_type = d_type
        p.C = _round_bits(c, d_type)
    return p


def config1(seed=1001) -> Problem:
    """fp16 256^3, uniform[-1,1], fp32 D, alpha 1, beta 0."""
    return dense(256, 256, 256, seed=seed, a_type=F16, d_type=F32, dist="uniform", name="C1 fp16 256^3")


def config2(seed=1002, M=4096, N=4096, K=4096) -> Problem:
    """bf16 4096^3, N(0,1)/sqrt(K), C bf16 N(0,1), alpha 1.5, beta 0.5, bf16 D."""
    return dense(M, N, K, seed=seed, a_type=BF16, d_type=BF16, dist="normal",
                 scale=1.0 / np.sqrt(K), alpha=1.5, beta=0.5, name=f"C2 bf16 {M}x{N}x{K}")


def config3(M, seed=1003, N=4096, K=14336) -> Problem:
    """Decode-shaped bf16: M in {1,16,64}, N 4096, K 14336, N(0, 0.02^2), bf16 D."""
    return dense(M, N, K, seed=seed + M, a_type=BF16, d_type=BF16, dist="normal", scale=0.02,
                 name=f"C3 decode M={M}")


def config2_fp8(seed=1002, M=4096, N=4096, K=4096, a_type=E4M3) -> Problem:
    """The dense 4096^3 workload with 8-bit float operands: A and B N(0,1) rounded
    once to E4M3 (or E5M2), C bf16 N(0,1), alpha 1.5/sqrt(K) (the per-tensor
    scale that the bf16 workload folds into its operands), beta 0.5, bf16 D."""
    return dense(M, N, K, seed=seed, a_type=a_type, d_type=BF16, dist="normal", scale=1.0,
                 alpha=1.5 / float(np.sqrt(K)), beta=0.5, name=f"C2-shaped {DTYPE_NAMES[a_type]} {M}x{N}x{K}")


def w4a16(M, N, K, *, seed, group=128, a_type=BF16, d_type=BF16, vlo=0.005, vhi=0.02,
          zero=False, name="") -> Problem:
    """Int4 weights with fp16 per-(group, column) scales; A ~ N(0,1).  zero=True
    adds asymmetric zero points, uniform integers in [-8, 7] per (group, column)."""
    g = _rng(seed)
    a = g.standard_normal(size=(M, K), dtype=np.float32)
    q = g.integers(-8, 8, size=(N, K), dtype=np.int64)
    v = g.uniform(vlo, vhi, size=(K // group, N)).astype(np.float32)
    p = Problem(M, N, K, a_type, S4, d_type, _round_bits(a, a_type), pack_int4(q),
                V=_round_bits(v, F16), v_type=F16, gb=group, name=name or f"W4A16 {M}x{N}x{K}")
    if zero:
        p.Z = g.integers(-8, 8, size=(K // group, N), dtype=np.int64).astype(np.int8)
    return p


def config4(seed=1004, M=128, N=11008, K=4096) -> Problem:
    """W4A16: M 128, K 4096, N 11008, group 128, V uniform[0.005, 0.02] fp16."""
    return w4a16(M, N, K, seed=seed, name="C4 W4A16")


def zipf_counts(tokens: int, experts: int, s: float, seed: int) -> np.ndarray:
    """Top-1 routing counts: i.i.d. draws from a Zipf(s) law truncated to ranks
    1..experts, ranks mapped to experts through a seeded permutation."""
    g = _rng(seed)
    ranks = np.arange(1, experts + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    draws = g.choice(experts, size=tokens, p=p)
    perm = g.permutation(experts)
    return np.bincount(perm[draws], minlength=experts).astype(np.int64)


@dataclasses.dataclass
class GroupedProblem:
    counts: np.ndarray           # tokens per expert
    offsets: np.ndarray          # [E+1] prefix sums (int32)
    N: int
    K: int
    a_type: int
    d_type: int
    A: np.ndarray                # [sum m_e, K] rows sorted by expert
    B: np.ndarray                # [E, N, K]
    alpha: float = 1.0
    beta: float = 0.0
    name: str = ""
    epilogue: int = 0
    bias: np.ndarray | None = None
    bias_type: int | None = None
    q_scale: np.ndarray | None = None
    q_zp: int = 0
    b_type: int | None = None    # None: same as a_type; S4 for int4 experts
    V: np.ndarray | None = None  # [E, K/gb, N] per-expert scales
    v_type: int | None = None
    gb: int = 0
    Z: np.ndarray | None = None  # [E, K/gb, N] int8 zero points (int4 B with V)
    U: np.ndarray | None = None  # [K/ga, sum m_e] per-token scales
    u_type: int | None = None
    ga: int = 0


def grouped_w4a16(counts, N, K, *, seed, group=128, a_type=BF16, zero=False, vlo=0.005, vhi=0.02,
                  name="") -> GroupedProblem:
    """Grouped problem with int4 experts: A ~ N(0,1) [sum m_e, K], B int4 uniform
    in [-8, 7] packed [E, N, K/2], V fp16 uniform[vlo, vhi] per (expert, group,
    column), and with zero=True integer zero points uniform in [-8, 7]."""
    counts = np.asarray(counts, dtype=np.int64)
    E = len(counts)
    g = _rng(seed)
    T = int(counts.sum())
    a = g.standard_normal(size=(T, K), dtype=np.float32)
    q = g.integers(-8, 8, size=(E, N, K), dtype=np.int64)
    v = g.uniform(vlo, vhi, size=(E, K // group, N)).astype(np.float32)
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    gp = GroupedProblem(counts, off, N, K, a_type, BF16, _round_bits(a, a_type), pack_int4(q),
                        name=name or f"grouped W4A16 {E}x{N}x{K}", b_type=S4, V=_round_bits(v, F16), v_type=F16,
                        gb=group)
    if zero:
        gp.Z = g.integers(-8, 8, size=(E, K // group, N), dtype=np.int64).astype(np.int8)
    return gp


def grouped(counts, N, K, *, seed, a_type=BF16, d_type=BF16, a_scale=1.0, b_scale=0.02,
            name="") -> GroupedProblem:
    counts = np.asarray(counts, dtype=np.int64)
    E = len(counts)
    g = _rng(seed)
    T = int(counts.sum())
    a = g.standard_normal(size=(T, K), dtype=np.float32) * np.float32(a_scale)
    b = g.standard_normal(size=(E, N, K), dtype=np.float32) * np.float32(b_scale)
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    return GroupedProblem(counts, off, N, K, a_type, d_type, _round_bits(a, a_type),
                          _round_bits(b, a_type), name=name)


def config5(seed=1005, tokens=4096, experts=8, N=14336, K=4096) -> GroupedProblem:
    """Grouped MoE: 8 experts, 4096 tokens with Zipf(1.2) counts, N 14336, K 4096."""
    counts = zipf_counts(tokens, experts, 1.2, seed)
    return grouped(counts, N, K, seed=seed + 1, name="C5 grouped MoE")


def batched(batch, M, N, K, *, seed, a_type=BF16, d_type=BF16, name="") -> GroupedProblem:
    """Uniform batch: every 'expert' gets M rows (offsets are multiples of M)."""
    return grouped([M] * batch, N, K, seed=seed, a_type=a_type, d_type=d_type, a_scale=1.0,
                   b_scale=1.0 / np.sqrt(K), name=name or f"batched {batch}x{M}x{N}x{K}")


def with_epilogue(p, epilogue, *, seed, bias_type=F32, scale=1.0):
    """Set fused-epilogue flags on a problem; with the bias flag, draw a bias
    of N(0, scale^2) values per output column, stored as bias_type."""
    p.epilogue = epilogue
    if epilogue & 1:
        b = _rng(seed).standard_normal(size=p.N, dtype=np.float32) * np.float32(scale)
        p.bias, p.bias_type = _round_bits(b, bias_type), bias_type
    return p


def with_out_quant(p, scales, zp=0):
    """Make D an int8 output with per-row (per-token) scales and a zero point."""
    p.d_type = S8
    p.q_scale = np.ascontiguousarray(scales, dtype=np.float32)
    p.q_zp = int(zp)
    return p
