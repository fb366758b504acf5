"""Pins for the CPU oracle: every oracle function is checked here against
something other than itself.

* storage decode / RN-even encode / ulp: numpy's float16, torch's bfloat16
  (library routines) over every bit pattern or dense random samples;
* the dense GEMM: numpy float64 matmul on library-decoded inputs (tiny random
  shapes), a pure-Python triple loop (<= 8^3), and closed forms (identity B,
  all-ones operands);
* dequantisation: one-hot A exposes b-hat bit-exactly; with unit scales it
  exposes the raw nibbles, pinned by a hand-made table of the packing reading;
* integer schedules: worked examples under tests/golden/ plus brute-force
  coverage invariants.

A plausible slip in the oracle (a dropped beta term, a transposed operand,
a wrong nibble order or group index, a sign error in decode) fails one of
these.
"""
import itertools
import math
import os
import random
import struct

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import BF16, F16, F32, S4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def lib_decode(dtype, bits):
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float64)
    t = torch.from_numpy(bits.astype(np.int16).view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


# ---- storage formats ---------------------------------------------------------

@pytest.mark.parametrize("dtype", [F16, BF16])
def test_decode_every_pattern(dtype):
    bits = np.arange(65536, dtype=np.uint32)
    got = oracle.decode(dtype, bits)
    want = lib_decode(dtype, bits.astype(np.uint16))
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros decode with their sign
    assert math.copysign(1.0, got[0x8000]) == -1.0


def test_encode_f16_matches_numpy():
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact halfway points between neighbouring fp16 values
        (np.arange(0, 4000, dtype=np.uint16).view(np.float16).astype(np.float64)
         + np.arange(1, 4001, dtype=np.uint16).view(np.float16).astype(np.float64)) / 2,
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001,
         6.1e-5, np.inf, -np.inf],
    ])
    got = oracle.encode_rn(F16, vals).astype(np.uint16)
    want = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_encode_bf16_matches_torch():
    rng = np.random.default_rng(6)
    f = np.concatenate([
        (rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000)).astype(np.float32),
        rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32).view(np.float32),
        np.array([1.00390625, 1.01171875, 3.3895e38, 3.4e38, 1e-40, -1e-42, 0.0, -0.0], dtype=np.float32),
    ])
    f = f[np.isfinite(f)]
    got = oracle.encode_rn(BF16, f.astype(np.float64)).astype(np.uint16)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_ulp_against_neighbours():
    rng = np.random.default_rng(7)
    for dtype in (F16, BF16):
        bits = rng.integers(1, 0x7B00 if dtype == F16 else 0x7F00, 2000).astype(np.uint16)
        vals = lib_decode(dtype, bits)
        nxt = lib_decode(dtype, bits + 1)
        # the spacing above a representable value that is not a power of two
        # equals the ulp of that binade
        keep = (bits & (0x3FF if dtype == F16 else 0x7F)) != 0
        assert np.array_equal(oracle.ulp(dtype, vals)[keep], (nxt - vals)[keep])
    h = np.float16(np.array([1.0, 3.0, 1e-6, 1000.0]))
    assert np.array_equal(oracle.ulp(F16, h.astype(np.float64)), np.spacing(h).astype(np.float64))


# ---- dense GEMM ----------------------------------------------------------------

def _decoded(p):
    a = lib_decode(p.a_type, p.A)
    b = lib_decode(p.b_type, p.B)  # N x K
    return a, b


def _c_values(p):
    if p.c_type == F32:
        return np.asarray(p.C, dtype=np.float32).astype(np.float64)
    return lib_decode(p.c_type, p.C)


def test_dense_matches_numpy_matmul():
    rng = random.Random(11)
    for case in range(40):
        M, N, K = (rng.randint(1, 33) for _ in range(3))
        a_type = rng.choice([F16, BF16])
        d_type = rng.choice([F32, F16, BF16])
        beta = rng.choice([0.0, 0.5, -1.25])
        p = synth.dense(M, N, K, seed=case, a_type=a_type, d_type=d_type, dist="normal",
                        alpha=rng.choice([1.0, 1.5, -0.75]), beta=beta)
        if beta != 0.0 and d_type == F32:
            p.C = np.random.default_rng(case).standard_normal((M, N)).astype(np.float32)
        ref, bound = oracle.gemm(p)
        a, b = _decoded(p)
        want = p.alpha * (a @ b.T)
        wb = abs(p.alpha) * (np.abs(a) @ np.abs(b.T))
        if beta != 0.0:
            c = _c_values(p)
            want = want + beta * c
            wb = wb + np.abs(beta * c)
        np.testing.assert_allclose(ref, want, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(bound, wb, rtol=1e-13, atol=1e-13)


def _py_value(dtype, bits):
    bits = int(bits)
    if dtype == F16:
        return struct.unpack("<e", struct.pack("<H", bits))[0]
    return struct.unpack("<f", struct.pack("<I", bits << 16))[0]


def test_dense_matches_python_triple_loop():
    for case, (M, N, K) in enumerate([(1, 1, 1), (2, 3, 4), (8, 8, 8), (5, 7, 3), (8, 1, 6)]):
        p = synth.dense(M, N, K, seed=100 + case, a_type=BF16 if case % 2 else F16, d_type=BF16,
                        dist="uniform", alpha=1.25, beta=-0.5)
        ref, _ = oracle.gemm(p)
        for i in range(M):
            for j in range(N):
                s = 0.0
                for k in range(K):
                    s += _py_value(p.a_type, p.A[i, k]) * _py_value(p.b_type, p.B[j, k])
                want = 1.25 * s + (-0.5) * _py_value(BF16, p.C[i, j])
                assert ref[i, j] == pytest.approx(want, rel=1e-14, abs=1e-14)


def test_identity_b_closed_form():
    K = 24
    p = synth.dense(13, K, K, seed=3, a_type=F16, d_type=F16, dist="normal", alpha=1.5, beta=0.5)
    one = np.uint16(0x3C00)
    p.B = np.where(np.eye(K, dtype=bool), one, np.uint16(0)).astype(np.uint16)
    ref, _ = oracle.gemm(p)
    a = lib_decode(F16, p.A)
    c = lib_decode(F16, p.C)
    assert np.array_equal(ref, 1.5 * a + 0.5 * c)


@pytest.mark.parametrize("dtype,one", [(F16, 0x3C00), (BF16, 0x3F80)])
def test_all_ones_closed_form(dtype, one):
    M, N, K = 5, 6, 1000
    p = synth.dense(M, N, K, seed=4, a_type=dtype, d_type=F32, alpha=0.75, beta=2.0)
    p.A = np.full((M, K), one, dtype=np.uint16)
    p.B = np.full((N, K), one, dtype=np.uint16)
    p.c_type = F32
    p.C = np.arange(M * N, dtype=np.float32).reshape(M, N)
    ref, bound = oracle.gemm(p)
    want = 0.75 * K + 2.0 * p.C.astype(np.float64)
    assert np.array_equal(ref, want)
    assert np.array_equal(bound, 0.75 * K + 2.0 * np.abs(p.C.astype(np.float64)))


def test_beta_zero_does_not_read_c():
    p = synth.dense(4, 4, 16, seed=9, a_type=BF16, d_type=F16)
    p.beta = 0.0
    p.c_type = F16
    p.C = np.full((4, 4), 0x7E00, dtype=np.uint16)  # NaN everywhere
    ref, _ = oracle.gemm(p)
    assert np.isfinite(ref).all()


# Standard normal CDF at 1, 2 and sqrt(2) (printed in every normal table).
PHI_1, PHI_2, PHI_SQRT2 = 0.8413447460685429, 0.9772498680518208, 0.9213503964748575


def _scalar_problem(x_bits, dtype=BF16):
    """A 1 x 3 x 1 product whose three outputs are the values x_bits decode to."""
    one = 0x3F80 if dtype == BF16 else 0x3C00
    p = synth.dense(1, len(x_bits), 1, seed=0, a_type=dtype, d_type=F32)
    p.A = np.array([[one]], dtype=np.uint16)
    p.B = np.array([[b] for b in x_bits], dtype=np.uint16)
    return p


def test_gelu_closed_forms():
    # GELU(x) = x * Phi(x): x = 1, 2, -1 (bf16 0x3F80, 0x4000, 0xBF80)
    p = synth.with_epilogue(_scalar_problem([0x3F80, 0x4000, 0xBF80]), 4, seed=0)
    ref, bound = oracle.gemm(p)
    assert ref[0] == pytest.approx([PHI_1, 2 * PHI_2, -(1 - PHI_1)], rel=1e-15, abs=1e-16)
    assert np.array_equal(bound[0], 1.129 * np.array([1.0, 2.0, 1.0]))
    # the bound's factor covers the largest slope of x * Phi(x), at x = sqrt 2
    phi = math.exp(-1.0) / math.sqrt(2 * math.pi)
    assert PHI_SQRT2 + math.sqrt(2) * phi < 1.129


def test_relu_bias_order_and_nan():
    # x = -1 (+ bias 2 before the activation gives 1; ReLU first would give 2),
    # x = 3 with bias 2 -> 5; a NaN input stays NaN
    p = synth.with_epilogue(_scalar_problem([0xBF80, 0x4040, 0x7FC0]), 1 | 2, seed=0)
    p.bias, p.bias_type = np.array([2.0, 2.0, 0.0], dtype=np.float32), F32
    ref, bound = oracle.gemm(p)
    assert ref[0][0] == 1.0 and ref[0][1] == 5.0 and math.isnan(ref[0][2])
    assert bound[0][0] == 3.0 and bound[0][1] == 5.0
    p.epilogue = 2
    ref, _ = oracle.gemm(p)
    assert ref[0][0] == 0.0 and ref[0][1] == 3.0


def test_bias_follows_alpha_and_beta():
    # D = act(alpha * acc + beta * c + bias_j); bias broadcast over rows, by column
    p = synth.dense(4, 3, 8, seed=31, a_type=F16, d_type=F16, alpha=1.5, beta=-0.5)
    ref0, b0 = oracle.gemm(p)
    synth.with_epilogue(p, 1, seed=32, bias_type=BF16)
    ref1, b1 = oracle.gemm(p)
    bias = lib_decode(BF16, p.bias)
    assert np.array_equal(ref1, ref0 + bias[None, :])
    assert np.array_equal(b1, b0 + np.abs(bias)[None, :])


def test_output_quantisation_closed_forms():
    # round half to even, saturation, zero point, NaN -> 0, scale per row
    x = np.array([[2.5, 3.5, -2.5, -0.5, 1000.0, -1000.0, float("nan"), 0.49999],
                  [1.0, 1.25, -1.0, 63.5, 64.5, 0.0, 2.0, -3.0]])
    q = oracle.quantize_s8(x, [1.0, 2.0], 0)
    assert q[0].tolist() == [2, 4, -2, 0, 127, -128, 0, 0]
    assert q[1].tolist() == [2, 2, -2, 127, 127, 0, 4, -6]
    q = oracle.quantize_s8(x[1:], [2.0], -3)
    assert q[0].tolist() == [-1, -0.0, -5, 124, 126, -3, 1, -9]


def test_entries_agree_with_full():
    p = synth.dense(37, 29, 40, seed=21, a_type=BF16, d_type=BF16, alpha=1.5, beta=0.5)
    ref, bound = oracle.gemm(p)
    ii = np.array([0, 36, 5, 17, 36])
    jj = np.array([0, 28, 11, 3, 0])
    r, b = oracle.gemm_entries(p, ii, jj)
    assert np.array_equal(r, ref[ii, jj])
    assert np.array_equal(b, bound[ii, jj])


# ---- scale operands and int4 -------------------------------------------------------

def _golden_nibbles():
    rows = []
    with open(os.path.join(GOLDEN, "int4_nibbles.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                h, lo, hi = line.split()
                rows.append((int(h, 16), int(lo), int(hi)))
    return rows


def test_int4_nibble_order_matches_table():
    table = _golden_nibbles()
    packed = np.array([[b for b, _, _ in table]], dtype=np.uint8)
    want = [v for _, lo, hi in table for v in (lo, hi)]
    assert oracle.unpack_int4(packed)[0].tolist() == want
    assert [oracle.int4_at(packed, 0, k) for k in range(len(want))] == want
    # synth's packer is the inverse of the reading
    q = np.array([want], dtype=np.int64)
    assert np.array_equal(synth.pack_int4(q), packed)


def _one_hot_a(M, K, ks, dtype):
    one = 0x3C00 if dtype == F16 else 0x3F80
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), ks] = one
    return A


def test_int4_unit_scale_exposes_raw_nibbles():
    M, N, K = 16, 12, 256
    p = synth.w4a16(M, N, K, seed=31, group=128)
    p.V = np.full_like(p.V, 0x3C00)           # fp16 1.0
    ks = np.random.default_rng(1).integers(0, K, M)
    p.A = _one_hot_a(M, K, ks, BF16)
    ref, _ = oracle.gemm(p)
    q = oracle.unpack_int4(p.B)                # N x K
    assert np.array_equal(ref, q[:, ks].T.astype(np.float64))


def test_int4_dequant_rounding_matches_torch():
    M, N, K = 24, 40, 512
    p = synth.w4a16(M, N, K, seed=32, group=128)
    ks = np.random.default_rng(2).integers(0, K, M)
    p.A = _one_hot_a(M, K, ks, BF16)
    ref, _ = oracle.gemm(p)
    q = oracle.unpack_int4(p.B).astype(np.float32)            # N x K
    v = lib_decode(F16, p.V).astype(np.float32)                # K/128 x N
    prod = q * v[np.arange(K) // 128, :].T                     # exact in fp32
    bhat = torch.from_numpy(prod).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ref, bhat[:, ks].T)


def test_v_scale_on_16bit_b_and_u_scale_on_a():
    # V on a 16-bit B: b-hat = RN_B(b * v); U on A: a-hat = RN_A(a * u).
    M, K, g = 6, 64, 16
    p = synth.dense(M, K, K, seed=41, a_type=F16, d_type=F32, dist="uniform")
    rng = np.random.default_rng(3)
    u = rng.uniform(0.5, 2.0, size=(K // g, M)).astype(np.float32)
    p.U, p.u_type, p.ga = synth._round_bits(u, F16), F16, g
    p.B = np.where(np.eye(K, dtype=bool), np.uint16(0x3C00), np.uint16(0)).astype(np.uint16)
    ref, _ = oracle.gemm(p)
    a = lib_decode(F16, p.A).astype(np.float32)
    uu = lib_decode(F16, p.U).astype(np.float32)[np.arange(K) // g, :].T   # M x K
    want = (a * uu).astype(np.float16).astype(np.float64)
    assert np.array_equal(ref, want)
    # now V on B with A = I
    p2 = synth.dense(K, 8, K, seed=42, a_type=BF16, d_type=F32, dist="uniform")
    p2.A = np.where(np.eye(K, dtype=bool), np.uint16(0x3F80), np.uint16(0)).astype(np.uint16)
    v = rng.uniform(0.5, 2.0, size=(K // g, 8)).astype(np.float32)
    p2.V, p2.v_type, p2.gb = synth._round_bits(v, F16), F16, g
    ref2, _ = oracle.gemm(p2)
    b = lib_decode(BF16, p2.B).astype(np.float32)                           # N x K
    vv = lib_decode(F16, p2.V).astype(np.float32)[np.arange(K) // g, :].T  # N x K
    want2 = torch.from_numpy(b * vv).to(torch.bfloat16).to(torch.float64).numpy().T
    assert np.array_equal(ref2, want2)


# ---- grouped and batched -------------------------------------------------------------

def test_grouped_matches_numpy_per_expert():
    gp = synth.grouped([3, 0, 17, 1, 9], 11, 24, seed=51)
    ref, _ = oracle.grouped(gp)
    a = lib_decode(BF16, gp.A)
    for e in range(5):
        lo, hi = gp.offsets[e], gp.offsets[e + 1]
        b = lib_decode(BF16, gp.B[e])
        np.testing.assert_allclose(ref[lo:hi], a[lo:hi] @ b.T, rtol=1e-13, atol=1e-13)
    ii = np.array([0, 2, 3, 19, 20, 29])
    jj = np.array([10, 0, 5, 6, 1, 2])
    r, _ = oracle.grouped_entries(gp, ii, jj)
    assert np.array_equal(r, ref[ii, jj])


def test_zipf_counts_shape():
    c = synth.zipf_counts(4096, 8, 1.2, 1005)
    assert c.sum() == 4096 and len(c) == 8
    # the largest expert gets the biggest share, roughly 1756/4096 in expectation
    assert 0.35 < c.max() / 4096 < 0.5


# ---- integer schedules ------------------------------------------------------------------

def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.strip() for l in f if l.strip() and not l.startswith("#")]


def test_streamk_plan_worked_examples():
    keys = ["iters_per_tile", "total_tiles", "streamk_tiles", "blocking_tiles", "full_tiles",
            "partial_tiles", "sm_partition_factor"]
    for line in _golden_lines("streamk_plan.txt"):
        args, want = line.split("|")
        plan = oracle.streamk_plan(*map(int, args.split()))
        assert [plan[k] for k in keys] == list(map(int, want.split()))


@pytest.mark.parametrize("m,n,k,bm,bn,bk,sm", [
    (256, 1024, 512, 16, 128, 32, 108), (4096, 16, 14336, 128, 16, 64, 148),
    (1280, 3840, 256, 128, 128, 64, 100), (4096, 4096, 4096, 128, 256, 64, 148),
    (300, 500, 700, 128, 128, 64, 7), (128, 128, 64, 128, 128, 64, 148), (1, 1, 1, 128, 16, 64, 3)])
def test_streamk_covers_every_iteration_once(m, n, k, bm, bn, bk, sm):
    plan = oracle.streamk_plan(m, n, k, bm, bn, bk, sm)
    ipt, T = plan["iters_per_tile"], plan["total_tiles"]
    seen = np.zeros((T, ipt), dtype=np.int64)
    counts = []
    for pid in range(sm):
        segs = oracle.streamk_program_work(plan, pid, sm)
        n_sk = 0
        for t, kb, ke in segs:
            assert 0 <= t < T and 0 <= kb < ke <= ipt
            seen[t, kb:ke] += 1
            if t < plan["streamk_tiles"]:
                n_sk += ke - kb
        counts.append(n_sk)
    assert (seen == 1).all()
    assert max(counts) - min(counts) <= 1


def test_grouped_tile_map_worked_examples():
    for line in _golden_lines("grouped_map.txt"):
        bm, sizes, blocks = line.split("|")
        want = [tuple(map(int, b.split())) for b in blocks.split(";")]
        assert oracle.grouped_tile_map(list(map(int, sizes.split())), int(bm)) == want


@pytest.mark.parametrize("sizes,bm", [([3, 0, 130], 128), ([0, 0, 0, 7], 16), ([1756, 764, 470, 333, 254, 204, 170, 145], 128),
                                      ([128, 128], 128), ([5], 4), ([0, 9, 0, 0, 3, 0], 2)])
def test_grouped_tile_map_covers_rows_once(sizes, bm):
    blocks = oracle.grouped_tile_map(sizes, bm)
    off = np.concatenate([[0], np.cumsum(sizes)])
    seen = np.zeros(int(off[-1]), dtype=np.int64)
    for e, ms, rows in blocks:
        assert 1 <= rows <= bm
        assert off[e] <= ms and ms + rows <= off[e + 1]
        seen[ms:ms + rows] += 1
    assert (seen == 1).all()
    assert len(blocks) == sum(-(-s // bm) for s in sizes)


@pytest.mark.parametrize("k_iters,splits", [(224, 8), (10, 3), (7, 8), (1, 4), (64, 64), (65, 2), (5, 1)])
def test_splitk_ranges_partition(k_iters, splits):
    r = oracle.splitk_ranges(k_iters, splits)
    assert r[0][0] == 0 and r[-1][1] == k_iters
    assert all(a < b for a, b in r)
    assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
    assert len(r) <= splits
    assert len({b - a for a, b in r[:-1]}) <= 1


def test_batched_block_is_a_bijection():
    m_num, n_num, batch = 3, 5, 4
    got = {oracle.batched_block(c, m_num, n_num) for c in range(batch * m_num * n_num)}
    assert got == set(itertools.product(range(batch), range(m_num), range(n_num)))
    assert oracle.batched_block(0, m_num, n_num) == (0, 0, 0)
    assert oracle.batched_block(16, m_num, n_num) == (1, 0, 1)


# ---- 8-bit float operands (DeepGEMM kernel-set blog, sections 1.2 and 6.3) ----

def lib_decode_fp8(dtype, bits):
    f8 = torch.float8_e4m3fn if dtype == oracle.E4M3 else torch.float8_e5m2
    t = torch.from_numpy(np.asarray(bits, dtype=np.uint8).copy()).view(f8)
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("dtype", [oracle.E4M3, oracle.E5M2])
def test_fp8_decode_every_pattern(dtype):
    bits = np.arange(256, dtype=np.uint32)
    got = oracle.decode(dtype, bits)
    want = lib_decode_fp8(dtype, bits.astype(np.uint8))
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert math.copysign(1.0, got[0x80]) == -1.0


def test_fp8_format_closed_forms():
    # values fixed by the two formats' definitions (sign, exponent with bias 7
    # or 15, 3 or 2 mantissa bits; E4M3 keeps only all-ones as NaN and has no
    # infinity; E5M2 has IEEE infinities and NaNs)
    e4 = {0x38: 1.0, 0x7E: 448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0xC4: -3.0,
          0x77: 240.0, 0x78: 256.0}
    e5 = {0x3C: 1.0, 0x7B: 57344.0, 0x04: 2.0 ** -14, 0x01: 2.0 ** -16, 0x03: 3 * 2.0 ** -16, 0xC2: -3.0,
          0x7C: math.inf, 0xFC: -math.inf}
    for bits, v in e4.items():
        assert oracle.decode(oracle.E4M3, [bits])[0] == v, hex(bits)
    for bits, v in e5.items():
        assert oracle.decode(oracle.E5M2, [bits])[0] == v, hex(bits)
    assert np.isnan(oracle.decode(oracle.E4M3, [0x7F, 0xFF])).all()
    assert not np.isnan(oracle.decode(oracle.E4M3, [0x7C, 0x7D, 0x7E])).any()  # exponent all ones, finite
    assert np.isnan(oracle.decode(oracle.E5M2, [0x7D, 0x7E, 0x7F, 0xFF])).all()


@pytest.mark.parametrize("dtype", [oracle.E4M3, oracle.E5M2])
def test_fp8_dense_matches_numpy_matmul(dtype):
    rng = random.Random(31 + dtype)
    for case in range(12):
        M, N, K = (rng.randint(1, 40) for _ in range(3))
        beta = rng.choice([0.0, 0.5])
        p = synth.dense(M, N, K, seed=200 + case, a_type=dtype, d_type=BF16, dist="normal",
                        alpha=rng.choice([1.0, 0.03125, -0.75]), beta=beta)
        ref, bound = oracle.gemm(p)
        a, b = lib_decode_fp8(dtype, p.A), lib_decode_fp8(dtype, p.B)
        want = p.alpha * (a @ b.T)
        wb = abs(p.alpha) * (np.abs(a) @ np.abs(b.T))
        if beta != 0.0:
            c = lib_decode(BF16, p.C)
            want, wb = want + beta * c, wb + np.abs(beta * c)
        np.testing.assert_allclose(ref, want, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(bound, wb, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("dtype,one", [(oracle.E4M3, 0x38), (oracle.E5M2, 0x3C)])
def test_fp8_identity_b_closed_form(dtype, one):
    K = 40
    p = synth.dense(9, K, K, seed=5, a_type=dtype, d_type=BF16, dist="normal", alpha=1.5, beta=0.5)
    p.B = np.where(np.eye(K, dtype=bool), np.uint8(one), np.uint8(0)).astype(np.uint8)
    ref, _ = oracle.gemm(p)
    assert np.array_equal(ref, 1.5 * lib_decode_fp8(dtype, p.A) + 0.5 * lib_decode(BF16, p.C))


# ---- asymmetric int4: a zero point per (K-group, column) ------------------------

def test_zero_point_byte_rule():
    # a 4-bit zero point stored one per byte: the low nibble, two's complement
    table = {0x00: 0, 0x07: 7, 0x08: -8, 0x0F: -1, 0x09: -7, 0xF3: 3, 0x80: 0, 0x7C: -4}
    Z = np.array([list(table)], dtype=np.uint8).view(np.int8)
    assert [oracle.zero_at(Z, 0, n) for n in range(len(table))] == list(table.values())


def test_zero_point_unit_scale_exposes_q_minus_z():
    M, N, K, g = 16, 12, 256, 64
    p = synth.w4a16(M, N, K, seed=33, group=g, zero=True)
    p.V = np.full_like(p.V, 0x3C00)           # fp16 1.0
    ks = np.random.default_rng(4).integers(0, K, M)
    p.A = _one_hot_a(M, K, ks, BF16)
    ref, _ = oracle.gemm(p)
    q = oracle.unpack_int4(p.B)                # N x K
    z = p.Z.astype(np.int64)[np.arange(K) // g, :].T   # N x K
    assert np.array_equal(ref, (q - z)[:, ks].T.astype(np.float64))


@pytest.mark.parametrize("a_type", [BF16, F16])
def test_zero_point_dequant_rounding_matches_torch(a_type):
    M, N, K = 24, 40, 512
    p = synth.w4a16(M, N, K, seed=34, group=128, zero=True, a_type=a_type)
    ks = np.random.default_rng(5).integers(0, K, M)
    p.A = _one_hot_a(M, K, ks, a_type)
    ref, _ = oracle.gemm(p)
    q = oracle.unpack_int4(p.B).astype(np.float32)                          # N x K
    z = p.Z.astype(np.float32)[np.arange(K) // 128, :].T
    v = lib_decode(F16, p.V).astype(np.float32)[np.arange(K) // 128, :].T  # N x K
    prod = (q - z) * v                                                      # exact in fp32
    tdt = torch.bfloat16 if a_type == BF16 else torch.float16
    bhat = torch.from_numpy(prod).to(tdt).to(torch.float64).numpy()
    assert np.array_equal(ref, bhat[:, ks].T)


def test_zero_points_of_zero_are_symmetric():
    p = synth.w4a16(9, 20, 256, seed=35, group=128, zero=True)
    p.Z = np.zeros_like(p.Z)
    r1, b1 = oracle.gemm(p)
    p.Z = None
    r2, b2 = oracle.gemm(p)
    assert np.array_equal(r1, r2) and np.array_equal(b1, b2)


def test_grouped_w4a16_matches_numpy_per_expert():
    # per-expert V and zero points: each expert's b-hat rounded by torch from
    # the exact fp32 product, then a numpy float64 matmul per expert
    gp = synth.grouped_w4a16([5, 0, 17, 9], 24, 256, seed=36, group=64, zero=True)
    ref, bound = oracle.grouped(gp)
    a = lib_decode(BF16, gp.A)
    for e in range(4):
        lo, hi = int(gp.offsets[e]), int(gp.offsets[e + 1])
        if hi == lo:
            continue
        q = oracle.unpack_int4(gp.B[e]).astype(np.float32)                       # N x K
        z = gp.Z[e].astype(np.float32)[np.arange(256) // 64, :].T
        v = lib_decode(F16, gp.V[e]).astype(np.float32)[np.arange(256) // 64, :].T
        bhat = torch.from_numpy((q - z) * v).to(torch.bfloat16).to(torch.float64).numpy()
        np.testing.assert_allclose(ref[lo:hi], a[lo:hi] @ bhat.T, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(bound[lo:hi], np.abs(a[lo:hi]) @ np.abs(bhat.T), rtol=1e-13, atol=1e-13)
