"""GPU parity of the scaled-operand path: int4 weights dequantised in the
mainloop (W4A16), group-wise U scales on A and V scales on 16-bit B.

The dequantised operand is checked bit-exactly through a one-hot A with an
fp32 D (D[i][j] = B-hat[k_i][j]); with unit scales that exposes the raw
nibbles and pins their order on the device.  Whole products are checked
against the oracle under the usual tolerance.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import Lib, assert_close, op, run_problem, sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


def _one_hot(M, K, seed, dtype):
    ks = np.random.default_rng(seed).integers(0, K, M)
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), ks] = 0x3F80 if dtype == synth.BF16 else 0x3C00
    return A


@pytest.mark.parametrize("a_type", [synth.BF16, synth.F16])
@pytest.mark.parametrize("M", [5, 128, 200])
def test_int4_unit_scales_expose_nibbles(lib, a_type, M):
    N, K = 192, 256
    p = synth.w4a16(M, N, K, seed=M, group=128, a_type=a_type, d_type=synth.F32)
    p.V = np.full_like(p.V, 0x3C00)  # fp16 1.0
    p.A = _one_hot(M, K, M, a_type)
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, _ = oracle.gemm(p)
    assert np.array_equal(D.double().cpu().numpy(), ref)


@pytest.mark.parametrize("group", [32, 64, 128])
def test_int4_dequant_bit_exact(lib, group):
    M, N, K = 128, 320, 512
    p = synth.w4a16(M, N, K, seed=group, group=group, d_type=synth.F32)
    p.A = _one_hot(M, K, group + 1, synth.BF16)
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, _ = oracle.gemm(p)
    assert np.array_equal(D.double().cpu().numpy(), ref)


@pytest.mark.parametrize("M", [1, 16, 64, 128, 130])
@pytest.mark.parametrize("N", [64, 200])
def test_w4a16_small(lib, M, N):
    for K, group in ((128, 128), (384, 128), (256, 32)):
        p = synth.w4a16(M, N, K, seed=M * N + K, group=group)
        rc, D = run_problem(lib, p)
        assert rc == 0
        ref, bound = oracle.gemm(p)
        assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"W4A16 {M}x{N}x{K} g{group}")


@pytest.mark.parametrize("group,K", [(8, 256), (16, 448), (32, 224), (64, 832), (192, 768), (256, 1280)])
@pytest.mark.parametrize("sched", ["auto", "streamk", "splitk3"])
def test_int4_groups_and_slot_edges(lib, group, K, sched):
    # int4 rows and their scale rows arrive four K-steps at a time: split-K
    # and stream-K units start and end inside such a chunk, groups under 64
    # need several scale rows per K-step, a group of 192 straddles chunks,
    # and K = 224 ends half-way through a K-step
    M, N = 128, 384
    p = synth.w4a16(M, N, K, seed=group + K, group=group)
    o = {"auto": op(gb=group), "streamk": op(streamk=1, gb=group), "splitk3": op(splitk=3, gb=group)}[sched]
    rc, D = run_problem(lib, p, o)
    assert rc == 0, f"status {rc}"
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"W4A16 g{group} K{K} {sched}")


@pytest.mark.parametrize("M", [1, 40])
def test_int4_swapped_groups(lib, M):
    # decode-sized M: the int4 weights are the 128-row X operand
    for group, K in ((8, 320), (192, 576), (64, 4096 + 64)):
        p = synth.w4a16(M, 520, K, seed=M + group, group=group)
        rc, D = run_problem(lib, p, op(gb=group))
        assert rc == 0
        ref, bound = oracle.gemm(p)
        assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"W4A16 swapped M{M} g{group} K{K}")


def test_config4_full(lib):
    p = synth.config4()
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "C4 W4A16")


@pytest.mark.parametrize("sched", ["splitk4", "streamk", "unsplit"])
def test_config4_schedules_sampled(lib, sched):
    p = synth.config4()
    o = {"splitk4": op(splitk=4, gb=128), "streamk": op(streamk=1, gb=128), "unsplit": op(splitk=1, gb=128)}[sched]
    rc, D = run_problem(lib, p, o)
    assert rc == 0
    ii, jj = sample_indices(p.M, p.N, 3000, seed=3)
    ref, bound = oracle.gemm_entries(p, ii, jj)
    assert_close(D.double().cpu().numpy()[ii, jj], ref, bound, p.d_type, f"C4 {sched}")


def test_u_scale_on_a(lib):
    M, N, K, g = 150, 130, 256, 32
    p = synth.dense(M, N, K, seed=61, a_type=synth.F16, d_type=synth.F32, dist="uniform")
    u = np.random.default_rng(1).uniform(0.25, 4.0, size=(K // g, M)).astype(np.float32)
    p.U, p.u_type, p.ga = synth._round_bits(u, synth.F16), synth.F16, g
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "U on A")


def test_v_scale_on_16bit_b_and_both(lib):
    M, N, K, g = 100, 300, 320, 64
    p = synth.dense(M, N, K, seed=62, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.1,
                    alpha=1.5, beta=0.5)
    rng = np.random.default_rng(2)
    v = rng.uniform(0.5, 2.0, size=(K // g, N)).astype(np.float32)
    p.V, p.v_type, p.gb = synth._round_bits(v, synth.BF16), synth.BF16, g
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "V on B")
    u = rng.uniform(0.5, 2.0, size=(K // 32, M)).astype(np.float32)
    p.U, p.u_type, p.ga = synth._round_bits(u, synth.BF16), synth.BF16, 32
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "U and V")


def test_int4_without_scales(lib):
    M, N, K = 64, 128, 192
    p = synth.w4a16(M, N, K, seed=70, group=64)
    p.V = None
    p.v_type = None
    p.gb = 0
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "int4 no V")


def test_scale_layout_rules(lib):
    import quantized_gemm_tcgen05_gb300 as qg
    import torch
    M, N, K = 64, 128, 256
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    V = torch.ones(K // 64, N + 8, dtype=torch.bfloat16, device="cuda")

    def call(gb, ldv, vptr=None):
        Vd = qg.layout(qg.GEMM_BF16, qg.GEMM_ROW_MAJOR, K // (gb or 64), N, ldv)
        return qg.gemm_run(lib.h, op(gb=gb), 1.0, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B),
                           qg.col_major_from_nk(B), vptr or qg.ptr(V), Vd, 0.0, None, None, qg.ptr(D),
                           qg.row_major(D), lib.ws.c, qg.current_stream())

    assert call(64, N + 8) == 0
    assert call(64, N + 3) == qg.GEMM_ERR_INVALID_ARG         # ld not a multiple of 16 bytes
    assert call(64, N + 8, qg.ptr(V) + 2) == qg.GEMM_ERR_INVALID_ARG
    assert call(48, N + 8) == qg.GEMM_ERR_INVALID_ARG          # neither divides nor is a multiple of 64
    assert call(0, N + 8) == qg.GEMM_ERR_INVALID_ARG           # V given without a group size
    torch.cuda.synchronize()
