"""GPU parity of asymmetric int4 weights (a zero point per (K-group, column)
that advances with the V scales, "InternLM Lmdeploy Gemm MainloopSm80V2",
section Description) and of grouped (MoE) problems with U/V scale operands
and int4 experts (TileLang tutorial "gemm_variants.py", section
gemm_grouped, with the scale operands of the Gemm interface's Run).

The dequantised operand is checked bit-exactly through a one-hot A with an
fp32 D: with unit scales D = q - z exposes the nibble and zero-point reading
on the device.  Whole products are checked against the oracle element by
element under the usual tolerance; the MoE-sized problem on sampled outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_gemm_tcgen05_gb300 as qg
import synth
from gpu_helpers import Lib, assert_close, dev_bits, op, run_grouped, run_problem, sample_indices, zero_rows

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


# M = 1 takes the small-M streaming kernel, 5 and 40 the swapped tensor-core
# path (int4 operand on the 128-row side), 128 and 200 the plain one
@pytest.mark.parametrize("M", [1, 5, 40, 128, 200])
@pytest.mark.parametrize("a_type", [synth.BF16, synth.F16])
@pytest.mark.parametrize("group", [32, 128])
def test_zero_point_unit_scale_exposes_q_minus_z(lib, M, a_type, group):
    N, K = 192, 512
    p = synth.w4a16(M, N, K, seed=M + group, group=group, a_type=a_type, d_type=synth.F32, zero=True)
    p.V = np.full_like(p.V, 0x3C00)  # fp16 1.0
    p.A = _one_hot(M, K, M + 7, a_type)
    rc, D = run_problem(lib, p)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, _ = oracle.gemm(p)
    assert np.array_equal(D.double().cpu().numpy(), ref), qg.gemm_last_choice(lib.h)


@pytest.mark.parametrize("M", [1, 16, 128])
@pytest.mark.parametrize("group", [64, 128])
def test_zero_point_dequant_bit_exact(lib, M, group):
    N, K = 320, 512
    p = synth.w4a16(M, N, K, seed=3 * M + group, group=group, d_type=synth.F32, zero=True)
    p.A = _one_hot(M, K, group + M, synth.BF16)
    rc, D = run_problem(lib, p)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, _ = oracle.gemm(p)
    assert np.array_equal(D.double().cpu().numpy(), ref), qg.gemm_last_choice(lib.h)


@pytest.mark.parametrize("M", [1, 2, 16, 128])
def test_zero_point_w4a16_workload_shape(lib, M):
    # the W4A16 workload's N, K and group with zero points, element by element
    p = synth.w4a16(M, 11008, 4096, seed=1004 + M, group=128, zero=True)
    rc, D = run_problem(lib, p)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"W4A16 + zero points M={M}")


@pytest.mark.parametrize("sched", ["splitk3", "streamk"])
def test_zero_point_split_schedules(lib, sched):
    p = synth.w4a16(96, 640, 1024, seed=55, group=64, zero=True)
    o = op(gb=64, splitk=3) if sched == "splitk3" else op(gb=64, streamk=1)
    rc, D = run_problem(lib, p, o)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"zero points {sched}")


def test_zero_point_rejections(lib):
    p = synth.w4a16(64, 128, 256, seed=5, group=128, zero=True)
    A, B = dev_bits(p.A, p.a_type), dev_bits(p.B, p.b_type)
    V = dev_bits(p.V, p.v_type)
    Z, ldz, _ = zero_rows(p.Z)
    D = torch.empty(64, 128, dtype=torch.bfloat16, device="cuda")
    st = qg.current_stream()
    Vd = qg.layout(qg.GEMM_F16, qg.GEMM_ROW_MAJOR, 2, 128, 128)

    def run(o, with_v=True):
        return qg.gemm_run(lib.h, o, 1.0, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B),
                           qg.col_major_from_nk(B, k=256, type_=qg.GEMM_S4), qg.ptr(V) if with_v else None,
                           Vd if with_v else None, 0.0, None, None, qg.ptr(D), qg.row_major(D), lib.ws.c, st)

    o = op(gb=128)
    o.b_zero, o.b_zero_ld = qg.ptr(Z), ldz
    assert run(o) == 0
    assert run(o, with_v=False) == qg.GEMM_ERR_INVALID_ARG       # zero points need V
    o.b_zero_ld = 136                                             # not a multiple of 16 bytes
    assert run(o) == qg.GEMM_ERR_INVALID_ARG
    o.b_zero_ld, o.b_zero = ldz, qg.ptr(Z) + 8                    # misaligned base
    assert run(o) == qg.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()


# ---- grouped problems with scale operands -------------------------------------

@pytest.mark.parametrize("counts", [[3, 0, 300, 0, 77, 129], [256, 1, 0, 511]])
@pytest.mark.parametrize("zero", [False, True])
@pytest.mark.parametrize("group", [64, 128])
def test_grouped_w4a16(lib, counts, zero, group):
    gp = synth.grouped_w4a16(counts, 384, 512, seed=sum(counts) + group, group=group, zero=zero)
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    assert qg.gemm_last_choice(lib.h).startswith("umma_dq_grouped")
    ref, bound = oracle.grouped(gp)
    assert_close(D.double().cpu().numpy(), ref, bound, gp.d_type, f"grouped W4A16 {counts} zero={zero}")


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_grouped_w4a16_dequant_bit_exact(lib, bn, monkeypatch):
    # one-hot token rows with an fp32 D expose each expert's b-hat exactly,
    # through every tile width the kernel is built for
    monkeypatch.setenv("GEMM_FORCE_KERNEL", f"umma_dq_grouped_bn{bn}/dp")
    gp = synth.grouped_w4a16([40, 0, 130, 7], 320, 384, seed=bn, group=64, zero=True)
    gp.d_type = synth.F32
    gp.A = _one_hot(int(gp.offsets[-1]), gp.K, bn, synth.BF16)
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    assert qg.gemm_last_choice(lib.h) == f"umma_dq_grouped_bn{bn}/dp"
    ref, _ = oracle.grouped(gp)
    assert np.array_equal(D.double().cpu().numpy(), ref)


def test_grouped_16bit_b_with_u_and_v(lib):
    # 16-bit experts scaled by per-expert V, token rows scaled by U
    counts = [100, 0, 200, 33]
    gp = synth.grouped(counts, 256, 512, seed=77, b_scale=0.05)
    rng = np.random.default_rng(8)
    T, E = int(sum(counts)), len(counts)
    gp.V, gp.v_type, gp.gb = synth._round_bits(rng.uniform(0.5, 2.0, (E, 512 // 64, 256)), synth.F16), synth.F16, 64
    gp.U, gp.u_type, gp.ga = synth._round_bits(rng.uniform(0.5, 2.0, (512 // 128, T)), synth.BF16), synth.BF16, 128
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.grouped(gp)
    assert_close(D.double().cpu().numpy(), ref, bound, gp.d_type, "grouped 16-bit B with U and V")


def test_grouped_w4a16_moe_shape_sampled(lib):
    # the MoE workload's routing and sizes with int4 experts and zero points
    counts = synth.zipf_counts(4096, 8, 1.2, 1005)
    gp = synth.grouped_w4a16(counts, 14336, 4096, seed=1006, group=128, zero=True)
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    ii, jj = sample_indices(int(gp.offsets[-1]), gp.N, 1500, seed=9)
    ref, bound = oracle.grouped_entries(gp, ii, jj)
    assert_close(D.double().cpu().numpy()[ii, jj], ref, bound, gp.d_type, "grouped W4A16 MoE (sampled)")
