"""GPU parity of the 8-bit float input path (E4M3 / E5M2 operands, the FP8
inputs of the DeepGEMM kernel-set blog, sections 1.2 and 6.3) against the CPU
oracle: tcgen05.mma.kind::f8f6f4 with fp32 accumulation in TMEM, through
every tile width and schedule of the single-CTA and CTA-pair kernels, the
swapped-operand decode path, batched and grouped problems, ragged tails in
all three dimensions, and the C2-shaped problem at full size on sampled
outputs.  Every product of two 8-bit floats is exact in fp32, so the
tolerance is the one every parity test uses."""
import numpy as np
import pytest
import torch

import oracle
import quantized_gemm_tcgen05_gb300 as qg
import synth
from gpu_helpers import Lib, assert_close, dev_bits, op, run_grouped, run_problem, sample_indices

pytestmark = pytest.mark.gpu

FP8 = [synth.E4M3, synth.E5M2]


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


def _check(lib, p, o=None, what=""):
    rc, D = run_problem(lib, p, o)
    assert rc == 0, f"{what}: {qg.gemm_status_string(rc)}"
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, what)
    assert qg.gemm_device_status(lib.h, qg.current_stream()) == 0
    return D


@pytest.mark.parametrize("dtype", FP8)
def test_fp8_one_hot_layout(lib, dtype):
    # A[i][k] = 1 at k = (5i) % K: D[i][j] = B[(5i) % K][j] exactly, which pins
    # the placement of 8-bit operands in the 128-element K-steps
    M, N, K = 128, 256, 256
    one = 0x38 if dtype == synth.E4M3 else 0x3C
    p = synth.dense(M, N, K, seed=2, a_type=dtype, d_type=synth.F32, dist="normal")
    A = np.zeros((M, K), dtype=np.uint8)
    A[np.arange(M), (5 * np.arange(M)) % K] = one
    p.A = A
    D = _check(lib, p, what="fp8 one-hot")
    ref, _ = oracle.gemm(p)
    assert np.array_equal(D.double().cpu().numpy(), ref)


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("d_type", [synth.BF16, synth.F16, synth.F32])
@pytest.mark.parametrize("shape", [(200, 328, 528), (64, 1024, 2048), (1, 300, 1040), (520, 700, 1024)])
def test_fp8_automatic_dispatch(lib, dtype, d_type, shape):
    M, N, K = shape
    p = synth.dense(M, N, K, seed=M + N + K + dtype, a_type=dtype, d_type=d_type, dist="normal", alpha=0.125,
                    beta=0.5 if d_type != synth.F32 else 0.0)
    _check(lib, p, what=f"fp8 {shape} -> {d_type}")


KERNELS = ["umma_bn16_swap/dp", "umma_bn32_swap/splitk3", "umma_bn64_swap/streamk", "umma_bn128_swap/dp",
           "umma_bn16/dp", "umma_bn64/dp", "umma_bn128/splitk2", "umma_bn192/streamk", "umma_bn224/dp",
           "umma_bn256/streamk", "umma2_bn128/dp", "umma2_bn224/streamk", "umma2_bn256/dp"]


@pytest.mark.parametrize("kernel", KERNELS)
# K a multiple of 128 copies several K-steps per box; 720 ends on a partial K-step
@pytest.mark.parametrize("K", [720, 1024])
def test_fp8_every_registered_kernel(lib, kernel, K, monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_KERNEL", kernel)
    M = 70 if "_swap" in kernel else 300
    p = synth.dense(M, 520, K, seed=len(kernel) + K, a_type=synth.E4M3, d_type=synth.BF16, alpha=0.25, beta=0.5,
                    dist="normal")
    _check(lib, p, what=f"{kernel} K={K}")
    assert qg.gemm_last_choice(lib.h) == kernel


def test_fp8_pair_kernel_many_waves(lib, monkeypatch):
    # 10 x 11 = 110 tiles of 256 x 224 on 76 clusters: every cluster reuses its
    # accumulators and turns its ring phases over, element by element
    monkeypatch.setenv("GEMM_FORCE_KERNEL", "umma2_bn224/dp")
    p = synth.dense(2560, 2304, 256, seed=91, a_type=synth.E4M3, d_type=synth.BF16, alpha=0.5, beta=0.5,
                    dist="normal")
    _check(lib, p, what="fp8 pair, many waves")


def test_fp8_batched(lib):
    gp = synth.batched(4, 192, 264, 640, seed=12, a_type=synth.E4M3)
    A = dev_bits(gp.A, gp.a_type).view(4, 192, 640)
    B = dev_bits(gp.B, gp.a_type)
    D = torch.full((4, 192, 264), float("nan"), dtype=torch.bfloat16, device="cuda")
    L = lib
    rc = qg.gemm_run(L.h, op(), 1.0, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B), qg.col_major_from_nk(B),
                     None, None, 0.0, None, None, qg.ptr(D), qg.row_major(D), L.ws.c, qg.current_stream())
    torch.cuda.synchronize()
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.grouped(gp)
    assert_close(D.reshape(-1, 264).double().cpu().numpy(), ref, bound, synth.BF16, "fp8 batched")


@pytest.mark.parametrize("counts", [[3, 0, 300, 0, 77, 129], [512, 512, 0, 1]])
def test_fp8_grouped(lib, counts):
    gp = synth.grouped(counts, 384, 512, seed=sum(counts), a_type=synth.E4M3, b_scale=0.5)
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.grouped(gp)
    assert_close(D.double().cpu().numpy(), ref, bound, synth.BF16, f"fp8 grouped {counts}")


def test_fp8_config2_shape_full_sampled(lib):
    p = synth.config2_fp8()
    rc, D = run_problem(lib, p)
    assert rc == 0, qg.gemm_status_string(rc)
    ii, jj = sample_indices(p.M, p.N, 2000, seed=15)
    ref, bound = oracle.gemm_entries(p, ii, jj)
    assert_close(D.double().cpu().numpy()[ii, jj], ref, bound, p.d_type, "C2-shaped e4m3 (sampled)")


def test_fp8_rejections(lib):
    # mixed 8-bit formats, an 8-bit A with a 16-bit B, scale operands on 8-bit
    # operands, and a row stride that is not a multiple of 16 bytes
    p = synth.dense(64, 64, 128, seed=3, a_type=synth.E4M3, d_type=synth.BF16)
    A, B = dev_bits(p.A, p.a_type), dev_bits(p.B, p.b_type)
    D = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    st = qg.current_stream()

    def run(Ad, Bd, V=None, Vd=None, o=None):
        return qg.gemm_run(lib.h, o or op(), 1.0, qg.ptr(A), Ad, None, None, qg.ptr(B), Bd, qg.ptr(V), Vd, 0.0, None,
                           None, qg.ptr(D), qg.row_major(D), lib.ws.c, st)

    good_a, good_b = qg.row_major(A), qg.col_major_from_nk(B)
    assert run(good_a, good_b) == 0
    mixed = qg.layout(qg.GEMM_E5M2, qg.GEMM_COL_MAJOR, 128, 64, 128)
    assert run(good_a, mixed) == qg.GEMM_ERR_UNSUPPORTED
    b16 = qg.layout(qg.GEMM_BF16, qg.GEMM_COL_MAJOR, 128, 64, 128)
    assert run(good_a, b16) == qg.GEMM_ERR_UNSUPPORTED
    V = torch.ones(1, 64, dtype=torch.float16, device="cuda")
    assert run(good_a, good_b, V, qg.layout(qg.GEMM_F16, qg.GEMM_ROW_MAJOR, 1, 64, 64), op(gb=128)) == \
        qg.GEMM_ERR_UNSUPPORTED
    odd = qg.layout(qg.GEMM_E4M3, qg.GEMM_ROW_MAJOR, 60, 120, 120)  # 120-byte rows
    assert qg.gemm_run(lib.h, op(), 1.0, qg.ptr(A), odd, None, None, qg.ptr(B),
                       qg.layout(qg.GEMM_E4M3, qg.GEMM_COL_MAJOR, 120, 64, 128), None, None, 0.0, None, None,
                       qg.ptr(D), qg.layout(qg.GEMM_BF16, qg.GEMM_ROW_MAJOR, 60, 64, 64), lib.ws.c, st) == \
        qg.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
