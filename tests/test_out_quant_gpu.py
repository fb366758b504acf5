"""GPU parity of the fused output quantisation: an int8 D receives
round(x * scale[row] + zp) with per-row (per-token) scales, against the
oracle's pre-rounding values.  Each code must equal the oracle's code unless
a rounding boundary lies within the fp32 value's tolerance, where either
neighbour is accepted.  Covers the register epilogue (whole tiles, split-K,
stream-K), swapped operands, the small-M kernel, the dequantising kernel,
grouped experts, the fused bias / GELU before it, saturation, and the
argument checks.
"""
import numpy as np
import pytest
import torch

import quantized_gemm_tcgen05_gb300 as qg
import oracle
import synth
from gpu_helpers import Lib, assert_quant, op, run_grouped, run_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


def _row_scales(ref, target, seed):
    """Scales mapping each row's largest value to about +-target codes."""
    m = np.nanmax(np.abs(ref), axis=1) + 1e-6
    return (target / m * np.random.default_rng(seed).uniform(0.7, 1.3, size=ref.shape[0])).astype(np.float32)


def _check(lib, p, target=100.0, zp=0, o=None, what=""):
    ref, bound = oracle.gemm(p)
    synth.with_out_quant(p, _row_scales(ref, target, seed=p.M + p.N), zp)
    rc, D = run_problem(lib, p, o)
    assert rc == 0, qg.gemm_status_string(rc)
    ambiguous = assert_quant(D.cpu().numpy(), ref, bound, p.q_scale, zp, f"{what} -> {qg.gemm_last_choice(lib.h)}")
    assert ambiguous < 0.25 * D.numel() + 4  # the band is narrow: most codes are pinned exactly
    return D


@pytest.mark.parametrize("zp", [0, -7])
@pytest.mark.parametrize("shape", [(200, 384, 320), (130, 100, 256), (1000, 1000, 64)])
def test_dense(lib, shape, zp):
    M, N, K = shape
    p = synth.dense(M, N, K, seed=sum(shape), a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.1,
                    alpha=1.5)
    _check(lib, p, zp=zp, what=f"dense {shape}")


@pytest.mark.parametrize("kernel", ["umma_bn128/splitk3", "umma_bn256/streamk", "umma2_bn224/dp"])
def test_schedules(lib, kernel, monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_KERNEL", kernel)
    p = synth.dense(512, 600, 640, seed=20, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.05)
    _check(lib, p, zp=3, what=kernel)
    assert qg.gemm_last_choice(lib.h) == kernel


@pytest.mark.parametrize("M", [1, 16, 64])
def test_decode_and_w4a16(lib, M):
    p = synth.dense(M, 1000, 1024, seed=30 + M, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.05)
    _check(lib, p, what=f"decode M={M}")
    q = synth.w4a16(M, 520, 512, seed=40 + M, group=128)
    _check(lib, q, zp=-2, what=f"W4A16 M={M}")


def test_fused_bias_gelu_then_quantise(lib):
    p = synth.dense(128, 256, 256, seed=50, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.1)
    synth.with_epilogue(p, qg.GEMM_EPILOGUE_BIAS | qg.GEMM_EPILOGUE_GELU, seed=51)
    _check(lib, p, zp=5, what="bias+GELU")


def test_saturation(lib):
    # scales large enough that most codes clip at -128 / 127
    p = synth.dense(64, 128, 64, seed=60, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.5)
    D = _check(lib, p, target=2000.0, what="saturation")
    d = D.cpu().numpy()
    assert (d == 127).sum() > 0.2 * d.size and (d == -128).sum() > 0.2 * d.size


def test_grouped(lib):
    gp = synth.grouped([3, 0, 130, 300], 600, 256, seed=12)
    ref, bound = oracle.grouped(gp)
    gp.d_type, gp.q_scale, gp.q_zp = synth.S8, _row_scales(ref, 100.0, seed=5), 1
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    assert_quant(D.cpu().numpy(), ref, bound, gp.q_scale, 1, "grouped")


def test_argument_checks(lib):
    p = synth.dense(64, 64, 64, seed=14, a_type=synth.BF16, d_type=synth.BF16)
    scales = torch.ones(64, dtype=torch.float32, device="cuda")
    host = torch.ones(64, dtype=torch.float32)
    D = torch.zeros(64, 64, dtype=torch.int8, device="cuda")
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.int8, device="cuda")

    def call(ptr, beta=0.0):
        o = op()
        o.out_scale = ptr
        return qg.gemm_run(lib.h, o, 1.0, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B), qg.col_major_from_nk(B),
                           None, None, beta, qg.ptr(C) if beta else None, qg.row_major(C) if beta else None,
                           qg.ptr(D), qg.row_major(D), lib.ws.c, qg.current_stream())

    assert call(qg.ptr(scales)) == qg.GEMM_OK
    assert call(None) == qg.GEMM_ERR_INVALID_ARG
    assert call(qg.ptr(scales) + 2) == qg.GEMM_ERR_INVALID_ARG
    assert call(qg.ptr(host)) == qg.GEMM_ERR_INVALID_ARG
    assert call(qg.ptr(scales), beta=1.0) == qg.GEMM_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(D.abs().sum()) == 0  # zero operands quantise to the zero point 0
