"""GPU parity of the fused epilogue (bias per output column, then ReLU or
GELU) against the oracle, through every path that writes D: the TMA and the
register epilogue of the 1-CTA kernel, the CTA pair, swapped operands,
split-K and stream-K fix-ups, grouped experts, the dequantising kernel, the
small-M streaming kernel and the K = 0 path; plus the argument checks.
"""
import numpy as np
import pytest
import torch

import quantized_gemm_tcgen05_gb300 as qg
import oracle
import synth
from gpu_helpers import Lib, assert_close, op, run_grouped, run_problem

pytestmark = pytest.mark.gpu

BIAS, RELU, GELU = qg.GEMM_EPILOGUE_BIAS, qg.GEMM_EPILOGUE_RELU, qg.GEMM_EPILOGUE_GELU
FLAGS = [BIAS, BIAS | RELU, BIAS | GELU, GELU, RELU]


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


def _check(lib, p, o=None, what=""):
    rc, D = run_problem(lib, p, o)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"{what} flags={p.epilogue} -> {qg.gemm_last_choice(lib.h)}")


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("d_type,bias_type", [(synth.BF16, synth.F32), (synth.F32, synth.BF16), (synth.F16, synth.F16)])
def test_dense_tma_epilogue(lib, flags, d_type, bias_type):
    p = synth.dense(200, 384, 320, seed=flags, a_type=synth.BF16 if d_type != synth.F16 else synth.F16,
                    d_type=d_type, dist="normal", scale=0.1, alpha=1.5, beta=0.5)
    _check(lib, synth.with_epilogue(p, flags, seed=7, bias_type=bias_type), what="dense TMA")


@pytest.mark.parametrize("flags", FLAGS)
def test_register_epilogue_unaligned_rows(lib, flags):
    # N = 100 makes D's rows 200 bytes: no TMA store, per-element tail stores
    p = synth.dense(130, 100, 256, seed=10 + flags, a_type=synth.BF16, d_type=synth.BF16, dist="normal",
                    scale=0.1, beta=-1.0)
    _check(lib, synth.with_epilogue(p, flags, seed=8), what="register epilogue")


@pytest.mark.parametrize("flags", [BIAS | GELU, BIAS | RELU])
@pytest.mark.parametrize("kernel", ["umma2_bn224/dp", "umma2_bn256/streamk", "umma_bn128/splitk3", "umma_bn256/streamk"])
def test_schedules_and_pairs(lib, flags, kernel, monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_KERNEL", kernel)
    p = synth.dense(512, 600, 640, seed=20, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.05,
                    alpha=1.0, beta=0.5)
    _check(lib, synth.with_epilogue(p, flags, seed=9, bias_type=synth.BF16), what=kernel)
    assert qg.gemm_last_choice(lib.h) == kernel


@pytest.mark.parametrize("flags", [BIAS | GELU, BIAS])
@pytest.mark.parametrize("M", [1, 16, 64])
def test_decode_paths(lib, flags, M):
    # M = 1: the small-M streaming kernel; 16 / 64: swapped operands
    p = synth.dense(M, 1000, 1024, seed=30 + M, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.05)
    _check(lib, synth.with_epilogue(p, flags, seed=10), what=f"decode M={M}")


@pytest.mark.parametrize("flags", [BIAS | GELU, BIAS | RELU])
def test_w4a16(lib, flags):
    for M in (1, 40, 128):
        p = synth.w4a16(M, 520, 512, seed=40 + M, group=128)
        _check(lib, synth.with_epilogue(p, flags, seed=11), what=f"W4A16 M={M}")


@pytest.mark.parametrize("flags", [BIAS | GELU, BIAS | RELU])
def test_grouped(lib, flags):
    gp = synth.with_epilogue(synth.grouped([3, 0, 130, 300], 600, 256, seed=12), flags, seed=12)
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.grouped(gp)
    assert_close(D.double().cpu().numpy(), ref, bound, gp.d_type, f"grouped flags={flags}")


def test_k_zero(lib):
    p = synth.dense(33, 70, 8, seed=13, a_type=synth.BF16, d_type=synth.F32, beta=0.5)
    p.K = 0
    p.A = np.zeros((33, 0), dtype=np.uint16)
    p.B = np.zeros((70, 0), dtype=np.uint16)
    _check(lib, synth.with_epilogue(p, BIAS | GELU, seed=13), what="K = 0")
    assert qg.gemm_last_choice(lib.h) == "scale_c"


def test_argument_checks(lib):
    p = synth.dense(64, 64, 64, seed=14, a_type=synth.BF16, d_type=synth.BF16)
    bias = torch.zeros(64, dtype=torch.float32, device="cuda")
    host = torch.zeros(64, dtype=torch.float32)
    for flags, ptr, btype, want in ((RELU | GELU, 0, 0, qg.GEMM_ERR_INVALID_ARG),
                                    (8, 0, 0, qg.GEMM_ERR_INVALID_ARG),
                                    (BIAS, None, qg.GEMM_F32, qg.GEMM_ERR_INVALID_ARG),
                                    (BIAS, qg.ptr(bias), qg.GEMM_S4, qg.GEMM_ERR_UNSUPPORTED),
                                    (BIAS, qg.ptr(bias) + 2, qg.GEMM_F32, qg.GEMM_ERR_INVALID_ARG),
                                    (BIAS, qg.ptr(host), qg.GEMM_F32, qg.GEMM_ERR_INVALID_ARG),
                                    (BIAS | RELU, qg.ptr(bias), qg.GEMM_F32, qg.GEMM_OK)):
        o = op()
        o.epilogue, o.bias, o.bias_type = flags, ptr, btype
        rc, _ = run_problem(lib, p, o)
        assert rc == want, (flags, btype, qg.gemm_status_string(rc))
