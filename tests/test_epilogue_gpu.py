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
from gpu_helpers import TORCH_DT, Lib, assert_close, dev_bits, op, run_grouped, run_problem

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


def _padded(rows, cols, ld, dtype, fill=float("nan")):
    """A [rows, cols] view with row stride ld (a multiple of 8 elements)."""
    return torch.full((rows, ld), fill, dtype=dtype, device="cuda")[:, :cols]


@pytest.mark.parametrize("kernel", ["umma_bn128/dp", "umma_bn128/splitk3", "umma_bn64/streamk", "umma2_bn256/dp",
                                    "umma_bn64_swap/splitk2", "umma_bn16_swap/dp"])
@pytest.mark.parametrize("d_type", [synth.BF16, synth.F16])
def test_register_epilogue_forced(lib, kernel, d_type, monkeypatch):
    # The register epilogue on every kernel shape (the TMA store switched
    # off): 16-byte row pieces of C and D when the rows allow them, the
    # swapped tile's transposed stores, the split-tile reductions, and the
    # ragged last columns and rows; C is read (beta != 0) and D's rows are
    # padded so that N is not a multiple of 8 while the rows stay aligned.
    monkeypatch.setenv("GEMM_EPI_TMA", "0")
    monkeypatch.setenv("GEMM_FORCE_KERNEL", kernel)
    swap = "swap" in kernel
    M, N, K = (40, 1001, 768) if swap else (200, 1001, 640)
    a_type = synth.F16 if d_type == synth.F16 else synth.BF16
    p = synth.dense(M, N, K, seed=40 + len(kernel), a_type=a_type, d_type=d_type, dist="normal", scale=0.05,
                    alpha=1.25, beta=0.5)
    p = synth.with_epilogue(p, BIAS | GELU, seed=11, bias_type=synth.F32)
    ld = 1008
    C = _padded(M, N, ld, TORCH_DT[d_type], 0.0)
    C.copy_(dev_bits(p.C, p.c_type))
    D = _padded(M, N, ld, TORCH_DT[d_type])
    rc, D = run_problem(lib, p, D=D, C=C)
    assert rc == 0, qg.gemm_status_string(rc)
    assert qg.gemm_last_choice(lib.h) == kernel
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"register epilogue {kernel}")
    # and with unpadded rows of a multiple of 8 columns (no ragged piece)
    p2 = synth.dense(M, 1000, K, seed=41, a_type=a_type, d_type=d_type, dist="normal", scale=0.05, alpha=1.0,
                     beta=-0.75)
    _check(lib, p2, what=f"register epilogue {kernel} N=1000")


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
