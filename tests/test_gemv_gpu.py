"""GPU parity of the small-M streaming kernel ("gemv"): decode-shaped
products with M <= 8 on the CUDA cores, against the CPU oracle.

Covers 16-bit B (bf16 / fp16), 16-bit B with V scales, and int4 B with and
without V over the group sizes the scale rules allow; ragged N (row groups of
four), K split across warps, alpha / beta with C, fp32 / fp16 / bf16 D.  The
dequantised operand is pinned bit-exactly through a one-hot A with fp32 D,
and results are bitwise run-to-run deterministic.
"""
import numpy as np
import pytest
import torch

import quantized_gemm_tcgen05_gb300 as qg
import oracle
import synth
from gpu_helpers import Lib, assert_close, op, run_problem, sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


@pytest.fixture
def force_gemv(monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_KERNEL", "gemv")


def _run(lib, p):
    rc, D = run_problem(lib, p)
    assert rc == 0, qg.gemm_status_string(rc)
    assert qg.gemm_last_choice(lib.h) == "gemv"
    return D


@pytest.mark.parametrize("a_type", [synth.BF16, synth.F16])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_dense_shapes(lib, force_gemv, a_type, M):
    for N, K in ((1, 8), (7, 64), (130, 200), (333, 1032), (64, 8192)):
        p = synth.dense(M, N, K, seed=M * 1000 + N + K, a_type=a_type, d_type=synth.F32, dist="uniform")
        D = _run(lib, p)
        ref, bound = oracle.gemm(p)
        assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"gemv dense M{M} N{N} K{K}")


@pytest.mark.parametrize("d_type", [synth.BF16, synth.F16, synth.F32])
def test_alpha_beta_and_output_types(lib, force_gemv, d_type):
    p = synth.dense(3, 257, 512, seed=11, a_type=synth.BF16, d_type=d_type, dist="normal", scale=0.1,
                    alpha=1.5, beta=-0.75)
    D = _run(lib, p)
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "gemv alpha/beta")


@pytest.mark.parametrize("group,K", [(8, 256), (16, 448), (32, 224), (64, 832), (128, 4096), (192, 768)])
@pytest.mark.parametrize("M", [1, 4, 7])
def test_int4_groups(lib, force_gemv, group, K, M):
    p = synth.w4a16(M, 300, K, seed=group + K + M, group=group)
    D = _run(lib, p)
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"gemv W4A16 g{group} K{K} M{M}")


@pytest.mark.parametrize("a_type", [synth.BF16, synth.F16])
def test_int4_dequant_bit_exact(lib, force_gemv, a_type):
    # one-hot rows of A read single elements of B^ = RN(q * v) into fp32 D
    M, N, K, g = 8, 96, 512, 64
    p = synth.w4a16(M, N, K, seed=5, group=g, a_type=a_type, d_type=synth.F32)
    ks = np.random.default_rng(6).integers(0, K, M)
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), ks] = 0x3F80 if a_type == synth.BF16 else 0x3C00
    p.A = A
    D = _run(lib, p)
    ref, _ = oracle.gemm(p)
    assert np.array_equal(D.double().cpu().numpy(), ref)


def test_int4_without_scales_and_v_on_16bit(lib, force_gemv):
    p = synth.w4a16(2, 200, 320, seed=70, group=64)
    p.V, p.v_type, p.gb = None, None, 0
    D = _run(lib, p)
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "gemv int4 no V")
    q = synth.dense(4, 130, 320, seed=71, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.1)
    v = np.random.default_rng(3).uniform(0.5, 2.0, size=(320 // 64, 130)).astype(np.float32)
    q.V, q.v_type, q.gb = synth._round_bits(v, synth.F16), synth.F16, 64
    D = _run(lib, q)
    ref, bound = oracle.gemm(q)
    assert_close(D.double().cpu().numpy(), ref, bound, q.d_type, "gemv V on 16-bit B")


def test_deterministic_and_full_decode_sizes(lib, force_gemv):
    # the decode workloads: bf16 M=1 N=4096 K=14336, and W4A16 M=1 N=11008 K=4096
    for p in (synth.config3(1), synth.w4a16(1, 11008, 4096, seed=8)):
        D1 = _run(lib, p)
        D2 = _run(lib, p)
        assert torch.equal(D1, D2), "not run-to-run deterministic"
        ii, jj = sample_indices(p.M, p.N, 1500, seed=4)
        ref, bound = oracle.gemm_entries(p, ii, jj)
        assert_close(D1.double().cpu().numpy()[ii, jj], ref, bound, p.d_type, f"gemv {p.name}")


def test_heuristic_takes_gemv_for_decode(lib):
    p = synth.config3(1)
    rc, _ = run_problem(lib, p)
    assert rc == 0 and qg.gemm_last_choice(lib.h) == "gemv"
    # an explicit split names a tensor-core schedule
    rc, _ = run_problem(lib, p, op(splitk=4))
    assert rc == 0 and qg.gemm_last_choice(lib.h) != "gemv"
    q = synth.config3(16)  # the tensor core keeps up from M = 4 on
    rc, _ = run_problem(lib, q)
    assert rc == 0 and qg.gemm_last_choice(lib.h) != "gemv"


def test_measured_choice_round_trips_through_the_cache(lib):
    # measure mode times the streaming kernel beside the tensor-core ones and
    # caches the winner; an exported cache makes a fresh handle choose the same
    p = synth.w4a16(1, 4096, 4096, seed=12)
    rc, D = run_problem(lib, p, op(dispatch=qg.GEMM_DISPATCH_MEASURE, gb=p.gb))
    assert rc == 0
    chosen = qg.gemm_last_choice(lib.h)
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "measured W4A16 M=1")
    blob = qg.gemm_export(lib.h)
    assert blob.startswith(b"qgemm-dispatch-cache 3\n")
    h2 = qg.gemm_create()
    try:
        assert qg.gemm_import(h2, blob) == 0
        other = Lib.__new__(Lib)
        other.h, other.ws = h2, lib.ws
        rc, D2 = run_problem(other, p, op(gb=p.gb))
        assert rc == 0 and qg.gemm_last_choice(h2) == chosen
        assert torch.equal(D, D2)
    finally:
        qg.gemm_destroy(h2)
