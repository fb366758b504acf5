"""GPU parity of the dense tcgen05 path against the CPU oracle.

Element-wise comparisons at sizes the oracle finishes in seconds (several
tiles plus ragged tails), full-size configurations on sampled outputs, the
odd/even K-step check of the DeepGEMM kernel-set blog (section 4.3), and the
closed forms (identity B, all-ones operands).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import Lib, assert_close, op, run_problem, sample_indices, dev_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


def _check(lib, p, o=None, what=""):
    rc, D = run_problem(lib, p, o)
    assert rc == 0, f"{what}: status {rc}"
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, what)
    return D


def test_one_hot_layout(lib):
    # A[i][k] = 1 at k = (3i) % K: D[i][j] = B-hat[(3i) % K][j] exactly, which
    # pins the row/column mapping of both operands and of the accumulator.
    M, N, K = 128, 256, 128
    p = synth.dense(M, N, K, seed=1, a_type=synth.BF16, d_type=synth.F32, dist="uniform")
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), (3 * np.arange(M)) % K] = 0x3F80
    p.A = A
    D = _check(lib, p, what="one-hot")
    ref, _ = oracle.gemm(p)
    assert np.array_equal(D.double().cpu().numpy(), ref)


def test_config1_fp16_256(lib):
    _check(lib, synth.config1(), what="C1")


def test_identity_b_closed_form(lib):
    K = 192
    p = synth.dense(200, K, K, seed=7, a_type=synth.F16, d_type=synth.F16, alpha=1.5, beta=0.5)
    p.B = np.where(np.eye(K, dtype=bool), np.uint16(0x3C00), np.uint16(0)).astype(np.uint16)
    _check(lib, p, what="identity B")


def test_all_ones_exact(lib):
    M, N, K = 130, 260, 1024
    p = synth.dense(M, N, K, seed=8, a_type=synth.BF16, d_type=synth.F32)
    p.A = np.full((M, K), 0x3F80, dtype=np.uint16)
    p.B = np.full((N, K), 0x3F80, dtype=np.uint16)
    rc, D = run_problem(lib, p)
    assert rc == 0
    assert torch.all(D == float(K)).item()


@pytest.mark.parametrize("a_type", [synth.BF16, synth.F16])
@pytest.mark.parametrize("d_type", [synth.F32, synth.BF16, synth.F16])
def test_config2_shape_reduced(lib, a_type, d_type):
    # C2's distributions and scalars at a size the oracle checks in full:
    # 3 x 2 tiles of 128 x 256 plus ragged edges.
    p = synth.dense(333, 517, 320, seed=1002, a_type=a_type, d_type=d_type, dist="normal",
                    scale=1 / np.sqrt(320), alpha=1.5, beta=0.5)
    _check(lib, p, what=f"C2-shaped a={a_type} d={d_type}")


@pytest.mark.parametrize("M", [1, 7, 63, 64, 65, 127, 129, 200])
@pytest.mark.parametrize("N", [1, 7, 65, 129, 200])
def test_tails(lib, M, N):
    for K in (8, 72, 200):
        p = synth.dense(M, N, K, seed=M * 1000 + N + K, a_type=synth.BF16, d_type=synth.BF16, alpha=1.0,
                        beta=0.25, dist="uniform")
        _check(lib, p, what=f"tails {M}x{N}x{K}")


@pytest.mark.parametrize("steps", [1, 2, 3, 4, 5, 7, 8, 9, 17])
def test_odd_and_even_k_steps(lib, steps):
    # an odd number of K-slices must agree with the oracle as well as an even one
    K = 64 * steps
    p = synth.dense(256, 256, K, seed=steps, a_type=synth.F16, d_type=synth.F32, dist="uniform")
    _check(lib, p, what=f"{steps} k-steps")


def test_beta_zero_ignores_nan_c(lib):
    p = synth.dense(128, 128, 64, seed=3, a_type=synth.BF16, d_type=synth.BF16)
    C = torch.full((128, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc, D = run_problem(lib, p, C=C)
    assert rc == 0 and torch.isfinite(D.float()).all().item()


def test_in_place_c_is_d(lib):
    p = synth.dense(256, 512, 256, seed=11, a_type=synth.BF16, d_type=synth.BF16, alpha=1.5, beta=0.5)
    C = dev_bits(p.C, p.c_type)
    rc, D = run_problem(lib, p, C=C, D=C)
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "in place")


def test_k_zero_gives_beta_c(lib):
    p = synth.dense(70, 90, 8, seed=12, a_type=synth.BF16, d_type=synth.F32, beta=0.5)
    p.K = 0
    p.A = np.zeros((70, 0), dtype=np.uint16)
    p.B = np.zeros((90, 0), dtype=np.uint16)
    p.c_type = synth.F32
    p.C = np.random.default_rng(0).standard_normal((70, 90)).astype(np.float32)
    rc, D = run_problem(lib, p)
    assert rc == 0
    assert np.array_equal(D.cpu().numpy(), (np.float32(0.5) * p.C).astype(np.float32))


def test_config2_full_sampled(lib):
    p = synth.config2()
    rc, D = run_problem(lib, p)
    assert rc == 0
    ii, jj = sample_indices(p.M, p.N, 2000, seed=5)
    ref, bound = oracle.gemm_entries(p, ii, jj)
    assert_close(D.double().cpu().numpy()[ii, jj], ref, bound, p.d_type, "C2 full (sampled)")


@pytest.mark.parametrize("sched", ["dp", "streamk"])
def test_config2_full_schedules_sampled(lib, sched):
    p = synth.config2()
    o = op(splitk=1) if sched == "dp" else op(streamk=1)
    rc, D = run_problem(lib, p, o)
    assert rc == 0
    ii, jj = sample_indices(p.M, p.N, 1500, seed=6)
    ref, bound = oracle.gemm_entries(p, ii, jj)
    assert_close(D.double().cpu().numpy()[ii, jj], ref, bound, p.d_type, f"C2 {sched}")


@pytest.mark.parametrize("kernel", ["umma_bn16_swap/dp", "umma_bn32_swap/splitk3", "umma_bn64_swap/streamk",
                                    "umma_bn128_swap/dp", "umma_bn16/dp", "umma_bn32/streamk", "umma_bn64/dp",
                                    "umma_bn128/splitk2", "umma_bn192/dp", "umma_bn192/streamk", "umma_bn224/dp",
                                    "umma_bn224/splitk3", "umma_bn256/streamk"])
def test_every_registered_kernel(lib, kernel, monkeypatch):
    # every tile width and schedule the registry can dispatch, pinned by
    # GEMM_FORCE_KERNEL, on a ragged problem that spans several tiles
    monkeypatch.setenv("GEMM_FORCE_KERNEL", kernel)
    swap = "_swap" in kernel
    M = 70 if swap else 300
    p = synth.dense(M, 520, 200 + 64 * 5, seed=len(kernel), a_type=synth.BF16, d_type=synth.BF16, alpha=1.5,
                    beta=0.5, dist="normal", scale=0.1)
    _check(lib, p, what=kernel)
    import quantized_gemm_tcgen05_gb300 as qg
    assert qg.gemm_last_choice(lib.h) == kernel
