"""GPU parity of the CTA-pair kernel (tcgen05.mma.cta_group::2, 256-row tiles
over clusters of two SMs) against the CPU oracle: every tile width it is
built for, ragged edges in all three dimensions, batched operands, the
row/column placement of both CTAs' halves, and the C2-shaped problem at full
size on sampled outputs."""
import numpy as np
import pytest
import torch

import oracle
import quantized_gemm_tcgen05_gb300 as qg
import synth
from gpu_helpers import Lib, assert_close, dev_bits, op, run_problem, sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


@pytest.mark.parametrize("bn", [128, 224, 256])
# K a multiple of 64 copies two K-steps per box (odd chunk counts end on a
# half-filled stage); other K one K-step per box
@pytest.mark.parametrize("shape", [(256, 256, 128), (300, 520, 712), (1000, 777, 64 * 9 + 8), (129, 33, 72),
                                   (384, 448, 64 * 13), (512, 300, 4096)])
def test_pair_kernel_parity(lib, bn, shape, monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_KERNEL", f"umma2_bn{bn}/dp")
    M, N, K = shape
    p = synth.dense(M, N, K, seed=M + N + K + bn, a_type=synth.BF16, d_type=synth.BF16, alpha=1.5, beta=0.5,
                    dist="normal", scale=0.1)
    rc, D = run_problem(lib, p)
    assert rc == 0, qg.gemm_status_string(rc)
    assert qg.gemm_last_choice(lib.h) == f"umma2_bn{bn}/dp"
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"pair bn{bn} {shape}")
    assert qg.gemm_device_status(lib.h, qg.current_stream()) == 0


@pytest.mark.parametrize("bn", [224, 256])
@pytest.mark.parametrize("shape", [(1024, 1500, 4096), (600, 900, 64 * 21), (2048, 700, 1000)])
def test_pair_kernel_streamk(lib, bn, shape, monkeypatch):
    # stream-K over CTA pairs: each CTA keeps its own partial slots and
    # arrival counter for its 128-row half of a split tile
    monkeypatch.setenv("GEMM_FORCE_KERNEL", f"umma2_bn{bn}/streamk")
    M, N, K = shape
    p = synth.dense(M, N, K, seed=M + N + K + bn + 1, a_type=synth.BF16, d_type=synth.BF16, alpha=0.75, beta=-0.5,
                    dist="normal", scale=0.1)
    rc, D = run_problem(lib, p)
    assert rc == 0, qg.gemm_status_string(rc)
    assert qg.gemm_last_choice(lib.h) == f"umma2_bn{bn}/streamk"
    ii, jj = sample_indices(M, N, 4000, seed=bn)
    ref, bound = oracle.gemm_entries(p, ii, jj)
    assert_close(D.double().cpu().numpy()[ii, jj], ref, bound, p.d_type, f"pair stream-K bn{bn} {shape}")
    assert int(lib.ws.barriers.view(torch.int32).abs().sum().item()) == 0, "arrival counters left set"
    rc, D2 = run_problem(lib, p)
    assert rc == 0 and torch.equal(D, D2), "pair stream-K is not run-to-run deterministic"
    assert qg.gemm_device_status(lib.h, qg.current_stream()) == 0


def test_pair_kernel_one_hot_layout(lib, monkeypatch):
    # rows of both CTAs and both halves of the Y tile land where they belong
    monkeypatch.setenv("GEMM_FORCE_KERNEL", "umma2_bn256/dp")
    M, N, K = 256, 256, 192
    p = synth.dense(M, N, K, seed=5, a_type=synth.F16, d_type=synth.F32, dist="uniform")
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), (5 * np.arange(M)) % K] = 0x3C00
    p.A = A
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, _ = oracle.gemm(p)
    assert np.array_equal(D.double().cpu().numpy(), ref)


def test_pair_kernel_batched(lib, monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_KERNEL", "umma2_bn224/dp")
    batch, M, N, K = 3, 300, 260, 200
    gp = synth.batched(batch, M, N, K, seed=17)
    A = dev_bits(gp.A, gp.a_type).view(batch, M, K)
    B = dev_bits(gp.B, gp.a_type)
    D = torch.full((batch, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = qg.gemm_run(lib.h, op(), 1.0, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B), qg.col_major_from_nk(B),
                     None, None, 0.0, None, None, qg.ptr(D), qg.row_major(D), lib.ws.c, qg.current_stream())
    torch.cuda.synchronize()
    assert rc == 0 and qg.gemm_last_choice(lib.h) == "umma2_bn224/dp"
    ref, bound = oracle.grouped(gp)
    assert_close(D.reshape(batch * M, N).double().cpu().numpy(), ref, bound, gp.d_type, "pair batched")


def test_pair_kernel_config2_full_sampled(lib, monkeypatch):
    monkeypatch.setenv("GEMM_FORCE_KERNEL", "umma2_bn256/dp")
    p = synth.config2()
    rc, D = run_problem(lib, p)
    assert rc == 0
    ii, jj = sample_indices(p.M, p.N, 2000, seed=8)
    ref, bound = oracle.gemm_entries(p, ii, jj)
    assert_close(D.double().cpu().numpy()[ii, jj], ref, bound, p.d_type, "pair C2 sampled")


def test_pair_kernel_many_waves_elementwise(lib, monkeypatch):
    # 10 x 11 = 110 tiles of 256 x 224 on at most 76 clusters: every cluster
    # reuses both TMEM accumulators and turns its ring phases over, checked
    # element by element
    monkeypatch.setenv("GEMM_FORCE_KERNEL", "umma2_bn224/dp")
    p = synth.dense(2560, 2304, 64, seed=2560, a_type=synth.BF16, d_type=synth.BF16, alpha=1.5, beta=0.5,
                    dist="normal", scale=0.25)
    rc, D = run_problem(lib, p)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "pair, many waves")


def test_pair_grouped_many_waves_elementwise(lib, monkeypatch):
    # 17 expert blocks of 256 rows x 8 column tiles = 136 pair tiles
    from gpu_helpers import run_grouped
    monkeypatch.setenv("GEMM_FORCE_KERNEL", "umma2_grouped_bn256/dp")
    gp = synth.grouped([1000, 0, 1500, 700, 900], 2048, 128, seed=4100)
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    assert qg.gemm_last_choice(lib.h) == "umma2_grouped_bn256/dp"
    ref, bound = oracle.grouped(gp)
    assert_close(D.double().cpu().numpy(), ref, bound, gp.d_type, "pair grouped, many waves")
