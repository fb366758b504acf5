"""GPU parity of the schedules: decode-shaped problems with swapped operands,
split-K and stream-K (fp32 partials + last-arriver reduction in the
workspace), batched and grouped (MoE) GEMMs, against the CPU oracle.

Invariants checked besides parity: split-K(S) and stream-K agree with the
unsplit run within tolerance, both are bitwise run-to-run deterministic (the
partials are reduced in a fixed K order), the barrier workspace is left
zeroed, batched equals a loop of single GEMMs and grouped equals a loop of
per-expert GEMMs (the oracle's definitions of those two).
"""
import numpy as np
import pytest
import torch

import quantized_gemm_tcgen05_gb300 as qg
import oracle
import synth
from gpu_helpers import (Lib, assert_close, dev_bits, grouped_to_device, op, run_grouped, run_problem,
                         sample_indices)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


def _barriers_clean(lib):
    return int(lib.ws.barriers.view(torch.int32).abs().sum().item()) == 0


@pytest.mark.parametrize("M", [1, 16, 64])
def test_config3_decode_all_schedules(lib, M):
    p = synth.config3(M)
    ref, bound = oracle.gemm(p)
    outs = {}
    for name, o in (("unsplit", op(splitk=1)), ("splitk8", op(splitk=8)), ("streamk", op(streamk=1)),
                    ("auto", op())):
        rc, D = run_problem(lib, p, o)
        assert rc == 0, f"{name}: {qg.gemm_status_string(rc)}"
        assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"C3 M={M} {name}")
        outs[name] = D
        assert _barriers_clean(lib), f"{name} left barrier counters set"
    for name in ("splitk8", "streamk"):
        o = op(splitk=8) if name == "splitk8" else op(streamk=1)
        rc, D2 = run_problem(lib, p, o)
        assert rc == 0 and torch.equal(D2, outs[name]), f"{name} is not run-to-run deterministic"


@pytest.mark.parametrize("S", [2, 3, 8])
def test_splitk_matches_unsplit(lib, S):
    p = synth.dense(200, 384, 64 * 13 + 8, seed=40 + S, a_type=synth.BF16, d_type=synth.F32, alpha=1.5,
                    beta=0.5)
    ref, bound = oracle.gemm(p)
    rc, D1 = run_problem(lib, p, op(splitk=1))
    assert rc == 0
    rc, DS = run_problem(lib, p, op(splitk=S))
    assert rc == 0
    assert_close(D1.double().cpu().numpy(), ref, bound, p.d_type, "unsplit")
    assert_close(DS.double().cpu().numpy(), ref, bound, p.d_type, f"split {S}")
    assert _barriers_clean(lib)


@pytest.mark.parametrize("shape", [(128, 128, 64 * 9), (300, 700, 1000), (64, 4096, 14336), (1000, 1000, 64)])
def test_streamk_matches_oracle(lib, shape):
    M, N, K = shape
    p = synth.dense(M, N, K, seed=sum(shape), a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.05,
                    beta=-0.75)
    rc, D = run_problem(lib, p, op(streamk=1))
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, f"stream-K {shape}")
    assert _barriers_clean(lib)


def test_splitk_needs_workspace(lib):
    p = synth.dense(64, 256, 1024, seed=3, a_type=synth.BF16, d_type=synth.BF16)
    rc, _ = run_problem(lib, p, op(splitk=4), workspace=False)
    assert rc == qg.GEMM_ERR_WORKSPACE


def test_batched_equals_loop(lib):
    # the tutorial's batched case: 8 x 512^3, plus a ragged one
    for batch, M, N, K in ((8, 512, 512, 512), (3, 130, 260, 200)):
        gp = synth.batched(batch, M, N, K, seed=batch + M)
        A = dev_bits(gp.A, gp.a_type).view(batch, M, K)
        B = dev_bits(gp.B, gp.a_type)
        D = torch.full((batch, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = qg.gemm_run(lib.h, op(), 1.0, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B),
                         qg.col_major_from_nk(B), None, None, 0.0, None, None, qg.ptr(D), qg.row_major(D),
                         lib.ws.c, qg.current_stream())
        torch.cuda.synchronize()
        assert rc == 0, qg.gemm_status_string(rc)
        ref, bound = oracle.grouped(gp)
        assert_close(D.reshape(batch * M, N).double().cpu().numpy(), ref, bound, gp.d_type, f"batched {batch}")


@pytest.mark.parametrize("counts", [[3, 0, 130], [0, 0, 0, 257], [128, 1, 0, 127, 129], [64] * 8, [0, 5]])
def test_grouped_ragged(lib, counts):
    gp = synth.grouped(counts, 320, 192, seed=len(counts))
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    ref, bound = oracle.grouped(gp)
    assert_close(D.double().cpu().numpy(), ref, bound, gp.d_type, f"grouped {counts}")


@pytest.mark.parametrize("bn", [224, 256])
@pytest.mark.parametrize("counts,K", [([3, 0, 130, 300, 0, 257], 320), ([256, 1, 0, 511, 129], 72 * 4),
                                      ([0, 0, 700], 64 * 5), ([40] * 8, 256)])
def test_grouped_on_cta_pairs(lib, bn, counts, K, monkeypatch):
    # 256-row expert blocks over CTA pairs: a block's second half may hold
    # none of its expert's rows; K a multiple of 64 copies two K-steps per box
    monkeypatch.setenv("GEMM_FORCE_KERNEL", f"umma2_grouped_bn{bn}/dp")
    gp = synth.grouped(counts, 600, K, seed=len(counts) + bn)
    rc, D = run_grouped(lib, gp)
    assert rc == 0, qg.gemm_status_string(rc)
    assert qg.gemm_last_choice(lib.h) == f"umma2_grouped_bn{bn}/dp"
    ref, bound = oracle.grouped(gp)
    assert_close(D.double().cpu().numpy(), ref, bound, gp.d_type, f"grouped pairs bn{bn} {counts}")
    assert qg.gemm_device_status(lib.h, qg.current_stream()) == 0


def test_config5_grouped_full_sampled(lib):
    gp = synth.config5()
    rc, D = run_grouped(lib, gp)
    assert rc == 0
    T = int(gp.offsets[-1])
    ii, jj = sample_indices(T, gp.N, 1500, seed=9)
    # make sure every expert with rows is sampled
    extra = np.array([int(gp.offsets[e]) for e in range(len(gp.counts)) if gp.counts[e] > 0])
    ii = np.concatenate([ii, extra, np.maximum(extra - 1, 0)])
    jj = np.concatenate([jj, np.arange(len(extra)) * 997 % gp.N, np.arange(len(extra)) * 131 % gp.N])
    ref, bound = oracle.grouped_entries(gp, ii, jj)
    assert_close(D.double().cpu().numpy()[ii, jj], ref, bound, gp.d_type, "C5 grouped (sampled)")


def test_cache_measure_export_import(lib):
    p = synth.dense(16, 1024, 2048, seed=5, a_type=synth.BF16, d_type=synth.BF16)
    n0 = qg.gemm_cache_size(lib.h)
    rc, D = run_problem(lib, p, op(dispatch=qg.GEMM_DISPATCH_MEASURE))
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "measured")
    assert qg.gemm_cache_size(lib.h) == n0 + 1
    blob = qg.gemm_export(lib.h)
    assert blob.startswith(b"qgemm-dispatch-cache 3\n")
    h2 = qg.gemm_create()
    try:
        assert qg.gemm_import(h2, blob) == 0
        assert qg.gemm_cache_size(h2) == qg.gemm_cache_size(lib.h)
        assert qg.gemm_export(h2) == blob
        for bad in (blob[:-5], blob.replace(b"sm ", b"sm 1"), b"qgemm-dispatch-cache 2\n" + blob[23:], b"garbage"):
            assert qg.gemm_import(h2, bad) == qg.GEMM_ERR_BAD_CACHE
        assert qg.gemm_export(h2) == blob
    finally:
        qg.gemm_destroy(h2)
    seq = qg.gemm_get_tuning_seq(lib.h)
    assert seq == sorted(seq) and seq[0] == 1


def test_device_timeout_selftest(lib):
    assert qg.gemm_device_status(lib.h, qg.current_stream()) == 0
    assert qg.gemm_selftest_wait_timeout(lib.h, 2_000_000, qg.current_stream()) == qg.GEMM_ERR_DEVICE_TIMEOUT
    # the record is cleared and the context still works
    assert qg.gemm_device_status(lib.h, qg.current_stream()) == 0
    p = synth.dense(128, 128, 128, seed=2, a_type=synth.BF16, d_type=synth.F32)
    rc, D = run_problem(lib, p)
    assert rc == 0
    ref, bound = oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, "after self-test")


def test_argument_errors(lib):
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    st = qg.current_stream()
    good = dict(A=qg.ptr(A), Ad=qg.row_major(A), B=qg.ptr(B), Bd=qg.col_major_from_nk(B), D=qg.ptr(D),
                Dd=qg.row_major(D))

    def call(**kw):
        a = dict(good, **kw)
        return qg.gemm_run(lib.h, kw.get("o", op()), 1.0, a["A"], a["Ad"], None, None, a["B"], a["Bd"], None,
                           None, kw.get("beta", 0.0), kw.get("C"), kw.get("Cd"), a["D"], a["Dd"], lib.ws.c, st)

    assert call() == 0
    assert call(A=None) == qg.GEMM_ERR_INVALID_ARG
    assert call(A=qg.ptr(A) + 2) == qg.GEMM_ERR_INVALID_ARG                     # misaligned for TMA
    assert call(Ad=qg.layout(qg.GEMM_BF16, qg.GEMM_ROW_MAJOR, 64, 64, 60)) == qg.GEMM_ERR_INVALID_ARG
    assert call(Ad=qg.layout(qg.GEMM_BF16, qg.GEMM_COL_MAJOR, 64, 64, 64)) == qg.GEMM_ERR_UNSUPPORTED
    assert call(Bd=qg.layout(qg.GEMM_F16, qg.GEMM_COL_MAJOR, 64, 64, 64)) == qg.GEMM_ERR_UNSUPPORTED
    assert call(beta=1.0) == qg.GEMM_ERR_INVALID_ARG                             # C missing
    assert call(o=op(splitk=2, streamk=1)) == qg.GEMM_ERR_INVALID_ARG
    host = torch.zeros(64, 64, dtype=torch.bfloat16)
    assert call(A=qg.ptr(host)) == qg.GEMM_ERR_INVALID_ARG                      # not device memory
    torch.cuda.synchronize()
