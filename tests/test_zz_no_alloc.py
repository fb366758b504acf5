"""gemm_run_noalloc: the entry point for callers that cannot allocate device
memory (a plug-in whose host framework owns every byte of the device, or code
where an allocation would synchronise the device).  Its split-K / stream-K
scratch is a fixed array in the library's own device memory, so the caller
passes only inputs and outputs.

Checked through the C ABI on two calls in a row (the array keeps the previous
call's contents): against the oracle within the tolerance every parity test
here uses, and bit for bit against gemm_run with a caller workspace (the
partial reduction runs in a fixed order, so the two must agree exactly).
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_gemm_tcgen05_gb300 as qg
import synth
from gpu_helpers import Lib, assert_close, dev_bits, op

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = Lib()
    yield L
    L.close()


def _run(lib, p, o, noalloc):
    A, B = dev_bits(p.A, p.a_type), dev_bits(p.B, p.b_type)
    C = dev_bits(p.C, p.c_type) if p.beta != 0.0 else None
    D = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    args = (lib.h, o, p.alpha, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B), qg.col_major_from_nk(B), None,
            None, p.beta, qg.ptr(C), qg.row_major(C) if C is not None else None, qg.ptr(D), qg.row_major(D))
    if noalloc:
        rc = qg.gemm_run_noalloc(*args, qg.current_stream())
    else:
        rc = qg.gemm_run(*args, lib.ws.c, qg.current_stream())
    torch.cuda.synchronize()
    return rc, D, qg.gemm_last_choice(lib.h)


@pytest.mark.parametrize("case", ["splitk4", "streamk"])
def test_noalloc_matches_gemm_run_twice(lib, case):
    p = synth.dense(16, 2048, 4096, seed=77, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.05,
                    alpha=1.5, beta=0.5)
    o = op(splitk=4) if case == "splitk4" else op(streamk=1)
    rc, want, kind = _run(lib, p, o, noalloc=False)
    assert rc == 0, qg.gemm_status_string(rc)
    assert ("splitk4" if case == "splitk4" else "streamk") in kind
    ref, bound = oracle.gemm(p)
    assert_close(want.double().cpu().numpy(), ref, bound, p.d_type, f"gemm_run {case}")
    for call in range(2):
        rc, got, kind2 = _run(lib, p, o, noalloc=True)
        assert rc == 0, qg.gemm_status_string(rc)
        assert kind2 == kind
        assert_close(got.double().cpu().numpy(), ref, bound, p.d_type, f"noalloc {case} call {call}")
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"noalloc {case} call {call}: not bitwise"


def test_noalloc_automatic_split_falls_back_to_unsplit(lib):
    # 36 tiles of 128 x 128: the automatic choice splits K four ways, whose
    # 9.4 MB of partials fit a 32 MB workspace but not the 8 MB array, so the
    # array-backed call runs the unsplit schedule instead
    p = synth.dense(128, 4608, 2048, seed=79, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.05)
    want_big = qg.gemm_heuristic_choice(p.M, p.N, p.K, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16, 0, 0, 0,
                                          torch.cuda.get_device_properties(0).multi_processor_count,
                                          qg.GEMM_PARTIALS_SIZE)
    want_small = qg.gemm_heuristic_choice(p.M, p.N, p.K, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16, 0, 0, 0,
                                            torch.cuda.get_device_properties(0).multi_processor_count,
                                            qg.GEMM_NOALLOC_PARTIALS_SIZE)
    assert "splitk" in want_big and want_small.endswith("/dp"), (want_big, want_small)
    ref, bound = oracle.gemm(p)
    rc, big, kind = _run(lib, p, op(), noalloc=False)
    assert rc == 0 and kind == want_big, (qg.gemm_status_string(rc), kind)
    assert_close(big.double().cpu().numpy(), ref, bound, p.d_type, "gemm_run automatic")
    for call in range(2):
        rc, got, kind = _run(lib, p, op(), noalloc=True)
        assert rc == 0, qg.gemm_status_string(rc)
        assert kind == want_small
        assert_close(got.double().cpu().numpy(), ref, bound, p.d_type, f"noalloc automatic call {call}")


def test_noalloc_rejects_scratch_beyond_its_array(lib):
    # 8 slices of 64 tiles of 128 x 256 fp32 partials need 64 MB > 8 MB
    p = synth.dense(1024, 2048, 4096, seed=78, a_type=synth.BF16, d_type=synth.BF16)
    rc, _, _ = _run(lib, p, op(splitk=8), noalloc=True)
    assert rc == qg.GEMM_ERR_WORKSPACE
