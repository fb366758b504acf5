"""gemm_run_noalloc: the entry point for callers that cannot allocate device
memory (for example under a stream capture that forbids allocation, or inside
a host whose allocator hands out no scratch).  Its split-K / stream-K scratch
is a fixed array in the library's own device memory, so the caller passes only
inputs and outputs.

Checked through the C ABI against gemm_run with a caller workspace, on two
calls in a row (the array keeps the previous call's contents), within the
tolerance every parity test here uses.  This file is collected last so that a
run stopping at the first failure has already run every other test.
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


def _operands(p):
    A, B = dev_bits(p.A, p.a_type), dev_bits(p.B, p.b_type)
    C = dev_bits(p.C, p.c_type) if p.beta != 0.0 else None
    return A, B, C


def _run(lib, p, o, noalloc):
    A, B, C = _operands(p)
    D = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    args = (lib.h, o, p.alpha, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B), qg.col_major_from_nk(B), None,
            None, p.beta, qg.ptr(C), qg.row_major(C) if C is not None else None, qg.ptr(D), qg.row_major(D))
    if noalloc:
        rc = qg.gemm_run_noalloc(*args, qg.current_stream())
    else:
        rc = qg.gemm_run(*args, lib.ws.c, qg.current_stream())
    torch.cuda.synchronize()
    return rc, D


@pytest.mark.parametrize("case", ["splitk4", "streamk"])
def test_noalloc_matches_gemm_run_twice(lib, case):
    p = synth.dense(16, 2048, 4096, seed=77, a_type=synth.BF16, d_type=synth.BF16, dist="normal", scale=0.05,
                    alpha=1.5, beta=0.5)
    o = op(splitk=4) if case == "splitk4" else op(streamk=1)
    rc, want = _run(lib, p, o, noalloc=False)
    assert rc == 0, qg.gemm_status_string(rc)
    _, bound = oracle.gemm(p)
    ref = want.double().cpu().numpy()
    for call in range(2):
        rc, got = _run(lib, p, o, noalloc=True)
        assert rc == 0, qg.gemm_status_string(rc)
        assert_close(got.double().cpu().numpy(), ref, bound, p.d_type, f"noalloc {case} call {call}")


def test_noalloc_rejects_scratch_beyond_its_array(lib):
    # 8 slices of 64 tiles of 128 x 256 fp32 partials need 64 MB > 8 MB
    p = synth.dense(1024, 2048, 4096, seed=78, a_type=synth.BF16, d_type=synth.BF16)
    rc, _ = _run(lib, p, op(splitk=8), noalloc=True)
    assert rc == qg.GEMM_ERR_WORKSPACE
