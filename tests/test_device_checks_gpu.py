"""The checked debug build (device-side bounds checks, QG_DEVICE_CHECKS):
every work unit's tile coordinates, K range, partial slots and tile counter
are checked against the problem and the workspace before they are used, and
every element the register epilogue reads or writes against C's / D's
extent.  This stands in for a memory checker on machines where none runs.

The test builds libqgemm_checked.so, then in a child process (which loads it
through GEMM_DEVICE_CHECKS=1) runs small problems through every kernel and
schedule, compares them with the oracle and requires that no check fired.
It then makes the checks fire without any out-of-bounds access: the host
tells the kernels a quarter of the partials buffer it passed (the buffer itself
is whole), so the split units whose slots lie past a quarter of it are refused,
recorded and skipped, and gemm_device_status reports GEMM_ERR_DEVICE_CHECK.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

CHILD = r'''
import os, sys
sys.path.insert(0, ROOT); sys.path.insert(0, os.path.join(ROOT, "tests"))
import numpy as np, torch
import quantized_gemm_tcgen05_gb300 as qg
import oracle, synth
from gpu_helpers import Lib, assert_close, op, run_grouped, run_problem
assert qg.lib().gemm_checked_build() == 1
lib = Lib()
st = qg.current_stream()

def check(p, o=None, grouped=False, force=None, what=""):
    if force:
        os.environ["GEMM_FORCE_KERNEL"] = force
    else:
        os.environ.pop("GEMM_FORCE_KERNEL", None)
    rc, D = run_grouped(lib, p, o) if grouped else run_problem(lib, p, o)
    assert rc == 0, (what, qg.gemm_status_string(rc))
    assert qg.gemm_device_status(lib.h, st) == 0, (what, qg.gemm_last_choice(lib.h))
    ref, bound = oracle.grouped(p) if grouped else oracle.gemm(p)
    assert_close(D.double().cpu().numpy(), ref, bound, p.d_type, what)
    print("ok", what, qg.gemm_last_choice(lib.h), flush=True)

bf = synth.BF16
d = lambda M, N, K, **kw: synth.dense(M, N, K, seed=M + N + K, a_type=kw.pop("a", bf), d_type=kw.pop("dt", bf),
                                     dist="normal", scale=0.1, **kw)
check(d(300, 520, 712, alpha=1.5, beta=0.5), what="dense automatic")
check(d(200, 328, 1024), o=op(splitk=4), what="split-K 4")
check(d(200, 328, 1024, beta=0.5), o=op(streamk=1), what="stream-K")
check(d(16, 2048, 2048), what="decode, swapped operands")
check(d(600, 900, 1344), force="umma2_bn224/streamk", what="CTA pairs, stream-K")
check(d(512, 520, 256, alpha=1.5, beta=0.5), force="umma2_bn256/dp", what="CTA pairs")
check(d(1, 300, 1024), what="small-M streaming kernel")
check(d(150, 260, 0, beta=0.5), what="K = 0")
check(synth.dense(200, 328, 528, seed=3, a_type=synth.E4M3, d_type=bf, alpha=0.125), what="fp8")
check(synth.w4a16(96, 640, 1024, seed=5, group=64, zero=True), o=op(gb=64, streamk=1), what="int4 + zero points")
check(synth.w4a16(1, 640, 1024, seed=6, group=128), what="int4 streaming")
check(synth.grouped([3, 0, 300, 77], 384, 512, seed=7), grouped=True, what="grouped")
check(synth.grouped([300, 0, 600], 512, 256, seed=8), grouped=True, force="umma2_grouped_bn256/dp",
      what="grouped CTA pairs")
check(synth.grouped_w4a16([40, 0, 130, 7], 320, 384, seed=9, group=64, zero=True), grouped=True,
      what="grouped W4A16")

# the checks fire, without any out-of-bounds access: the kernels are told a
# quarter of the partials buffer they were given (16 MiB of 64 KB slots are
# needed here), so split units with slots past 8 MiB are refused and skipped
os.environ["GEMM_FORCE_KERNEL"] = "umma_bn128/splitk8"
os.environ["GEMM_CHECK_SHRINK_WORKSPACE"] = "1"
fresh = qg.Workspace()  # its counters are left unbalanced by the skipped units
p = d(512, 1024, 4096)
A = torch.zeros(512, 4096, dtype=torch.bfloat16, device="cuda")
B = torch.zeros(1024, 4096, dtype=torch.bfloat16, device="cuda")
D = torch.zeros(512, 1024, dtype=torch.bfloat16, device="cuda")
rc = qg.gemm_run(lib.h, op(), 1.0, qg.ptr(A), qg.row_major(A), None, None, qg.ptr(B), qg.col_major_from_nk(B),
                 None, None, 0.0, None, None, qg.ptr(D), qg.row_major(D), fresh.c, st)
assert rc == 0, qg.gemm_status_string(rc)
got = qg.gemm_device_status(lib.h, st)
assert got == qg.GEMM_ERR_DEVICE_CHECK, qg.gemm_status_string(got)
assert qg.gemm_device_status(lib.h, st) == 0  # the record is cleared
print("checks fire", flush=True)
'''


def test_checked_build_parity_and_firing():
    from quantized_gemm_tcgen05_gb300 import _build

    _build.build(checks=True)
    env = dict(os.environ, GEMM_DEVICE_CHECKS="1")
    env.pop("GEMM_FORCE_KERNEL", None)
    r = subprocess.run([sys.executable, "-c", "ROOT = " + repr(ROOT) + "\n" + CHILD], env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checks fire" in r.stdout
