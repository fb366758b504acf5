"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/gemm.h declares, and its host planners (stream-K plan,
grouped tile map -- the code the kernels run) agree bit-exactly with the
oracle's restatement of the pages."""
import os
import re

import pytest

import oracle
import quantized_gemm_tcgen05_gb300 as qg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "gemm.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(gemm_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    return qg.lib()


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(qg.SYMBOLS)


def test_status_strings(L):
    for code in range(8):
        assert qg.gemm_status_string(code)
    assert qg.gemm_status_string(0) == "ok"
    assert "unknown" in qg.gemm_status_string(99)


def test_null_handle_rejected(L):
    import ctypes
    assert L.gemm_run(None, None, 1.0, *([None] * 8), 0.0, *([None] * 6)) == qg.GEMM_ERR_INVALID_ARG
    assert L.gemm_export(None, None, 0, None) == qg.GEMM_ERR_INVALID_ARG
    assert L.gemm_import(None, b"x", 1) == qg.GEMM_ERR_INVALID_ARG
    assert L.gemm_create(None) == qg.GEMM_ERR_INVALID_ARG
    n = ctypes.c_int32()
    assert L.gemm_cache_size(None, ctypes.byref(n)) == qg.GEMM_ERR_INVALID_ARG
    assert qg.gemm_last_choice(None) == "none"


@pytest.mark.parametrize("args", [
    (256, 1024, 512, 16, 128, 32, 108), (4096, 16, 14336, 128, 16, 64, 148), (4096, 4096, 4096, 128, 256, 64, 148),
    (4096, 4096, 4096, 128, 256, 64, 152), (1, 1, 1, 128, 16, 64, 3), (11008, 128, 4096, 128, 128, 64, 148),
    (99999, 77777, 12345, 128, 64, 64, 1000), (128, 128, 0, 128, 128, 64, 148)])
def test_streamk_plan_bit_exact(args):
    assert qg.gemm_plan_streamk(*args) == oracle.streamk_plan(*args)


@pytest.mark.parametrize("sizes,bm", [([3, 0, 130], 128), ([0, 0, 5], 64), ([64, 65, 1], 64),
                                      ([1756, 764, 470, 333, 254, 204, 170, 145], 128), ([0] * 7 + [9], 128),
                                      ([129, 0, 0, 1], 16)])
def test_grouped_block_bit_exact(sizes, bm):
    want = oracle.grouped_tile_map(sizes, bm)
    for b, w in enumerate(want):
        assert qg.gemm_grouped_block(sizes, bm, b) == w
    # past the last block the map yields no rows
    for b in range(len(want), len(want) + len(sizes) + 2):
        assert qg.gemm_grouped_block(sizes, bm, b)[2] == 0


def test_gemm_create_without_gpu_reports_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import ctypes
    h = ctypes.c_void_p()
    assert qg.lib().gemm_create(ctypes.byref(h)) in (qg.GEMM_ERR_CUDA, qg.GEMM_ERR_UNSUPPORTED)
