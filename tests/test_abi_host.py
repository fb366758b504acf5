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


def test_binding_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of gemm_op_t, gemm_layout_t and gemm_workspace_t have
    the header's sizes and field offsets (compiled with the host C compiler),
    and the binding's enum values are the header's."""
    import ctypes
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    structs = {"gemm_op_t": qg.gemm_op_t, "gemm_layout_t": qg.gemm_layout_t, "gemm_workspace_t": qg.gemm_workspace_t}
    lines = []
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{name}.{field} %zu\\n", offsetof({name}, {field}));')
    consts = ["GEMM_F32", "GEMM_F16", "GEMM_BF16", "GEMM_S4", "GEMM_S8", "GEMM_E4M3", "GEMM_E5M2", "GEMM_EPILOGUE_BIAS", "GEMM_EPILOGUE_RELU",
              "GEMM_EPILOGUE_GELU", "GEMM_DISPATCH_MEASURE", "GEMM_BARRIERS_SIZE", "GEMM_PARTIALS_SIZE",
              "GEMM_NOALLOC_BARRIERS_SIZE", "GEMM_NOALLOC_PARTIALS_SIZE"]
    lines += [f'printf("{c} %d\\n", (int){c});' for c in consts]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "gemm.h"\nint main(void) {\n' +
                   "\n".join(lines) + "\nreturn 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = dict(line.rsplit(" ", 1) for line in subprocess.check_output([str(exe)], text=True).splitlines())
    for name, cls in structs.items():
        assert int(got[f"{name} size"]) == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert int(got[f"{name}.{field}"]) == getattr(cls, field).offset, f"{name}.{field}"
    for c in consts:
        assert int(got[c]) == getattr(qg, c), c


@pytest.mark.parametrize("args,want", [
    # the benchmark workloads on a 152-SM GB300 with the 32 MB partials buffer
    ((256, 256, 256, qg.GEMM_F16, qg.GEMM_F16, qg.GEMM_F32), "umma_bn128/splitk8"),
    ((4096, 4096, 4096, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16), "umma2_bn224/dp"),
    ((1, 4096, 14336, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16), "gemv"),
    ((16, 4096, 14336, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16), "umma_bn16_swap/splitk4"),
    ((64, 4096, 14336, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16), "umma_bn64_swap/splitk4"),
    ((128, 11008, 4096, qg.GEMM_BF16, qg.GEMM_S4, qg.GEMM_BF16, 0, 128), "umma_dq_bn128/streamk"),
    ((1, 11008, 4096, qg.GEMM_BF16, qg.GEMM_S4, qg.GEMM_BF16, 0, 128), "gemv"),
    ((4096, 14336, 4096, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16, 0, 0, 8), "umma2_grouped_bn256/dp"),
])
def test_heuristic_choices_of_the_workloads(args, want):
    assert qg.gemm_heuristic_choice(*args) == want


def test_heuristic_choice_rejects_bad_arguments():
    with pytest.raises(qg.GemmError):
        qg.gemm_heuristic_choice(0, 16, 16, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16)
    with pytest.raises(qg.GemmError):
        qg.gemm_heuristic_choice(16, 16, 16, qg.GEMM_BF16, qg.GEMM_F16, qg.GEMM_BF16)
    # a workspace too small for a split falls back to the unsplit schedule
    assert qg.gemm_heuristic_choice(16, 4096, 14336, qg.GEMM_BF16, qg.GEMM_BF16, qg.GEMM_BF16,
                                    partials_size=0) == "umma_bn16_swap/dp"


def test_small_m_kernel_limits(monkeypatch):
    # M <= 2 by default; U scales and grouped problems never take it; the
    # environment limit moves or removes it
    bf = qg.GEMM_BF16
    assert qg.gemm_heuristic_choice(2, 4096, 4096, bf, bf, bf) == "gemv"
    assert qg.gemm_heuristic_choice(3, 4096, 4096, bf, bf, bf) != "gemv"
    assert qg.gemm_heuristic_choice(1, 4096, 4096, bf, bf, bf, quant_a_group=128) != "gemv"
    assert qg.gemm_heuristic_choice(1, 4096, 4096, bf, bf, bf, num_experts=4) != "gemv"
    assert qg.gemm_heuristic_choice(1, 4096, 4096, bf, qg.GEMM_S4, qg.GEMM_S8, quant_b_group=64) == "gemv"
    monkeypatch.setenv("GEMM_GEMV_MAX_M", "0")
    assert qg.gemm_heuristic_choice(1, 4096, 4096, bf, bf, bf) != "gemv"
    monkeypatch.setenv("GEMM_GEMV_MAX_M", "8")
    assert qg.gemm_heuristic_choice(8, 4096, 4096, bf, bf, bf) == "gemv"
    assert qg.gemm_heuristic_choice(9, 4096, 4096, bf, bf, bf) != "gemv"


def test_checked_build_compiles(tmp_path):
    """The device-side bounds checks (QG_DEVICE_CHECKS) compile for sm_103a
    (one kernel instantiation; the checks live in the code every kernel
    shares), and the regular library reports that it is not the checked
    build."""
    import shutil
    import subprocess

    from quantized_gemm_tcgen05_gb300 import _build

    if shutil.which(_build._nvcc()) is None and not os.path.exists(_build._nvcc()):
        pytest.skip("no nvcc")
    for src in ("umma_gemm_bn16.cu",):  # the checks live in the shared epilogue / unit code
        cmd = [_build._nvcc(), "-gencode", _build.GENCODE, "-O1", "-std=c++17", "-DQG_DEVICE_CHECKS", "-I",
               os.path.join(ROOT, "include"), "-I", _build.CSRC, "-c", os.path.join(_build.CSRC, src), "-o",
               str(tmp_path / (src + ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
    assert qg.lib().gemm_checked_build() == 0
