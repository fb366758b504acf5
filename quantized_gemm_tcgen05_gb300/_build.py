"""Build the GEMM library (libqgemm.so) in-tree for sm_103a.

CUDA sources are compiled by nvcc for ``-gencode arch=compute_103a,code=sm_103a``,
host sources by g++, in parallel, then linked into one shared library with the
CUDA runtime linked statically.  Objects go to ``_build/`` beside the package.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqgemm.so")
# the checked debug build: device-side bounds checks compiled in (QG_DEVICE_CHECKS)
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libqgemm_checked.so")
GENCODE = "arch=compute_103a,code=sm_103a"


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _cuda_include():
    return os.path.join(os.path.dirname(os.path.dirname(_nvcc())), "include")


def sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _headers_mtime():
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    paths.append(os.path.join(ROOT, "include", "gemm.h"))
    return max(os.path.getmtime(p) for p in paths)


def _compile(cmd, out, src, hdr_mtime, force):
    if not force and os.path.exists(out):
        m = os.path.getmtime(out)
        if m >= os.path.getmtime(src) and m >= hdr_mtime:
            return None
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        return f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
    return None


def build(force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    """Build libqgemm.so, or with checks=True the checked debug build
    libqgemm_checked.so (device-side bounds checks, see gemm_checked_build)."""
    build_dir, lib_path = (BUILD_CHECKED, LIB_CHECKED) if checks else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    inc = ["-I", os.path.join(ROOT, "include"), "-I", CSRC] + (["-DQG_DEVICE_CHECKS"] if checks else [])
    cu, cpp = sources()
    hdr = _headers_mtime()
    jobs = []
    for f in cu:
        out = os.path.join(build_dir, f + ".o")
        cmd = [nvcc, "-gencode", GENCODE, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
               "-Xcompiler", "-Wall", *inc, "-c", os.path.join(CSRC, f), "-o", out]
        jobs.append((cmd, out, os.path.join(CSRC, f)))
    for f in cpp:
        out = os.path.join(build_dir, f + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", *inc, "-I", _cuda_include(), "-c",
               os.path.join(CSRC, f), "-o", out]
        jobs.append((cmd, out, os.path.join(CSRC, f)))
    with cf.ThreadPoolExecutor(max_workers=max(2, min(len(jobs), os.cpu_count() or 4))) as ex:
        errs = [e for e in ex.map(lambda j: _compile(*j, hdr, force), jobs) if e]
    if errs:
        raise RuntimeError("libqgemm build failed:\n" + "\n".join(errs))
    objs = [j[1] for j in jobs]
    if force or not os.path.exists(lib_path) or any(os.path.getmtime(o) > os.path.getmtime(lib_path) for o in objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc, "-shared", "-gencode", GENCODE, "-Xcompiler", "-fPIC", "-o", tmp, *objs,
               "-cudart", "static", "-lpthread", "-ldl", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"libqgemm link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    if verbose:
        print("built", lib_path)
    return lib_path


if __name__ == "__main__":
    import sys

    build(verbose=True, checks="--checks" in sys.argv[1:])
