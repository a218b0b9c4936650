"""In-tree build of libbsolve.so (and the arithmetic-throughput probe) with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked into a
shared library next to this file. Nothing is installed into site-packages.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbsolve.so")
PROBE_LIB = os.path.join(PKG, "libbsolve_probe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--fmad=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]
LIB_SOURCES = ["api.cu", "lu_reg.cu", "lu_reg_f32_row.cu", "lu_reg_f32_col.cu", "lu_reg_f64_row.cu",
               "lu_reg_f64_col.cu", "lu_reg_il_f32_row.cu", "lu_reg_il_f32_col.cu", "lu_reg_il_f64_row.cu",
               "lu_reg_il_f64_col.cu", "lu_rows2.cu", "lu_cta.cu",
               "smem_solvers.cu", "chol_sys.cu", "chol_cluster.cu", "bdsv.cu", "bdmv.cu", "solve.cu",
               "solve_lane.cu"]
PROBE_SOURCES = ["fma_peak.cu"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libbsolve")
    return path


def _newest_input_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "bsolve.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files if os.path.isfile(f))


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    subprocess.check_call(cmd)
    return obj


def _link(objs: list[str], out: str) -> None:
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
    os.replace(tmp, out)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile and link libbsolve.so (and libbsolve_probe.so) if stale; returns the path."""
    os.makedirs(BUILD, exist_ok=True)
    newest = _newest_input_mtime()
    stale = force or any(
        (not os.path.exists(p)) or os.path.getmtime(p) < newest for p in (LIB, PROBE_LIB))
    if not stale:
        return LIB
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with cf.ThreadPoolExecutor(max_workers=len(LIB_SOURCES) + len(PROBE_SOURCES)) as ex:
        lib_objs = list(ex.map(lambda s: _compile(s, extra), LIB_SOURCES))
        probe_objs = list(ex.map(lambda s: _compile(s, extra), PROBE_SOURCES))
    _link(lib_objs, LIB)
    _link(probe_objs, PROBE_LIB)
    return LIB
