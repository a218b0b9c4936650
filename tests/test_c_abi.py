"""The boundary from C: a C99 program (tests/c_abi/abi_check.c) compiles against
include/bsolve.h with warnings as errors, links libbsolve.so and checks the statuses of
every call that returns before a launch; the header also compiles as C++ (its extern "C"
block). No GPU is used."""
import os
import shutil
import subprocess

import pytest

from dense_linear_solvers_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_check.c")


@pytest.fixture(scope="module")
def libdir():
    return os.path.dirname(_build.build())


def test_c99_program_links_and_checks_statuses(libdir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_check")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Wpedantic", "-Werror", "-I", INCLUDE,
                    SRC, "-L", libdir, "-lbsolve", f"-Wl,-rpath,{libdir}", "-o", exe],
                   check=True, capture_output=True, text=True)
    env = dict(os.environ)
    cuda_lib = "/usr/local/cuda/lib64"
    env["LD_LIBRARY_PATH"] = os.pathsep.join(p for p in (libdir, cuda_lib,
                                                         env.get("LD_LIBRARY_PATH")) if p)
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr + r.stdout
    assert "all checks passed" in r.stdout


def test_header_compiles_as_cxx(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "use.cpp"
    src.write_text('#include "bsolve.h"\nint main() { return bs_version() > 0 ? 0 : 1; }\n')
    subprocess.run([cxx, "-std=c++17", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I",
                    INCLUDE, str(src)], check=True, capture_output=True, text=True)
