"""The C ABI from C: include/w4a16.h compiles as C11 and as C++17 with the host
compilers, a C program that references every declared entry point links
against the built library, and run without a GPU it gets the documented
answers from the host functions and the validation paths (tests/abi_from_c.c).
"""

import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "abi_from_c.c")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(ROOT, "bit_weight_only_wise_b300")
CUDA_INCLUDE = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")


def _need(tool):
    if shutil.which(tool) is None:
        pytest.skip(f"{tool} not available")


def _flags():
    return ["-I", INCLUDE, "-isystem", CUDA_INCLUDE, "-Wall", "-Wextra", "-Werror"]


def test_c_program_references_every_declared_entry_point():
    src = open(os.path.join(INCLUDE, "w4a16.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    declared = set(re.findall(r"^\s*(?:w4a16_status|size_t|const char\*)\s+(\w+)\s*\(", src, flags=re.M))
    assert declared
    prog = open(SRC).read()
    for name in declared:
        assert f"(fn_t){name}" in prog, name


def test_header_compiles_as_c_and_cxx():
    _need("gcc")
    _need("g++")
    subprocess.run(["gcc", "-std=c11", "-fsyntax-only", *_flags(), SRC], check=True)
    subprocess.run(["g++", "-std=c++17", "-fsyntax-only", "-x", "c++", *_flags(), SRC], check=True)


def test_c_program_links_and_runs_without_gpu(tmp_path):
    _need("gcc")
    if not os.path.exists(os.path.join(LIBDIR, "libw4a16.so")):
        pytest.fail("libw4a16.so is not built (python -c 'import __graft_entry__ as g; g.build()')")
    exe = str(tmp_path / "abi_from_c")
    subprocess.run(["gcc", "-std=c11", *_flags(), SRC, "-L", LIBDIR, "-lw4a16", f"-Wl,-rpath,{LIBDIR}", "-o", exe],
                   check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip().endswith("ok")
