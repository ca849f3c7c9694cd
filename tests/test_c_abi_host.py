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


CSRC = os.path.join(ROOT, "bit_weight_only_wise_b300", "csrc")
NVCC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
SAN = "-fsanitize=address,-fsanitize=undefined,-fno-sanitize-recover=undefined,-fno-omit-frame-pointer"


def test_host_code_under_address_and_undefined_behaviour_sanitizers(tmp_path):
    # The library's host code (validation, size arithmetic, dispatch up to the
    # launch) built with ASan and UBSan, device code as PTX only; the C
    # program's checks and its size fuzz then run with every overflow, bad
    # shift, division by zero or out-of-bounds access aborting the process.
    _need("gcc")
    if not os.path.exists(NVCC):
        pytest.skip("nvcc not available")
    sources = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    procs = [subprocess.Popen([NVCC, "-O1", "-g", "-std=c++17", "-Xcompiler", "-fPIC," + SAN, "-I", INCLUDE, "-I",
                               CSRC, "--expt-relaxed-constexpr", "-gencode", "arch=compute_103a,code=compute_103a",
                               "-c", os.path.join(CSRC, f), "-o", str(tmp_path / (f[:-3] + ".o"))],
                              stderr=subprocess.PIPE, text=True) for f in sources]
    for p, f in zip(procs, sources):
        _, err = p.communicate(timeout=600)
        assert p.returncode == 0, f + ": " + err[-2000:]
    lib = tmp_path / "libw4a16_san.so"
    subprocess.run([NVCC, "-shared", "-cudart", "static", "-Xcompiler", "-fsanitize=address,-fsanitize=undefined",
                    "-o", str(lib), *[str(tmp_path / (f[:-3] + ".o")) for f in sources]], check=True)
    exe = str(tmp_path / "abi_from_c_san")
    subprocess.run(["gcc", "-std=c11", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
                    *_flags(), SRC, str(lib), f"-Wl,-rpath,{tmp_path}", "-o", exe], check=True)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0", UBSAN_OPTIONS="print_stacktrace=1")
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300, env=env)
    assert out.returncode == 0, (out.stdout + out.stderr)[-4000:]
    assert out.stdout.strip().endswith("ok")
