"""The C ABI used from plain C99 (tests/c/abi_gemm.c): the header compiles
as strict C99 with -pedantic (CUDA's own headers taken as system headers)
on the CPU, and the program, linked against the library and the
CUDA runtime, quantises and multiplies on the GPU with results within the
oracle's tolerance (GPU)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_gemm.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _gcc():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    return gcc


def test_header_is_c99():
    r = subprocess.run([_gcc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        "-isystem", os.path.join(CUDA, "include"), SRC],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_program_gemm_matches_oracle(tmp_path, fp8g, oracle_lib):
    import oracle
    from gpu_util import assert_within
    libdir = os.path.dirname(fp8g.LIB_PATH)
    exe = str(tmp_path / "abi_gemm")
    r = subprocess.run([_gcc(), "-std=c99", "-O2", "-I", os.path.join(ROOT, "include"),
                        "-isystem", os.path.join(CUDA, "include"), SRC, "-o", exe,
                        "-L", libdir, "-lfp8g", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                        "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = str(tmp_path / "out.bin")
    M, N, K = 300, 264, 512
    r = subprocess.run([exe, str(M), str(N), str(K), out], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = open(out, "rb").read()
    dims = np.frombuffer(raw[:24], dtype=np.int64)
    assert tuple(dims) == (M, N, K)
    body = np.frombuffer(raw[24:], dtype=np.float32)
    a = body[:M * K].reshape(M, K)
    b = body[M * K:M * K + N * K].reshape(N, K)
    c = body[M * K + N * K:].reshape(M, N)
    qa, sa = oracle.quantize_block32(a)
    qb, sb = oracle.quantize_block32(b)
    ref, bound, _ = oracle.gemm(qa, qb, sa, sb, True, oracle.OUT_BF16)
    assert_within(c, ref, bound, "C program")
