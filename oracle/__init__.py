"""CPU oracle for the FP8 (E4M3) block-scaled GEMM library.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library itself
never does, and this package never imports the library.

The arithmetic lives in ``oracle.c`` (plain C, fp64, threads over output rows);
this module compiles it with gcc and wraps it with ctypes over numpy arrays.
Each wrapper names the passage of the source pages that it follows in the C
file's comments:

- E4M3 decode / RNE-satfinite encode (``float8_e4m3fn``; format paragraph of
  "Optimizing FP8 GEMM kernels in JAX with Triton for Blackwell GPUs" and the
  dtype in "Triton FP8 CUTLASS-named kernel benchmarking"); the same for E5M2,
  the other FP8 format that paragraph weighs, E2M1 (FP4) and E2M3 / E3M2
  (FP6), the element formats of the micro-scaling variants (Triton tutorial
  ch. 12, 12.6.1 and 12.6.4), and GEMMs whose operands mix them (``fmt``
  arguments: E4M3 = 0, E5M2 = 1, E2M1 = 2, E2M3 = 3, E3M2 = 4).
- per-tensor (s = amax/448) and 1x32 power-of-two block quantisation
  (microscaling paragraph of the JAX/Blackwell page; Triton tutorial ch. 12,
  section 12.6.1, MXFP8).
- the GEMM C = (sA A)(sB B)^T, its grouped (MoE) form, the grouped raster
  tile order ("GROUP_M" swizzle, Triton tutorial ch. 12, section 12.7) and the
  tolerance bound 2^-8 * sum_k |sA a||sB b| + 1 bf16 ulp.

Parity unpinned: the rounding order of the tensor core's fp32 accumulation
(only the tolerance bounds it).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

OUT_BF16 = 0
OUT_F32 = 1
E4M3 = 0
E5M2 = 1
E2M1 = 2
E2M3 = 3
E3M2 = 4
ACT_NONE = 0
ACT_RELU = 1
ACT_GELU = 2


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, pthreads)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fvisibility=hidden",
               "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            i32 = ctypes.c_int32
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_table.argtypes = [P]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e5m2_decode.restype = ctypes.c_double
            lib.oracle_e5m2_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e5m2_table.argtypes = [P]
            lib.oracle_e2m1_decode.restype = ctypes.c_double
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_table.argtypes = [P]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
            for f in ("e2m3", "e3m2"):
                getattr(lib, f"oracle_{f}_decode").restype = ctypes.c_double
                getattr(lib, f"oracle_{f}_decode").argtypes = [ctypes.c_uint8]
                getattr(lib, f"oracle_{f}_table").argtypes = [P]
                getattr(lib, f"oracle_{f}_encode").restype = ctypes.c_uint8
                getattr(lib, f"oracle_{f}_encode").argtypes = [ctypes.c_float]
            lib.oracle_e5m2_encode.restype = ctypes.c_uint8
            lib.oracle_e5m2_encode.argtypes = [ctypes.c_float]
            lib.oracle_quantize_tensor_fmt.argtypes = [P, i64, i64, ctypes.c_int, P, P]
            lib.oracle_pow2_scale_fmt.restype = ctypes.c_float
            lib.oracle_pow2_scale_fmt.argtypes = [ctypes.c_float, ctypes.c_int]
            lib.oracle_quantize_block32_fmt.argtypes = [P, i64, i64, ctypes.c_int, P, P]
            lib.oracle_quantize_block32_literal.argtypes = [P, i64, i64, ctypes.c_int, P, P]
            lib.oracle_act.restype = ctypes.c_double
            lib.oracle_act.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.oracle_gemm_ex.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                           ctypes.c_int, i64, i64, i64, ctypes.c_int, P, P, P,
                                           ctypes.c_int]
            lib.oracle_gemm_sample_ex.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, P, ctypes.c_int, i64, i64, i64,
                                                  ctypes.c_int, P, P, i64, P, P, P, ctypes.c_int]
            lib.oracle_gemm_fmt.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            i64, i64, i64, ctypes.c_int, P, P, P, ctypes.c_int]
            lib.oracle_gemm_sample_fmt.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, i64, i64, i64, ctypes.c_int, P,
                                                   P, i64, P, P, P, ctypes.c_int]
            lib.oracle_bf16_round.restype = ctypes.c_float
            lib.oracle_bf16_round.argtypes = [ctypes.c_double]
            lib.oracle_bf16_ulp.restype = ctypes.c_double
            lib.oracle_bf16_ulp.argtypes = [ctypes.c_double]
            lib.oracle_quantize_tensor.argtypes = [P, i64, i64, P, P]
            lib.oracle_pow2_scale.restype = ctypes.c_float
            lib.oracle_pow2_scale.argtypes = [ctypes.c_float]
            lib.oracle_quantize_block32.argtypes = [P, i64, i64, P, P]
            lib.oracle_gemm.argtypes = [P, P, P, P, ctypes.c_int, i64, i64, i64, ctypes.c_int,
                                        P, P, P, ctypes.c_int]
            lib.oracle_gemm_sample.argtypes = [P, P, P, P, ctypes.c_int, i64, i64, i64,
                                               ctypes.c_int, P, P, i64, P, P, P, ctypes.c_int]
            lib.oracle_grouped_offsets.argtypes = [P, i32, P]
            lib.oracle_raster.argtypes = [i64, i64, i64, i64, P, P]
            lib.oracle_tile_map.restype = i64
            lib.oracle_tile_map.argtypes = [i64, i64, i64, i64, i64, P, i64]
            lib.oracle_grouped_tile_map.restype = i64
            lib.oracle_grouped_tile_map.argtypes = [P, i32, i64, i64, i64, i64, P, i64]
            lib.oracle_grouped_gemm.argtypes = [P, P, P, P, P, i32, i64, i64, ctypes.c_int, P,
                                                P, P, ctypes.c_int]
            lib.oracle_quantize_nvfp4.argtypes = [P, i64, i64, P, P, P]
            lib.oracle_gemm_nvfp4.argtypes = [P, P, P, P, ctypes.c_float, ctypes.c_float, P,
                                              ctypes.c_int, i64, i64, i64, ctypes.c_int, P, P, P,
                                              ctypes.c_int]
            lib.oracle_gemm_nvfp4_sample.argtypes = [P, P, P, P, ctypes.c_float, ctypes.c_float,
                                                     P, ctypes.c_int, i64, i64, i64, ctypes.c_int,
                                                     P, P, i64, P, P, P, ctypes.c_int]
            lib.oracle_gemm_flops.restype = ctypes.c_double
            lib.oracle_gemm_flops.argtypes = [i64, i64, i64]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _threads(threads):
    return int(threads if threads else (os.cpu_count() or 1))


# --------------------------------------------------------------------- E4M3
def e4m3_decode(code: int) -> float:
    return float(_L().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_table() -> np.ndarray:
    out = np.zeros(256, dtype=np.float64)
    _L().oracle_e4m3_table(_p(out))
    return out


def e4m3_encode(y: float) -> int:
    return int(_L().oracle_e4m3_encode(float(np.float32(y))))


def e5m2_decode(code: int) -> float:
    return float(_L().oracle_e5m2_decode(int(code) & 0xFF))


def e5m2_table() -> np.ndarray:
    out = np.zeros(256, dtype=np.float64)
    _L().oracle_e5m2_table(_p(out))
    return out


def e5m2_encode(y: float) -> int:
    return int(_L().oracle_e5m2_encode(float(np.float32(y))))


def e2m1_decode(code: int) -> float:
    return float(_L().oracle_e2m1_decode(int(code) & 0xFF))


def e2m1_table() -> np.ndarray:
    out = np.zeros(256, dtype=np.float64)
    _L().oracle_e2m1_table(_p(out))
    return out


def e2m1_encode(y: float) -> int:
    return int(_L().oracle_e2m1_encode(float(np.float32(y))))


def fp6_table(fmt: int) -> np.ndarray:
    """Values of the 256 byte codes of E2M3 (fmt 3) or E3M2 (fmt 4); the high
    two bits of a byte are ignored."""
    out = np.zeros(256, dtype=np.float64)
    getattr(_L(), "oracle_e2m3_table" if fmt == E2M3 else "oracle_e3m2_table")(_p(out))
    return out


def fp6_encode(y: float, fmt: int) -> int:
    fn = _L().oracle_e2m3_encode if fmt == E2M3 else _L().oracle_e3m2_encode
    return int(fn(float(np.float32(y))))


def bf16_round(x: float) -> float:
    return float(_L().oracle_bf16_round(float(x)))


def bf16_ulp(x: float) -> float:
    return float(_L().oracle_bf16_ulp(float(x)))


# --------------------------------------------------------------- quantisers
def quantize_tensor(x: np.ndarray, fmt: int = E4M3):
    """Per-tensor: returns (codes uint8 same shape, scale float32 scalar array)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.zeros(1, dtype=np.float32)
    _L().oracle_quantize_tensor_fmt(_p(x), rows, cols, int(fmt), _p(q), _p(s))
    return q, s


def pow2_scale(amax: float, fmt: int = E4M3) -> float:
    return float(_L().oracle_pow2_scale_fmt(float(np.float32(amax)), int(fmt)))


def quantize_block32(x: np.ndarray, fmt: int = E4M3, literal: bool = False):
    """1x32 along the last axis: returns (codes uint8, scales float32 [rows, cols/32]).
    literal: block scale fl32(amax / fmax) instead of the power of two."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % 32 == 0
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.empty((rows, cols // 32), dtype=np.float32)
    fn = _L().oracle_quantize_block32_literal if literal else _L().oracle_quantize_block32_fmt
    fn(_p(x), rows, cols, int(fmt), _p(q), _p(s))
    return q, s


# --------------------------------------------------------------------- GEMM
def act(y: float, kind: int) -> float:
    """The fused epilogue's activation in fp64 (ACT_NONE, ACT_RELU, ACT_GELU)."""
    return float(_L().oracle_act(float(y), int(kind)))


def gemm(A: np.ndarray, B: np.ndarray, sfa: np.ndarray, sfb: np.ndarray, block: bool,
         out_kind: int = OUT_BF16, want_exact: bool = False, threads=None, a_fmt: int = E4M3,
         b_fmt: int = E4M3, bias=None, act_kind: int = ACT_NONE):
    """C = (sA A)(sB B)^T.  Returns (C_rounded float32 [M,N], bound float64 [M,N], exact|None)."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfa = np.ascontiguousarray(sfa, dtype=np.float32)
    sfb = np.ascontiguousarray(sfb, dtype=np.float32)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    if block:
        assert K % 32 == 0 and sfa.shape == (M, K // 32) and sfb.shape == (N, K // 32)
    else:
        assert sfa.size == 1 and sfb.size == 1
    C = np.empty((M, N), dtype=np.float32)
    bound = np.empty((M, N), dtype=np.float64)
    exact = np.empty((M, N), dtype=np.float64) if want_exact else None
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        assert bias.shape == (N,)
    _L().oracle_gemm_ex(_p(A), _p(B), _p(sfa), _p(sfb), int(bool(block)), int(a_fmt), int(b_fmt),
                        _p(bias) if bias is not None else None, int(act_kind), M, N, K,
                        int(out_kind), _p(C), _p(exact) if exact is not None else None,
                        _p(bound), _threads(threads))
    return C, bound, exact


def gemm_sample(A, B, sfa, sfb, block: bool, pi, pj, out_kind: int = OUT_BF16, threads=None,
                a_fmt: int = E4M3, b_fmt: int = E4M3, bias=None, act_kind: int = ACT_NONE):
    """Only the elements (pi[s], pj[s]).  Returns (C float32 [n], bound float64 [n], exact [n])."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfa = np.ascontiguousarray(sfa, dtype=np.float32)
    sfb = np.ascontiguousarray(sfb, dtype=np.float32)
    pi = np.ascontiguousarray(pi, dtype=np.int64)
    pj = np.ascontiguousarray(pj, dtype=np.int64)
    M, K = A.shape
    N = B.shape[0]
    n = pi.size
    C = np.empty(n, dtype=np.float32)
    bound = np.empty(n, dtype=np.float64)
    exact = np.empty(n, dtype=np.float64)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        assert bias.shape == (N,)
    _L().oracle_gemm_sample_ex(_p(A), _p(B), _p(sfa), _p(sfb), int(bool(block)), int(a_fmt),
                               int(b_fmt), _p(bias) if bias is not None else None, int(act_kind),
                               M, N, K, int(out_kind), _p(pi), _p(pj), n, _p(C), _p(exact),
                               _p(bound), _threads(threads))
    return C, bound, exact


# ----------------------------------------------------------------- NVFP4
def quantize_nvfp4(x: np.ndarray):
    """NVFP4 along the last axis (cols % 16 == 0): returns (E2M1 codes uint8
    [rows, cols], one per byte; E4M3 block-scale codes uint8 [rows, cols/16];
    the tensor scale g, a float)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % 16 == 0
    q = np.empty((rows, cols), dtype=np.uint8)
    sf = np.empty((rows, cols // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    _L().oracle_quantize_nvfp4(_p(x), rows, cols, _p(q), _p(sf), _p(g))
    return q, sf, float(g[0])


def nvfp4_scales(sf_codes: np.ndarray) -> np.ndarray:
    """E4M3 block-scale codes -> their values (exact in fp32)."""
    return e4m3_table()[np.asarray(sf_codes, dtype=np.uint8)].astype(np.float32)


def _bias(bias, N):
    if bias is None:
        return None
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    assert bias.shape == (N,)
    return bias


def gemm_nvfp4(A, B, sfa_codes, sfb_codes, ga: float, gb: float, out_kind: int = OUT_BF16,
               threads=None, bias=None, act_kind: int = ACT_NONE):
    """C = out(act(fl32(fl32(ga gb) * sum_kb16 sa sb sum a b) + bias)) over E2M1
    codes (one per byte).  Returns (C float32 [M,N], bound float64 [M,N], exact [M,N])."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfa = np.ascontiguousarray(nvfp4_scales(sfa_codes))
    sfb = np.ascontiguousarray(nvfp4_scales(sfb_codes))
    M, K = A.shape
    N = B.shape[0]
    assert K % 16 == 0 and sfa.shape == (M, K // 16) and sfb.shape == (N, K // 16)
    C = np.empty((M, N), dtype=np.float32)
    bound = np.empty((M, N), dtype=np.float64)
    exact = np.empty((M, N), dtype=np.float64)
    bias = _bias(bias, N)
    _L().oracle_gemm_nvfp4(_p(A), _p(B), _p(sfa), _p(sfb), float(ga), float(gb),
                           _p(bias) if bias is not None else None, int(act_kind), M, N, K,
                           int(out_kind), _p(C), _p(exact), _p(bound), _threads(threads))
    return C, bound, exact


def gemm_nvfp4_sample(A, B, sfa_codes, sfb_codes, ga: float, gb: float, pi, pj,
                      out_kind: int = OUT_BF16, threads=None, bias=None, act_kind: int = ACT_NONE):
    """Only the elements (pi[s], pj[s]) of gemm_nvfp4."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfa = np.ascontiguousarray(nvfp4_scales(sfa_codes))
    sfb = np.ascontiguousarray(nvfp4_scales(sfb_codes))
    pi = np.ascontiguousarray(pi, dtype=np.int64)
    pj = np.ascontiguousarray(pj, dtype=np.int64)
    M, K = A.shape
    N = B.shape[0]
    n = pi.size
    C = np.empty(n, dtype=np.float32)
    bound = np.empty(n, dtype=np.float64)
    exact = np.empty(n, dtype=np.float64)
    bias = _bias(bias, N)
    _L().oracle_gemm_nvfp4_sample(_p(A), _p(B), _p(sfa), _p(sfb), float(ga), float(gb),
                                  _p(bias) if bias is not None else None, int(act_kind), M, N, K,
                                  int(out_kind), _p(pi), _p(pj), n, _p(C), _p(exact), _p(bound),
                                  _threads(threads))
    return C, bound, exact


def grouped_offsets(counts) -> np.ndarray:
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    out = np.zeros(counts.size + 1, dtype=np.int32)
    _L().oracle_grouped_offsets(_p(counts), counts.size, _p(out))
    return out


def raster(t: int, npm: int, npn: int, G: int):
    pm = ctypes.c_int64()
    pn = ctypes.c_int64()
    _L().oracle_raster(t, npm, npn, G, ctypes.byref(pm), ctypes.byref(pn))
    return pm.value, pn.value


def tile_map(M: int, N: int, BM: int, BN: int, G: int) -> np.ndarray:
    T = ((M + BM - 1) // BM) * ((N + BN - 1) // BN)
    out = np.zeros((max(T, 1), 2), dtype=np.int64)
    _L().oracle_tile_map(M, N, BM, BN, G, _p(out), T)
    return out[:T]


def grouped_tile_map(counts, N: int, BM: int, BN: int, G: int) -> np.ndarray:
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    npn = (N + BN - 1) // BN
    cap = int(sum(((int(c) + BM - 1) // BM) * npn for c in counts))
    out = np.zeros((max(cap, 1), 4), dtype=np.int32)
    T = _L().oracle_grouped_tile_map(_p(counts), counts.size, N, BM, BN, G, _p(out), cap)
    assert T == cap
    return out[:T]


def grouped_gemm(A, B, sfa, sfb, counts, out_kind: int = OUT_BF16, want_exact=False,
                 threads=None):
    """A [sum M_e, K], B [E, N, K], sfa [sum M_e, K/32], sfb [E, N, K/32]."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sfa = np.ascontiguousarray(sfa, dtype=np.float32)
    sfb = np.ascontiguousarray(sfb, dtype=np.float32)
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    E, N, K = B.shape
    rows = A.shape[0]
    assert counts.size == E and int(counts.sum()) == rows
    C = np.zeros((rows, N), dtype=np.float32)
    bound = np.zeros((rows, N), dtype=np.float64)
    exact = np.zeros((rows, N), dtype=np.float64) if want_exact else None
    _L().oracle_grouped_gemm(_p(A), _p(B), _p(sfa), _p(sfb), _p(counts), E, N, K, int(out_kind),
                             _p(C), _p(exact) if exact is not None else None, _p(bound),
                             _threads(threads))
    return C, bound, exact


def gemm_flops(M: int, N: int, K: int) -> float:
    return float(_L().oracle_gemm_flops(M, N, K))
