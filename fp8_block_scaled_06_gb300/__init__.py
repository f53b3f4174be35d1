"""Python binding of the FP8 (E4M3) GEMM C ABI (``include/fp8gemm.h``).

Argument marshalling only: every computation runs in the CUDA kernels of
``libfp8g.so`` (built in-tree for sm_103a by ``buildlib.py``).  Tensor arguments
may be torch tensors (their ``data_ptr()`` is passed) or raw integer device
addresses.  ``stream`` defaults to torch's current CUDA stream.  A non-OK
status raises :class:`Fp8gError` carrying the ``fp8g_status`` code.

There is no fallback: if the shared library is missing or cannot be loaded,
the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8g.so")

FP8G_OK = 0
FP8G_ERR_INVALID_ARG = 1
FP8G_ERR_ALIGNMENT = 2
FP8G_ERR_UNSUPPORTED_SHAPE = 3
FP8G_ERR_SCALE_FORMAT = 4
FP8G_ERR_CUDA = 5
FP8G_ERR_TIMEOUT = 6
FP8G_ERR_DEVICE = 7

FP8G_OUT_BF16 = 0
FP8G_OUT_F32 = 1
FP8G_E4M3 = 0
FP8G_E5M2 = 1
FP8G_E2M1 = 2
FP8G_E2M3 = 3
FP8G_E3M2 = 4
FP8G_BLOCK32_LITERAL = 33
FP8G_IN_F32 = 0
FP8G_IN_BF16 = 1
FP8G_ACT_NONE = 0
FP8G_ACT_RELU = 1
FP8G_ACT_GELU = 2
FP8G_MAX_EXPERTS = 64
FP8G_QUANT_FUSED = 1

# Every symbol include/fp8gemm.h declares.
EXPORTS = (
    "fp8_gemm", "fp8_gemm_blockscaled", "fp8_gemm_blockscaled_noalloc", "fp8_grouped_gemm", "fp8g_grouped_plan",
    "fp8g_gemm_plan", "fp8g_quantize_e4m3", "fp8g_quantize", "fp8_gemm_fmt",
    "fp8_gemm_blockscaled_fmt", "fp8_grouped_gemm_fmt", "fp8_gemm_ex", "fp8_gemm_blockscaled_ex",
    "fp8_grouped_gemm_ex", "fp8_grouped_gemm_scatter", "fp8_grouped_gemm_quant",
    "fp8g_quantize_rows",
    "fp8_gemm_blockscaled_promote", "fp8g_quantize_nvfp4", "fp8_gemm_nvfp4",
    "fp8_grouped_gemm_nvfp4", "fp8g_wait_selftest",
    "fp8g_kernel_timing_begin", "fp8g_kernel_timing_end",
    "fp8_gemm_status", "fp8g_status_string",
    "fp8g_set_wait_timeout_ms", "fp8g_shutdown", "fp8g_version",
)


class Fp8gError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {fp8g_status_string(status)} (status {status})")


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    from . import buildlib
    return buildlib.build(force=force)


def load():
    """Load libfp8g.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "fp8_block_scaled_06_gb300.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int32
        st = ctypes.c_int
        lib.fp8_gemm.restype = st
        lib.fp8_gemm.argtypes = [P, P, P, P, P, ctypes.c_int, i64, i64, i64, P]
        lib.fp8_gemm_blockscaled.restype = st
        lib.fp8_gemm_blockscaled.argtypes = [P, P, P, P, P, ctypes.c_int, i64, i64, i64, P]
        lib.fp8_gemm_blockscaled_noalloc.restype = st
        lib.fp8_gemm_blockscaled_noalloc.argtypes = [P, P, P, P, P, ctypes.c_int, i64, i64, i64, P]
        lib.fp8_grouped_gemm.restype = st
        lib.fp8_grouped_gemm.argtypes = [P, P, P, P, P, ctypes.c_int, P, i32, i64, i64, i64, P,
                                         P, P]
        lib.fp8g_grouped_plan.restype = st
        lib.fp8g_grouped_plan.argtypes = [i64, i64, i64, i32, P, P, P, P]
        lib.fp8g_gemm_plan.restype = st
        lib.fp8g_gemm_plan.argtypes = [ctypes.c_int, i64, i64, i64, P, P, P, P, P]
        lib.fp8g_quantize_e4m3.restype = st
        lib.fp8g_quantize_e4m3.argtypes = [P, i64, i64, i32, P, P, P]
        lib.fp8g_quantize.restype = st
        lib.fp8g_quantize.argtypes = [P, i64, i64, i32, i32, P, P, P]
        lib.fp8g_quantize_nvfp4.restype = st
        lib.fp8g_quantize_nvfp4.argtypes = [P, i32, i64, i64, P, P, P, P]
        lib.fp8_gemm_nvfp4.restype = st
        lib.fp8_gemm_nvfp4.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, P, i32, i64, i64, i64,
                                       P]
        lib.fp8_grouped_gemm_nvfp4.restype = st
        lib.fp8_grouped_gemm_nvfp4.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, P, i32, P, i32,
                                               i64, i64, i64, P, P, P]
        lib.fp8_gemm_fmt.restype = st
        lib.fp8_gemm_fmt.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, i64, i64, i64, P]
        lib.fp8_gemm_blockscaled_fmt.restype = st
        lib.fp8_gemm_blockscaled_fmt.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, i64, i64,
                                                 i64, P]
        lib.fp8_gemm_ex.restype = st
        lib.fp8_gemm_ex.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, i32, i64, i64, i64,
                                    P]
        lib.fp8_gemm_blockscaled_ex.restype = st
        lib.fp8_gemm_blockscaled_ex.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, i32, i64,
                                                i64, i64, P]
        lib.fp8_grouped_gemm_ex.restype = st
        lib.fp8_grouped_gemm_ex.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, i32, P, i32,
                                            i64, i64, i64, P, P, P]
        lib.fp8_grouped_gemm_scatter.restype = st
        lib.fp8_grouped_gemm_scatter.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, i32, P,
                                                 i32, i64, i64, i64, P, i64, P, P, P]
        lib.fp8_grouped_gemm_quant.restype = st
        lib.fp8_grouped_gemm_quant.argtypes = [P, i32, i64, P, P, P, P, ctypes.c_int, i32, P, i32,
                                               P, i32, i64, i64, i64, P, i64, P, P, P, P, i32, P]
        lib.fp8_gemm_blockscaled_promote.restype = st
        lib.fp8_gemm_blockscaled_promote.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, i32,
                                                     i64, i64, i64, P]
        lib.fp8g_kernel_timing_begin.restype = st
        lib.fp8g_kernel_timing_begin.argtypes = [i32]
        lib.fp8g_kernel_timing_end.restype = st
        lib.fp8g_kernel_timing_end.argtypes = [P, i32, P]
        lib.fp8g_wait_selftest.restype = st
        lib.fp8g_wait_selftest.argtypes = [ctypes.c_uint32, P]
        lib.fp8g_quantize_rows.restype = st
        lib.fp8g_quantize_rows.argtypes = [P, i32, i64, i64, P, i64, i32, i32, P, P, P]
        lib.fp8_grouped_gemm_fmt.restype = st
        lib.fp8_grouped_gemm_fmt.argtypes = [P, P, P, P, P, ctypes.c_int, i32, i32, P, i32, i64,
                                             i64, i64, P, P, P]
        lib.fp8_gemm_status.restype = st
        lib.fp8_gemm_status.argtypes = [P, P]
        lib.fp8g_status_string.restype = ctypes.c_char_p
        lib.fp8g_status_string.argtypes = [st]
        lib.fp8g_set_wait_timeout_ms.restype = None
        lib.fp8g_set_wait_timeout_ms.argtypes = [ctypes.c_uint32]
        lib.fp8g_shutdown.restype = None
        lib.fp8g_shutdown.argtypes = []
        lib.fp8g_version.restype = ctypes.c_int
        lib.fp8g_version.argtypes = []
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != FP8G_OK:
        raise Fp8gError(status, where)


def fp8g_status_string(status: int) -> str:
    return load().fp8g_status_string(int(status)).decode()


def fp8_gemm(A, B, scale_a, scale_b, C, out: int, M: int, N: int, K: int, stream=None):
    _check(load().fp8_gemm(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), _ptr(C), int(out),
                           M, N, K, _stream(stream)), "fp8_gemm")


def fp8_gemm_blockscaled(A, B, sfa, sfb, C, out: int, M: int, N: int, K: int, stream=None):
    _check(load().fp8_gemm_blockscaled(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C), int(out),
                                       M, N, K, _stream(stream)), "fp8_gemm_blockscaled")


def fp8_gemm_blockscaled_noalloc(A, B, sfa, sfb, C, out: int, M: int, N: int, K: int,
                                 stream=None):
    """Allocation-free fp8_gemm_blockscaled (packed scales in the library's fixed array)."""
    _check(load().fp8_gemm_blockscaled_noalloc(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C),
                                               int(out), M, N, K, _stream(stream)),
           "fp8_gemm_blockscaled_noalloc")


def fp8_grouped_gemm(A, B, sfa, sfb, C, out: int, counts, E: int, N: int, K: int,
                     total_rows: int, offsets_out=None, tile_map_out=None, stream=None):
    _check(load().fp8_grouped_gemm(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C), int(out),
                                   _ptr(counts), E, N, K, total_rows, _ptr(offsets_out),
                                   _ptr(tile_map_out), _stream(stream)), "fp8_grouped_gemm")


def fp8g_grouped_plan(N: int, K: int, total_rows: int, E: int) -> dict:
    BM, BN, G = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    T = ctypes.c_int64()
    _check(load().fp8g_grouped_plan(N, K, total_rows, E, ctypes.byref(BM), ctypes.byref(BN),
                                    ctypes.byref(G), ctypes.byref(T)), "fp8g_grouped_plan")
    return {"BM": BM.value, "BN": BN.value, "G": G.value, "max_tiles": T.value}


def fp8g_gemm_plan(block: int, M: int, N: int, K: int) -> dict:
    BM, BN, G, S, grid = (ctypes.c_int32() for _ in range(5))
    _check(load().fp8g_gemm_plan(int(block), M, N, K, ctypes.byref(BM), ctypes.byref(BN),
                                 ctypes.byref(G), ctypes.byref(S), ctypes.byref(grid)),
           "fp8g_gemm_plan")
    return {"BM": BM.value, "BN": BN.value, "G": G.value, "split_k": S.value, "grid": grid.value}


def fp8g_quantize_e4m3(x, rows: int, cols: int, block: int, q, scales, stream=None):
    _check(load().fp8g_quantize_e4m3(_ptr(x), rows, cols, int(block), _ptr(q), _ptr(scales),
                                     _stream(stream)), "fp8g_quantize_e4m3")


def fp8g_quantize(x, rows: int, cols: int, block: int, fmt: int, q, scales, stream=None):
    _check(load().fp8g_quantize(_ptr(x), rows, cols, int(block), int(fmt), _ptr(q),
                                _ptr(scales), _stream(stream)), "fp8g_quantize")


def fp8_gemm_fmt(A, B, scale_a, scale_b, C, out: int, a_fmt: int, b_fmt: int, M: int, N: int,
                 K: int, stream=None):
    _check(load().fp8_gemm_fmt(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), _ptr(C), int(out),
                               int(a_fmt), int(b_fmt), M, N, K, _stream(stream)), "fp8_gemm_fmt")


def fp8_gemm_blockscaled_fmt(A, B, sfa, sfb, C, out: int, a_fmt: int, b_fmt: int, M: int,
                             N: int, K: int, stream=None):
    _check(load().fp8_gemm_blockscaled_fmt(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C),
                                           int(out), int(a_fmt), int(b_fmt), M, N, K,
                                           _stream(stream)), "fp8_gemm_blockscaled_fmt")


def fp8_grouped_gemm_fmt(A, B, sfa, sfb, C, out: int, a_fmt: int, b_fmt: int, counts, E: int,
                         N: int, K: int, total_rows: int, offsets_out=None, tile_map_out=None,
                         stream=None):
    _check(load().fp8_grouped_gemm_fmt(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C), int(out),
                                       int(a_fmt), int(b_fmt), _ptr(counts), E, N, K, total_rows,
                                       _ptr(offsets_out), _ptr(tile_map_out), _stream(stream)),
           "fp8_grouped_gemm_fmt")


def fp8_gemm_ex(A, B, scale_a, scale_b, C, out: int, a_fmt: int, b_fmt: int, bias, act: int,
                M: int, N: int, K: int, stream=None):
    _check(load().fp8_gemm_ex(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), _ptr(C), int(out),
                              int(a_fmt), int(b_fmt), _ptr(bias), int(act), M, N, K,
                              _stream(stream)), "fp8_gemm_ex")


def fp8_gemm_blockscaled_ex(A, B, sfa, sfb, C, out: int, a_fmt: int, b_fmt: int, bias, act: int,
                            M: int, N: int, K: int, stream=None):
    _check(load().fp8_gemm_blockscaled_ex(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C),
                                          int(out), int(a_fmt), int(b_fmt), _ptr(bias), int(act),
                                          M, N, K, _stream(stream)), "fp8_gemm_blockscaled_ex")


def fp8_grouped_gemm_ex(A, B, sfa, sfb, C, out: int, a_fmt: int, b_fmt: int, bias, act: int,
                        counts, E: int, N: int, K: int, total_rows: int, offsets_out=None,
                        tile_map_out=None, stream=None):
    _check(load().fp8_grouped_gemm_ex(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C), int(out),
                                      int(a_fmt), int(b_fmt), _ptr(bias), int(act), _ptr(counts),
                                      E, N, K, total_rows, _ptr(offsets_out), _ptr(tile_map_out),
                                      _stream(stream)), "fp8_grouped_gemm_ex")


def fp8_grouped_gemm_scatter(A, B, sfa, sfb, C, out: int, a_fmt: int, b_fmt: int, bias,
                             act: int, counts, E: int, N: int, K: int, total_rows: int, c_row_of,
                             c_rows: int, offsets_out=None, tile_map_out=None, stream=None):
    _check(load().fp8_grouped_gemm_scatter(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C),
                                           int(out), int(a_fmt), int(b_fmt), _ptr(bias), int(act),
                                           _ptr(counts), E, N, K, total_rows, _ptr(c_row_of),
                                           c_rows, _ptr(offsets_out), _ptr(tile_map_out),
                                           _stream(stream)), "fp8_grouped_gemm_scatter")


def fp8_grouped_gemm_quant(X, x_dtype: int, x_rows: int, rows, B, sfb, C, out: int, b_fmt: int,
                           bias, act: int, counts, E: int, N: int, K: int, total_rows: int,
                           c_row_of=None, c_rows: int = 0, qa_out=None, sfa_out=None,
                           offsets_out=None, tile_map_out=None, flags: int = 0, stream=None):
    """Grouped GEMM from fp32 / bf16 activations: gather, 1x32 E4M3 quantisation
    (inside the GEMM kernel with flags FP8G_QUANT_FUSED when the plan runs
    single-CTA tiles) and the grouped GEMM with bias / activation and row
    scatter."""
    _check(load().fp8_grouped_gemm_quant(_ptr(X), int(x_dtype), x_rows, _ptr(rows), _ptr(B),
                                         _ptr(sfb), _ptr(C), int(out), int(b_fmt), _ptr(bias),
                                         int(act), _ptr(counts), int(E), N, K, total_rows,
                                         _ptr(c_row_of), c_rows, _ptr(qa_out), _ptr(sfa_out),
                                         _ptr(offsets_out), _ptr(tile_map_out), int(flags),
                                         _stream(stream)), "fp8_grouped_gemm_quant")


def fp8_gemm_blockscaled_promote(A, B, sfa, sfb, C, out: int, a_fmt: int, b_fmt: int, bias,
                                 act: int, M: int, N: int, K: int, stream=None):
    _check(load().fp8_gemm_blockscaled_promote(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C),
                                               int(out), int(a_fmt), int(b_fmt), _ptr(bias),
                                               int(act), M, N, K, _stream(stream)),
           "fp8_gemm_blockscaled_promote")


def fp8g_quantize_nvfp4(x, in_dtype: int, rows: int, cols: int, q, sf, g, stream=None):
    _check(load().fp8g_quantize_nvfp4(_ptr(x), int(in_dtype), rows, cols, _ptr(q), _ptr(sf),
                                      _ptr(g), _stream(stream)), "fp8g_quantize_nvfp4")


def fp8_gemm_nvfp4(A, B, sfa, sfb, ga, gb, C, out: int, bias, act: int, M: int, N: int, K: int,
                   stream=None):
    _check(load().fp8_gemm_nvfp4(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(ga), _ptr(gb),
                                 _ptr(C), int(out), _ptr(bias), int(act), M, N, K,
                                 _stream(stream)), "fp8_gemm_nvfp4")


def fp8_grouped_gemm_nvfp4(A, B, sfa, sfb, ga, gb, C, out: int, bias, act: int, counts, E: int,
                           N: int, K: int, total_rows: int, offsets_out=None, tile_map_out=None,
                           stream=None):
    _check(load().fp8_grouped_gemm_nvfp4(_ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(ga),
                                         _ptr(gb), _ptr(C), int(out), _ptr(bias), int(act),
                                         _ptr(counts), E, N, K, total_rows, _ptr(offsets_out),
                                         _ptr(tile_map_out), _stream(stream)),
           "fp8_grouped_gemm_nvfp4")


def quantize_nvfp4(x, stream=None):
    """fp32 or bf16 CUDA tensor [rows, cols] -> (codes uint8 [rows, cols/2],
    E4M3 block-scale codes uint8 [rows, cols/16], tensor scale fp32 [1])."""
    import torch
    assert x.is_cuda and x.dim() == 2 and x.dtype in (torch.float32, torch.bfloat16)
    x = x.contiguous()
    rows, cols = x.shape
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    sf = torch.empty((rows, cols // 16), dtype=torch.uint8, device=x.device)
    g = torch.empty((1,), dtype=torch.float32, device=x.device)
    dt = FP8G_IN_BF16 if x.dtype == torch.bfloat16 else FP8G_IN_F32
    fp8g_quantize_nvfp4(x, dt, rows, cols, q, sf, g, stream)
    return q, sf, g


def fp8g_quantize_rows(x, in_dtype: int, x_rows: int, cols: int, rows, n_rows: int, block: int,
                       fmt: int, q, scales, stream=None):
    _check(load().fp8g_quantize_rows(_ptr(x), int(in_dtype), x_rows, cols, _ptr(rows), n_rows,
                                     int(block), int(fmt), _ptr(q), _ptr(scales),
                                     _stream(stream)), "fp8g_quantize_rows")


def fp8g_kernel_timing_begin(n: int):
    _check(load().fp8g_kernel_timing_begin(int(n)), "fp8g_kernel_timing_begin")


def fp8g_kernel_timing_end(cap: int) -> list:
    """GEMM-kernel durations (ms) of the calls recorded since begin."""
    ms = (ctypes.c_float * max(int(cap), 1))()
    n = ctypes.c_int32(0)
    _check(load().fp8g_kernel_timing_end(ms, int(cap), ctypes.byref(n)), "fp8g_kernel_timing_end")
    return [float(ms[i]) for i in range(n.value)]


def fp8g_wait_selftest(timeout_us: int, stream=None):
    _check(load().fp8g_wait_selftest(int(timeout_us), _stream(stream)), "fp8g_wait_selftest")


def fp8_gemm_status(stream=None):
    """Returns (status, detail) and clears the device status word."""
    detail = ctypes.c_int32(0)
    st = load().fp8_gemm_status(_stream(stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def fp8g_set_wait_timeout_ms(ms: int):
    load().fp8g_set_wait_timeout_ms(int(ms))


def fp8g_shutdown():
    load().fp8g_shutdown()


def fp8g_version() -> int:
    return int(load().fp8g_version())


# ---------------------------------------------------------------- conveniences
# Allocation helpers over torch (device memory is plumbing); the work is the
# ABI call above.

def packed_cols(cols: int, fmt: int) -> int:
    """Bytes of a row of `cols` codes in format fmt."""
    if fmt == FP8G_E2M1:
        return cols // 2
    if fmt in (FP8G_E2M3, FP8G_E3M2):
        return cols * 3 // 4
    return cols


def quantize(x, block: int = 32, stream=None, fmt: int = FP8G_E4M3):
    """fp32 CUDA tensor [rows, cols] -> (uint8 codes, fp32 scales) in format fmt
    (E2M1: two codes per byte, codes [rows, cols/2]; FP6: four codes per three
    bytes, codes [rows, 3 cols/4])."""
    import torch
    assert x.is_cuda and x.dtype == torch.float32 and x.dim() == 2
    x = x.contiguous()
    rows, cols = x.shape
    qcols = packed_cols(cols, fmt)
    q = torch.empty((rows, qcols), dtype=torch.uint8, device=x.device)
    if block != 0:
        s = torch.empty((rows, cols // 32), dtype=torch.float32, device=x.device)
    else:
        s = torch.empty((1,), dtype=torch.float32, device=x.device)
    fp8g_quantize(x, rows, cols, block, fmt, q, s, stream)
    return q, s


def gemm(A, B, sa, sb, out: str = "bf16", block: bool = True, stream=None):
    """Allocates C and runs fp8_gemm_blockscaled (block) or fp8_gemm (per-tensor)."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = torch.empty((M, N), dtype=dt, device=A.device)
    o = FP8G_OUT_BF16 if out == "bf16" else FP8G_OUT_F32
    if block:
        fp8_gemm_blockscaled(A, B, sa, sb, C, o, M, N, K, stream)
    else:
        fp8_gemm(A, B, sa, sb, C, o, M, N, K, stream)
    return C
