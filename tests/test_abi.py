"""The C ABI library (no GPU needed): it builds, loads, exports every function
include/fp8gemm.h declares, and its host-side argument checks return the
documented status codes before touching a device."""
import ctypes
import os
import re

import pytest

import fp8_block_scaled_06_gb300 as fp8g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(fp8\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_abi():
    names = _declared_functions()
    assert {"fp8_gemm", "fp8_gemm_blockscaled", "fp8_grouped_gemm",
            "fp8g_quantize_e4m3", "fp8_gemm_status"} <= names
    assert names == set(fp8g.EXPORTS)


def test_library_exports_every_declared_symbol(fp8g):
    lib = ctypes.CDLL(fp8g.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(fp8g):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fp8g.LIB_PATH], capture_output=True,
                         text=True).stdout
    ours = {ln.split()[-1] for ln in out.splitlines() if " T " in ln and "fp8" in ln}
    assert ours == _declared_functions()


def test_status_strings(fp8g):
    assert fp8g.fp8g_status_string(0) == "ok"
    for code in range(1, 8):
        assert fp8g.fp8g_status_string(code) not in ("ok", "unknown status")
    assert fp8g.fp8g_version() >= 100


def _err(fn, *args):
    with pytest.raises(fp8g.Fp8gError) as e:
        fn(*args)
    return e.value.status


def test_host_argument_checks(fp8g):
    P = 1 << 20                                   # a 16-byte aligned fake address; never dereferenced
    assert _err(fp8g.fp8_gemm, 0, P, P, P, P, 0, 8, 8, 16, 0) == fp8g.FP8G_ERR_INVALID_ARG
    assert _err(fp8g.fp8_gemm, P, P, P, P, P, 3, 8, 8, 16, 0) == fp8g.FP8G_ERR_INVALID_ARG
    assert _err(fp8g.fp8_gemm, P, P, P, P, P, 0, 0, 8, 16, 0) == fp8g.FP8G_ERR_INVALID_ARG
    assert _err(fp8g.fp8_gemm, P + 8, P, P, P, P, 0, 8, 8, 16, 0) == fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8_gemm, P, P, P, P, P, 0, 8, 8, 24, 0) == fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8_gemm, P, P, P, P, P, 0, 8, 4, 16, 0) == fp8g.FP8G_ERR_ALIGNMENT  # N*2 % 16
    assert _err(fp8g.fp8_gemm, P, P, P, P, P, 1, 8, 2, 16, 0) == fp8g.FP8G_ERR_ALIGNMENT  # N*4 % 16
    assert _err(fp8g.fp8_gemm_blockscaled, P, P, P, P, P, 0, 8, 8, 48, 0) == \
        fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(fp8g.fp8_gemm_blockscaled, P, P, P + 4, P, P, 0, 8, 8, 64, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8_grouped_gemm, P, P, P, P, P, 0, P, 65, 8, 64, 8, None, None, 0) == \
        fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(fp8g.fp8_grouped_gemm, P, P, P, P, P, 0, 0, 2, 8, 64, 8, None, None, 0) == \
        fp8g.FP8G_ERR_INVALID_ARG
    assert _err(fp8g.fp8_grouped_gemm, P, P, P, P, P, 0, P, 2, 8, 64, 8, None, P + 4, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8g_quantize_e4m3, P, 4, 40, 32, P, P, 0) == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(fp8g.fp8g_quantize_e4m3, P, 4, 64, 16, P, P, 0) == fp8g.FP8G_ERR_INVALID_ARG


def test_grouped_plan_host_only(fp8g):
    p = fp8g.fp8g_grouped_plan(14336, 4096, 32768, 8)
    assert p["BM"] in (128, 256) and p["G"] == 16 and p["BN"] in (128, 256)
    npn = -(-14336 // p["BN"])
    assert p["max_tiles"] == (32768 // p["BM"] + 8) * npn
    small = fp8g.fp8g_grouped_plan(256, 256, 300, 3)       # far less than a wave of tiles
    assert small["BM"] == 128


def test_host_checks_of_the_wider_entry_points(fp8g):
    """Formats, epilogue, literal scales, gather/scatter and the self-test all
    reject bad arguments on the host, before any device work (no GPU here)."""
    P = 1 << 20
    E = fp8g.FP8G_ERR_INVALID_ARG
    assert _err(fp8g.fp8_gemm_fmt, P, P, P, P, P, 0, 5, 0, 8, 8, 16, 0) == E      # bad A format
    # packed E2M1 operands: K % 128, the operand 32-byte aligned
    assert _err(fp8g.fp8_gemm_fmt, P, P, P, P, P, 0, 2, 0, 8, 8, 64, 0) == \
        fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(fp8g.fp8_gemm_blockscaled_fmt, P, P + 16, P, P, P, 0, 0, 2, 8, 8, 128, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8_gemm_blockscaled_promote, P + 16, P, P, P, P, 0, 2, 0, None, 0, 8, 8,
                128, 0) == fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8_gemm_blockscaled_fmt, P, P, P, P, P, 0, 0, 5, 8, 8, 64, 0) == E
    assert _err(fp8g.fp8_gemm_blockscaled_fmt, P, P, P, P, P, 0, 0, -1, 8, 8, 64, 0) == E
    # packed FP6 operands (E2M3 3, E3M2 4): the rules of E2M1
    assert _err(fp8g.fp8_gemm_fmt, P, P, P, P, P, 0, 3, 0, 8, 8, 64, 0) == \
        fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(fp8g.fp8_gemm_blockscaled_fmt, P, P + 16, P, P, P, 0, 0, 4, 8, 8, 128, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8_grouped_gemm_ex, P + 16, P, P, P, P, 0, 4, 3, None, 0, P, 2, 8, 128, 8,
                None, None, 0) == fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8_gemm_ex, P, P, P, P, P, 0, 0, 0, None, 3, 8, 8, 16, 0) == E  # bad act
    assert _err(fp8g.fp8_gemm_blockscaled_ex, P, P, P, P, P, 0, 0, 0, P + 2, 1, 8, 8, 64, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT                                                  # bias alignment
    assert _err(fp8g.fp8_grouped_gemm_ex, P, P, P, P, P, 0, 1, 1, None, 9, P, 2, 8, 64, 8, None,
                None, 0) == E
    assert _err(fp8g.fp8_gemm_blockscaled_promote, P, P, P, P, P, 0, 0, 0, None, 0, 8, 8, 96,
                0) == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE                            # K % 128
    assert _err(fp8g.fp8_gemm_blockscaled_promote, P, P, P, P, P, 0, 0, 5, None, 0, 8, 8, 128,
                0) == E
    assert _err(fp8g.fp8_grouped_gemm_scatter, P, P, P, P, P, 0, 0, 0, None, 0, P, 2, 8, 64, 8,
                P + 2, 16, None, None, 0) == E                                   # misaligned map
    assert _err(fp8g.fp8_grouped_gemm_scatter, P, P, P, P, P, 0, 0, 0, None, 0, P, 2, 8, 64, 8,
                P, 0, None, None, 0) == E                                        # no rows of C
    # quantiser: source type, format, block mode, gather without rows > source rows
    assert _err(fp8g.fp8g_quantize_rows, P, 2, 4, 64, None, 4, 32, 0, P, P, 0) == E
    assert _err(fp8g.fp8g_quantize_rows, P, 0, 4, 64, None, 4, 32, 5, P, P, 0) == E
    assert _err(fp8g.fp8g_quantize_rows, P, 0, 4, 64, None, 4, 17, 0, P, P, 0) == E
    assert _err(fp8g.fp8g_quantize_rows, P, 0, 4, 64, None, 5, 32, 0, P, P, 0) == E
    assert _err(fp8g.fp8g_quantize_rows, P, 1, 4, 40, None, 4, fp8g.FP8G_BLOCK32_LITERAL, 0, P,
                P, 0) == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(fp8g.fp8g_quantize_rows, P, 0, 4, 64, P + 2, 4, 32, 0, P, P, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8g_wait_selftest, 0, 0) == E
    # NVFP4: K % 256, 32-byte aligned operands, the tensor scales given, cols % 16
    assert _err(fp8g.fp8_gemm_nvfp4, P, P, P, P, P, P, P, 0, None, 0, 8, 8, 128, 0) == \
        fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(fp8g.fp8_gemm_nvfp4, P + 16, P, P, P, P, P, P, 0, None, 0, 8, 8, 256, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(fp8g.fp8_gemm_nvfp4, P, P, P, P, None, P, P, 0, None, 0, 8, 8, 256, 0) == E
    assert _err(fp8g.fp8_gemm_nvfp4, P, P, P + 4, P, P, P, P, 0, None, 0, 8, 8, 256, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    # grouped NVFP4: as the dense one, plus the experts, the counts and the tile map
    gn = fp8g.fp8_grouped_gemm_nvfp4
    assert _err(gn, P, P, P, P, P, P, P, 0, None, 0, P, 2, 8, 128, 8, None, None, 0) == \
        fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(gn, P, P, P, P, P, P, P, 0, None, 0, None, 2, 8, 256, 8, None, None, 0) == E
    assert _err(gn, P, P, P, P, P, P, P, 0, None, 0, P, 0, 8, 256, 8, None, None, 0) == E
    assert _err(gn, P, P, P, P, P, P, P, 0, None, 0, P, fp8g.FP8G_MAX_EXPERTS + 1, 8, 256, 8,
                None, None, 0) == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert _err(gn, P, P, P, P, P, P, P, 0, None, 0, P, 2, 8, 256, -1, None, None, 0) == E
    assert _err(gn, P, P + 16, P, P, P, P, P, 0, None, 0, P, 2, 8, 256, 8, None, None, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(gn, P, P, P, P, P, P + 2, P, 0, None, 0, P, 2, 8, 256, 8, None, None, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(gn, P, P, P, P, P, P, P, 0, None, 0, P, 2, 8, 256, 8, None, P + 4, 0) == \
        fp8g.FP8G_ERR_ALIGNMENT
    assert _err(gn, P, P, P, P, P, P, P, 0, None, 3, P, 2, 8, 256, 8, None, None, 0) == E
    assert _err(fp8g.fp8g_quantize_nvfp4, P, 0, 4, 40, P, P, P, 0) == \
        fp8g.FP8G_ERR_UNSUPPORTED_SHAPE


def test_noalloc_checks_match_blockscaled(fp8g):
    """The allocation-free block-scaled GEMM applies fp8_gemm_blockscaled's
    argument checks in the same order: the same bad call gets the same status
    from both (host only; nothing here reaches a device)."""
    P = 1 << 20
    cases = [
        (0, P, P, P, P, 0, 8, 8, 64),          # null A
        (P, P, None, P, P, 0, 8, 8, 64),       # null sfa
        (P, P, P, P, P, 2, 8, 8, 64),          # bad output kind
        (P, P, P, P, P, 0, 0, 8, 64),          # M = 0
        (P, P, P, P, P, 0, 8, 8, 1 << 31),     # K too large
        (P + 8, P, P, P, P, 0, 8, 8, 64),      # A misaligned
        (P, P, P, P, P, 0, 8, 8, 40),          # K % 16
        (P, P, P, P, P, 0, 8, 4, 64),          # N * 2 % 16
        (P, P, P, P, P, 0, 8, 8, 48),          # K % 32
        (P, P, P + 4, P, P, 0, 8, 8, 64),      # sfa misaligned
        (P, P, P + 4, P, P, 0, 8, 8, 48),      # sfa misaligned and K % 32: shape first
        (P, P, None, P, P, 0, 8, 8, 48),       # null sfa and K % 32: null first
        (P, P, None, P, P, 0, 0, 8, 64),       # null sfa and M = 0: shape first
    ]
    for args in cases:
        a = _err(fp8g.fp8_gemm_blockscaled, *args, 0)
        b = _err(fp8g.fp8_gemm_blockscaled_noalloc, *args, 0)
        assert a == b, (args, a, b)


def test_fused_quant_host_checks(fp8g):
    """fp8_grouped_gemm_quant: source type, copies both-or-neither, gather
    without an index past the source, alignment of X and the copies, and the
    grouped GEMM's own rules, all before any device work."""
    P = 1 << 20
    f = fp8g.fp8_grouped_gemm_quant
    E = fp8g.FP8G_ERR_INVALID_ARG
    A = fp8g.FP8G_ERR_ALIGNMENT
    ok = dict(X=P, x_dtype=1, x_rows=8, rows=P, B=P, sfb=P, C=P, out=0, b_fmt=0, bias=None,
              act=0, counts=P, E=2, N=8, K=64, total_rows=8)

    def call(**kw):
        a = dict(ok, **kw)
        return _err(f, a["X"], a["x_dtype"], a["x_rows"], a["rows"], a["B"], a["sfb"], a["C"],
                    a["out"], a["b_fmt"], a["bias"], a["act"], a["counts"], a["E"], a["N"],
                    a["K"], a["total_rows"], None, 0, a.get("qa"), a.get("sa"), None, None,
                    a.get("flags", 0), 0)
    assert call(x_dtype=2) == E
    assert call(qa=P) == E                                  # codes without scales
    assert call(rows=None, x_rows=4) == E                   # 8 routed rows from 4 sources
    assert call(X=P + 8) == A
    assert call(rows=P + 2) == A
    assert call(qa=P + 8, sa=P) == A
    assert call(K=48) == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert call(E=0) == E
    assert call(counts=None) == E
    assert call(b_fmt=7) == E
    assert call(flags=2) == E
    assert _err(f, P, 1, 8, P, P, P, P, 0, 0, None, 5, P, 2, 8, 64, 8, None, 0, None, None,
                None, None, 0, 0) == E                                   # activation
    assert _err(f, P, 1, 8, P, P + 16, P, P, 0, 2, None, 0, P, 2, 8, 128, 8, None, 0, None, None,
                None, None, 0, 0) == A                                   # packed B alignment
    assert _err(f, P, 1, 8, P, P, P, P, 0, 2, None, 0, P, 2, 8, 64, 8, None, 0, None, None,
                None, None, 0, 0) == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE     # packed B, K % 128
