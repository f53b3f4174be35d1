"""Pins of the oracle's FP6 formats (E2M3: bias 1, 3 mantissa bits, up to
7.5; E3M2: bias 3, 2 mantissa bits, up to 28; both without infinities or
NaNs) against facts fixed without it: the value lists written out by hand
from the format definitions, a brute-force nearest-value search for every
encoding (ties to the even code, saturation, signs, NaN), the power-of-two
block scale by exhaustive search, and GEMMs that reduce to the pinned E4M3
GEMM because every FP6 value is also an E4M3 value."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _lib(oracle_lib):
    yield


# positive values of codes 0 .. 31, listed by hand: E2M3 subnormals k/8
# (k < 8), then binades [1, 2) and [2, 4) in eighths of the binade base, then
# [4, 8) in steps of 0.5; E3M2 subnormals k/16 (k < 4), then binades 2^-2 ..
# 2^4 in quarters of the binade base
E2M3_VALUES = [0, 0.125, 0.25, 0.375, 0.5, 0.625, 0.75, 0.875,
               1, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875,
               2, 2.25, 2.5, 2.75, 3, 3.25, 3.5, 3.75,
               4, 4.5, 5, 5.5, 6, 6.5, 7, 7.5]
E3M2_VALUES = [0, 0.0625, 0.125, 0.1875, 0.25, 0.3125, 0.375, 0.4375,
               0.5, 0.625, 0.75, 0.875, 1, 1.25, 1.5, 1.75,
               2, 2.5, 3, 3.5, 4, 5, 6, 7,
               8, 10, 12, 14, 16, 20, 24, 28]
FORMATS = [(oracle.E2M3, E2M3_VALUES, 7.5), (oracle.E3M2, E3M2_VALUES, 28.0)]


@pytest.mark.parametrize("fmt,vals,fmax", FORMATS)
def test_value_tables(fmt, vals, fmax):
    t = oracle.fp6_table(fmt)
    assert t[:32].tolist() == vals
    assert t[32:64].tolist() == [-v for v in vals]          # sign bit 5
    assert np.array_equal(np.signbit(t[32:64]), np.ones(32, bool))
    for hi in (0x40, 0x80, 0xC0):                           # high two bits ignored
        assert np.array_equal(t[hi:hi + 64], t[:64])
    assert max(vals) == fmax


def _nearest_code(y: float, vals) -> int:
    """Brute force: the code whose value is nearest |y| (ties: the even
    code), saturating, with y's sign."""
    a = min(abs(y), vals[-1]) if np.isfinite(y) else vals[-1]
    d = np.abs(np.asarray(vals) - a)
    best = np.flatnonzero(d == d.min())
    c = int(best[0]) if best.size == 1 else int(best[best % 2 == 0][0])
    return c | (0x20 if np.signbit(y) else 0)


@pytest.mark.parametrize("fmt,vals,fmax", FORMATS)
def test_encode_brute_force(fmt, vals, fmax):
    rng = np.random.default_rng(fmt)
    ys = np.concatenate([
        rng.standard_normal(4000) * fmax / 3,
        rng.uniform(-fmax * 1.5, fmax * 1.5, 2000),
        rng.uniform(-0.3, 0.3, 2000),                       # subnormals and zero
        np.array(vals) + 1e-4, np.array(vals) - 1e-4,
    ]).astype(np.float32)
    for y in ys:
        assert oracle.fp6_encode(float(y), fmt) == _nearest_code(float(y), vals), y


@pytest.mark.parametrize("fmt,vals,fmax", FORMATS)
def test_encode_ties_specials(fmt, vals, fmax):
    """Every midpoint between neighbours goes to the even code; beyond the
    largest value and +-inf saturate; -0 keeps its sign; NaN takes the
    largest positive code (0x1F)."""
    for c in range(31):
        mid = (vals[c] + vals[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert oracle.fp6_encode(mid, fmt) == want, (c, mid)
        assert oracle.fp6_encode(-mid, fmt) == want | 0x20
    assert oracle.fp6_encode(fmax * 1.02, fmt) == 0x1F
    assert oracle.fp6_encode(float("inf"), fmt) == 0x1F
    assert oracle.fp6_encode(float("-inf"), fmt) == 0x3F
    assert oracle.fp6_encode(-0.0, fmt) == 0x20
    assert oracle.fp6_encode(float("nan"), fmt) == 0x1F


@pytest.mark.parametrize("fmt,vals,fmax", FORMATS)
def test_block_scale_exhaustive(fmt, vals, fmax):
    """The 1x32 scale is the smallest power of two s with fmax s >= amax."""
    rng = np.random.default_rng(10 + fmt)
    for amax in np.concatenate([np.exp(rng.uniform(-60, 60, 300)), [fmax, fmax * 2, 1.0, 3e-30]]):
        amax = float(np.float32(amax))
        s = oracle.pow2_scale(amax, fmt)
        e = int(np.log2(s))
        assert s == 2.0 ** e
        assert fmax * s >= amax and fmax * s / 2 < amax, (amax, s)


@pytest.mark.parametrize("fmt,vals,fmax", FORMATS)
def test_quantize_block32_nearest(fmt, vals, fmax):
    rng = np.random.default_rng(20 + fmt)
    x = (rng.standard_normal((16, 128)) * np.exp(rng.standard_normal((16, 1)) * 3)).astype(np.float32)
    q, s = oracle.quantize_block32(x, fmt)
    assert q.max() < 64
    for r in range(16):
        for k in range(128):
            y = np.float32(x[r, k]) / np.float32(s[r, k // 32])
            assert q[r, k] == _nearest_code(float(y), vals)
    qt, st = oracle.quantize_tensor(x, fmt)
    assert st[0] == np.float32(np.abs(x).max()) / np.float32(fmax)


def _as_e4m3(codes, fmt):
    """The same values as E4M3 codes (exact: every FP6 value is an E4M3
    value, checked here)."""
    vals = oracle.fp6_table(fmt)[codes]
    lut = np.array([oracle.e4m3_encode(v) for v in oracle.fp6_table(fmt)[:64]], np.uint8)
    out = lut[codes & 63]
    assert np.array_equal(oracle.e4m3_table()[out], vals)
    return out


@pytest.mark.parametrize("a_fmt,b_fmt", [(3, 3), (4, 4), (3, 4), (4, 0), (0, 3)])
@pytest.mark.parametrize("block", [True, False])
def test_gemm_reduces_to_e4m3(a_fmt, b_fmt, block):
    """FP6 (or mixed) operands give bit for bit the E4M3 GEMM of the same
    values, for block and per-tensor scales."""
    rng = np.random.default_rng(a_fmt * 10 + b_fmt)
    M, N, K = 20, 28, 96
    A = rng.integers(0, 64 if a_fmt else 255, (M, K)).astype(np.uint8)
    B = rng.integers(0, 64 if b_fmt else 255, (N, K)).astype(np.uint8)
    if a_fmt == 0:
        A[(A & 0x7F) == 0x7F] = 0            # no E4M3 NaN
    if b_fmt == 0:
        B[(B & 0x7F) == 0x7F] = 0
    if block:
        sa = 2.0 ** rng.integers(-3, 4, (M, K // 32)).astype(np.float32)
        sb = 2.0 ** rng.integers(-3, 4, (N, K // 32)).astype(np.float32)
    else:
        sa = np.array([0.37], np.float32)
        sb = np.array([1.9], np.float32)
    A8 = _as_e4m3(A, a_fmt) if a_fmt else A
    B8 = _as_e4m3(B, b_fmt) if b_fmt else B
    C, _, e = oracle.gemm(A, B, sa, sb, block, oracle.OUT_F32, want_exact=True, a_fmt=a_fmt,
                          b_fmt=b_fmt)
    C8, _, e8 = oracle.gemm(A8, B8, sa, sb, block, oracle.OUT_F32, want_exact=True)
    assert np.array_equal(e, e8) and np.array_equal(C, C8)
