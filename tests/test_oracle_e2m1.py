"""Pins for the oracle's E2M1 (FP4) element format: all 16 codes from the
format definition, ties-to-even midpoints, saturation, the power-of-two block
scale's closed form for the range 6, and a brute-force GEMM in exact
rationals with E2M1 operands (also mixed with E4M3)."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dec(code):
    s = -1 if code & 0x8 else 1
    e, m = (code >> 1) & 3, code & 1
    return s * (Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1))


def test_e2m1_golden_codes(oracle_lib):
    tab = oracle_lib.e2m1_table()
    n = 0
    for line in open(os.path.join(GOLDEN, "e2m1_codes.txt")):
        if line.startswith("#") or not line.strip():
            continue
        c, v = line.split()
        c = int(c, 16)
        if v == "-0":
            assert tab[c] == 0.0 and math.copysign(1.0, tab[c]) < 0
        else:
            assert Fraction(tab[c]) == Fraction(v) == dec(c)
        n += 1
    assert n == 16
    assert np.all(np.diff(tab[:8]) > 0) and tab[7] == 6.0


def test_e2m1_encode(oracle_lib):
    enc = oracle_lib.e2m1_encode
    for c in range(16):
        assert enc(float(dec(c))) == c or (c == 8 and enc(-0.0) == 8)
    for c in range(7):                                   # midpoints -> even code
        mid = (dec(c) + dec(c + 1)) / 2
        assert enc(float(mid)) == (c if c % 2 == 0 else c + 1), c
        assert enc(-float(mid)) == 8 | (c if c % 2 == 0 else c + 1)
    assert enc(7.0) == 7 and enc(1e30) == 7 and enc(float("inf")) == 7 and enc(-100.0) == 0xF
    assert enc(float("nan")) == 7


def test_e2m1_block_scales(oracle_lib):
    F = oracle_lib.E2M1
    for e in range(-100, 100, 11):
        a = 6.0 * 2.0 ** e
        assert oracle_lib.pow2_scale(a, F) == 2.0 ** e
        assert oracle_lib.pow2_scale(float(np.nextafter(np.float32(a), np.float32(np.inf))), F) == 2.0 ** (e + 1)
    x = np.random.default_rng(3).normal(size=(4, 64)).astype(np.float32)
    q, s = oracle_lib.quantize_block32(x, F)
    for r in range(4):
        for b in range(2):
            blk = x[r, 32 * b:32 * b + 32]
            assert s[r, b] == oracle_lib.pow2_scale(float(np.abs(blk).max()), F)
            assert all(q[r, 32 * b + j] == oracle_lib.e2m1_encode(float(blk[j] / s[r, b]))
                       for j in range(32))
    assert (q < 16).all()


@pytest.mark.parametrize("fa,fb", [(2, 2), (0, 2), (2, 1)])
def test_e2m1_gemm_bruteforce(oracle_lib, fa, fb):
    rng = np.random.default_rng(fa * 3 + fb)
    M, N, K = 3, 4, 64
    def codes(fmt, shape):
        if fmt == 2:
            return rng.integers(0, 16, size=shape, dtype=np.uint8)
        c = rng.integers(0, 256, size=shape, dtype=np.uint8)
        c[(c & 0x7C) == 0x7C] = 0x3C
        return c
    A, B = codes(fa, (M, K)), codes(fb, (N, K))
    sfa = (2.0 ** rng.integers(-4, 4, size=(M, 2))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-4, 4, size=(N, 2))).astype(np.float32)
    _, _, exact = oracle_lib.gemm(A, B, sfa, sfb, True, oracle_lib.OUT_F32, want_exact=True,
                                  a_fmt=fa, b_fmt=fb)
    tabs = {0: oracle_lib.e4m3_table(), 1: oracle_lib.e5m2_table()}
    def val(fmt, c):
        return dec(int(c)) if fmt == 2 else Fraction(tabs[fmt][c])
    for i in range(M):
        for j in range(N):
            tot = sum(Fraction(float(sfa[i, kb])) * Fraction(float(sfb[j, kb])) *
                      sum((val(fa, A[i, k]) * val(fb, B[j, k]) for k in range(32 * kb, 32 * kb + 32)),
                          Fraction(0)) for kb in range(2))
            assert abs(Fraction(exact[i, j]) - tot) <= abs(tot) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 80)
