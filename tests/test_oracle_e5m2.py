"""Pins for the oracle's E5M2 format and mixed-format GEMMs: the format
definition (golden codes written from it, exact fractions), an independent
decoder (torch.float8_e5m2), ties-to-even midpoints, saturation, the
power-of-two scale's closed form, and brute-force GEMMs in exact rational
arithmetic for every operand-format pairing."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dec5(code: int):
    """E5M2 value as a Fraction (None for NaN, +-inf as floats), from the definition."""
    s = -1 if code & 0x80 else 1
    e = (code >> 2) & 31
    m = code & 3
    if e == 31:
        return None if m else s * math.inf
    if e == 0:
        return s * Fraction(m, 65536)
    return s * (1 + Fraction(m, 4)) * Fraction(2) ** (e - 15)


def dec4(code: int):
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return None
    if e == 0:
        return s * Fraction(m, 512)
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


DEC = {0: dec4, 1: dec5}


def test_e5m2_golden_codes(oracle_lib):
    tab = oracle_lib.e5m2_table()
    n = 0
    for line in open(os.path.join(GOLDEN, "e5m2_codes.txt")):
        if line.startswith("#") or not line.strip():
            continue
        code_s, val_s = line.split()
        c = int(code_s, 16)
        if val_s == "nan":
            assert math.isnan(tab[c]), hex(c)
        elif val_s in ("inf", "-inf"):
            assert tab[c] == float(val_s), hex(c)
        elif val_s == "-0":
            assert tab[c] == 0.0 and math.copysign(1.0, tab[c]) < 0
        else:
            assert Fraction(tab[c]) == Fraction(val_s), hex(c)
            assert Fraction(tab[c]) == dec5(c)
        n += 1
    assert n >= 25


def test_e5m2_decode_matches_torch_all_codes(oracle_lib):
    tab = oracle_lib.e5m2_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float32).double().numpy()
    nan_o, nan_r = np.isnan(tab), np.isnan(ref)
    assert (nan_o == nan_r).all()
    assert np.array_equal(tab[~nan_o], ref[~nan_r])
    assert set(np.flatnonzero(nan_o).tolist()) == {0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF}


def test_e5m2_decode_structure(oracle_lib):
    tab = oracle_lib.e5m2_table()
    pos = tab[:0x7C]
    assert np.all(np.diff(pos) > 0)
    assert pos.max() == 57344.0 and tab[0x01] == 2.0 ** -16 and tab[0x04] == 2.0 ** -14
    for c in range(0x7C):
        assert tab[c | 0x80] == -tab[c]
    assert np.isinf(tab).sum() == 2


def test_e5m2_encode_roundtrip_ties_saturation(oracle_lib):
    enc = oracle_lib.e5m2_encode
    for c in range(256):
        v = dec5(c)
        if v is None or isinstance(v, float):
            continue
        assert enc(float(v)) == c or (c == 0x80 and enc(-0.0) == 0x80), hex(c)
    for c in range(0x7B):                     # midpoints of consecutive positive codes
        mid = (dec5(c) + dec5(c + 1)) / 2
        assert enc(float(mid)) == (c if c % 2 == 0 else c + 1), hex(c)
    assert enc(1.125) == 0x3C and enc(1.375) == 0x3E
    assert enc(61440.0) == 0x7B               # tie 57344 / (65536): even -> 65536 -> saturate
    assert enc(1e9) == 0x7B and enc(float("inf")) == 0x7B and enc(float("-inf")) == 0xFB
    assert enc(float("nan")) == 0x7F
    assert enc(2.0 ** -17) == 0x00 and enc(3 * 2.0 ** -17) == 0x02
    assert enc(-0.0) == 0x80


def test_e5m2_encode_matches_torch_in_range(oracle_lib):
    g = torch.Generator().manual_seed(12)
    x = torch.cat([torch.randn(4000, generator=g) * s for s in (1e-4, 1.0, 300.0, 2e4)])
    x = x.clamp(-57344.0, 57344.0)
    ref = x.to(torch.float8_e5m2).view(torch.uint8).numpy()
    got = np.array([oracle_lib.e5m2_encode(float(v)) for v in x.numpy()], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e5m2_scales(oracle_lib):
    E5 = oracle_lib.E5M2
    for e in range(-120, 100, 9):
        a = 57344.0 * 2.0 ** e
        assert oracle_lib.pow2_scale(a, E5) == 2.0 ** e
        assert oracle_lib.pow2_scale(float(np.nextafter(np.float32(a), np.float32(np.inf))), E5) == 2.0 ** (e + 1)
    assert oracle_lib.pow2_scale(1.0, E5) == 2.0 ** -15   # 57344 * 2^-16 = 0.875 < 1 <= 1.75
    g = torch.Generator().manual_seed(5)
    x = torch.randn(3, 96, generator=g) * 50
    x[1, 32:64] = 0.0
    x = x.numpy()
    q, s = oracle_lib.quantize_block32(x, E5)
    for r in range(3):
        for b in range(3):
            blk = x[r, 32 * b:32 * b + 32]
            assert s[r, b] == oracle_lib.pow2_scale(float(np.abs(blk).max()), E5)
            for j in range(32):
                assert q[r, 32 * b + j] == oracle_lib.e5m2_encode(float(np.float32(blk[j]) / s[r, b]))
    assert s[1, 1] == 1.0 and not q[1, 32:64].any()
    qt, st = oracle_lib.quantize_tensor(x, E5)
    assert st[0] == np.float32(np.float32(np.abs(x).max()) / np.float32(57344.0))
    ref = (torch.from_numpy(x) / torch.tensor(st[0])).clamp(-57344, 57344).to(torch.float8_e5m2)
    assert np.array_equal(qt, ref.view(torch.uint8).numpy())


def _codes(rng, shape, fmt):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    if fmt == 1:
        c[(c & 0x7C) == 0x7C] = 0x3D          # no inf / NaN codes
    else:
        c[(c & 0x7F) == 0x7F] = 0x3C
    return c


@pytest.mark.parametrize("fa,fb", [(0, 1), (1, 0), (1, 1)])
def test_mixed_format_gemm_bruteforce(oracle_lib, fa, fb):
    rng = np.random.default_rng(10 * fa + fb)
    M, N, K = 3, 4, 64
    A = _codes(rng, (M, K), fa)
    B = _codes(rng, (N, K), fb)
    sfa = (2.0 ** rng.integers(-6, 6, size=(M, K // 32))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-6, 6, size=(N, K // 32))).astype(np.float32)
    C, bound, exact = oracle_lib.gemm(A, B, sfa, sfb, block=True, out_kind=oracle_lib.OUT_F32,
                                      want_exact=True, a_fmt=fa, b_fmt=fb)
    sa, sb = np.float32(0.75), np.float32(3.0e-3)
    Ct, _, _ = oracle_lib.gemm(A, B, np.array([sa]), np.array([sb]), block=False,
                               out_kind=oracle_lib.OUT_F32, a_fmt=fa, b_fmt=fb)
    alpha = Fraction(float(np.float32(sa * sb)))
    for i in range(M):
        for j in range(N):
            tot, acc, absum = Fraction(0), Fraction(0), Fraction(0)
            for kb in range(K // 32):
                part = sum((DEC[fa](int(A[i, k])) * DEC[fb](int(B[j, k]))
                            for k in range(32 * kb, 32 * kb + 32)), Fraction(0))
                tot += Fraction(float(sfa[i, kb])) * Fraction(float(sfb[j, kb])) * part
                acc += part
            # fp64 sums: exact unless the E5M2 products span more than 53 bits
            assert abs(Fraction(exact[i, j]) - tot) <= abs(tot) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 60)
            assert C[i, j] == np.float32(exact[i, j])
            want_t = np.float32(float(alpha * acc))
            assert abs(float(Ct[i, j]) - float(want_t)) <= abs(float(want_t)) * 2.0 ** -23
    # the sampled path agrees with the full one
    pi, pj = np.array([0, 2, 1]), np.array([3, 0, 1])
    Cs, _, _ = oracle_lib.gemm_sample(A, B, sfa, sfb, True, pi, pj, oracle_lib.OUT_F32,
                                      a_fmt=fa, b_fmt=fb)
    assert np.array_equal(Cs, C[pi, pj])
