"""Pins of the CPU oracle against facts fixed independently of it.

Each test names what pins it: the E4M3 format definition (golden codes), a
library routine used as a check only (torch's float8_e4m3fn / bfloat16 casts,
numpy cumsum), exact rational arithmetic (fractions.Fraction) on tiny inputs,
closed forms (identity / permutation / exhaustive-code GEMMs, scaling and
transposition laws) and hand-enumerated raster orders.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(s: str):
    if s == "nan":
        return None
    if s == "-0":
        return Fraction(0)
    return Fraction(s)


def dec_exact(code: int):
    """E4M3 value as a Fraction, written from the format definition (test-side)."""
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return None
    if e == 0:
        return s * Fraction(m, 512)
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


# ------------------------------------------------------------------ decode
def test_decode_golden_codes(oracle_lib):
    tab = oracle_lib.e4m3_table()
    n = 0
    for line in open(os.path.join(GOLDEN, "e4m3_codes.txt")):
        if line.startswith("#") or not line.strip():
            continue
        code_s, val_s = line.split()
        code = int(code_s, 16)
        want = _frac(val_s)
        if want is None:
            assert math.isnan(tab[code])
        else:
            assert Fraction(tab[code]) == want, hex(code)
            if val_s == "-0":
                assert math.copysign(1.0, tab[code]) < 0
        n += 1
    assert n >= 25


def test_decode_matches_torch_all_codes(oracle_lib):
    tab = oracle_lib.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).double()
    ref = ref.numpy()
    nan_o, nan_r = np.isnan(tab), np.isnan(ref)
    assert (nan_o == nan_r).all()
    assert np.array_equal(tab[~nan_o], ref[~nan_r])
    assert set(np.flatnonzero(nan_o).tolist()) == {0x7F, 0xFF}


def test_decode_structure(oracle_lib):
    tab = oracle_lib.e4m3_table()
    pos = tab[:0x7F]
    assert np.all(np.diff(pos) > 0)                  # monotone over finite positive codes
    assert pos.max() == 448.0 and tab[0x7E] == 448.0
    assert tab[0x01] == 2.0 ** -9 and tab[0x08] == 2.0 ** -6
    for c in range(0x7F):
        assert tab[c | 0x80] == -tab[c] or (c == 0 and tab[0x80] == 0.0)
    assert not np.isinf(tab).any()


# ------------------------------------------------------------------ encode
def test_encode_roundtrip_all_finite_codes(oracle_lib):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = oracle_lib.e4m3_decode(c)
        assert oracle_lib.e4m3_encode(v) == c


def test_encode_ties_to_even_and_saturation(oracle_lib):
    enc = oracle_lib.e4m3_encode
    assert enc(1.0625) == 0x38        # tie 1 / 1.125 -> even mantissa (1.0)
    assert enc(1.1875) == 0x3A        # tie 1.125 / 1.25 -> 1.25
    assert enc(464.0) == 0x7E         # tie 448 / (480) -> 448
    assert enc(480.0) == 0x7E and enc(1e4) == 0x7E and enc(float("inf")) == 0x7E
    assert enc(-1e4) == 0xFE and enc(float("-inf")) == 0xFE
    assert enc(float("nan")) == 0x7F
    assert enc(-0.0) == 0x80 and enc(0.0) == 0x00
    assert enc(2.0 ** -10) == 0x00    # tie 0 / 2^-9 -> 0 (even)
    assert enc(3 * 2.0 ** -10) == 0x02  # tie 2^-9 / 2^-8 -> 2*2^-9 (even)
    # every midpoint between consecutive positive finite codes rounds to the even code
    for c in range(0x7E):
        a, b = dec_exact(c), dec_exact(c + 1)
        mid = (a + b) / 2
        got = enc(float(mid))
        assert got == (c if c % 2 == 0 else c + 1), hex(c)


def test_encode_matches_torch_in_range(oracle_lib):
    g = torch.Generator().manual_seed(11)
    x = torch.cat([torch.randn(4000, generator=g) * s for s in (1e-3, 1.0, 30.0, 200.0)])
    x = x.clamp(-463.0, 463.0)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_lib.e4m3_encode(float(v)) for v in x.numpy()], dtype=np.uint8)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------- bf16
def _bf16_exact(fr: Fraction) -> Fraction:
    """RNE of an exact rational to 8 significant bits (normal range only)."""
    if fr == 0:
        return Fraction(0)
    s = -1 if fr < 0 else 1
    a = abs(fr)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 7)
    n = a / q
    fl = math.floor(n)
    rem = n - fl
    r = fl + 1 if rem > Fraction(1, 2) else fl if rem < Fraction(1, 2) else (fl if fl % 2 == 0 else fl + 1)
    return s * r * q


def test_bf16_round_matches_torch_on_floats(oracle_lib):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 10)
    ref = x.to(torch.bfloat16).to(torch.float32).numpy()
    got = np.array([oracle_lib.bf16_round(float(v)) for v in x.numpy()], dtype=np.float32)
    assert np.array_equal(got, ref)


def test_bf16_round_direct_from_fp64(oracle_lib):
    # a value just above a bf16 tie whose fp32 rounding lands on the tie:
    # direct rounding goes up, rounding through fp32 first would go to even (down)
    tie = 1.0 + 2.0 ** -8
    x = tie + 2.0 ** -40
    assert np.float32(x) == np.float32(tie)
    assert oracle_lib.bf16_round(x) == 1.0 + 2.0 ** -7
    assert oracle_lib.bf16_round(tie) == 1.0
    for v in (3.3, -7.77e-3, 1e30, 123456.789, 2.0 ** -120 * 1.3):
        assert Fraction(oracle_lib.bf16_round(v)) == _bf16_exact(Fraction(v))
    assert oracle_lib.bf16_ulp(1.0) == 2.0 ** -7
    assert oracle_lib.bf16_ulp(3.0) == 2.0 ** -6
    assert oracle_lib.bf16_ulp(0.0) == 2.0 ** -133


# -------------------------------------------------------------- quantisers
def test_quantize_tensor_scale_and_codes(oracle_lib):
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(64, 96, generator=g) * 3).numpy()
    q, s = oracle_lib.quantize_tensor(x)
    amax = np.float32(np.abs(x).max())
    assert s[0] == np.float32(amax / np.float32(448.0))
    y = (torch.from_numpy(x) / torch.tensor(s[0])).clamp(-463, 463)
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    # the largest element maps to +-448 or just below it
    i = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert abs(oracle_lib.e4m3_decode(q[i])) >= 416.0
    zq, zs = oracle_lib.quantize_tensor(np.zeros((4, 8), np.float32))
    assert zs[0] == 1.0 and not zq.any()


def test_pow2_scale_closed_form(oracle_lib):
    for e in range(-120, 110, 7):
        a = 448.0 * 2.0 ** e
        assert oracle_lib.pow2_scale(a) == 2.0 ** e
        assert oracle_lib.pow2_scale(float(np.nextafter(np.float32(a), np.float32(np.inf)))) == 2.0 ** (e + 1)
    assert oracle_lib.pow2_scale(0.0) == 1.0
    assert oracle_lib.pow2_scale(1.0) == 2.0 ** -8    # 448 * 2^-8 = 1.75 >= 1 > 0.875
    rng = np.random.default_rng(1)
    for a in np.exp(rng.uniform(-60, 60, 500)).astype(np.float32):
        s = oracle_lib.pow2_scale(float(a))
        m, ex = math.frexp(s)
        assert m == 0.5                               # power of two
        assert 448.0 * s >= a and 448.0 * s / 2 < a


def test_quantize_block32_definition(oracle_lib):
    g = torch.Generator().manual_seed(4)
    x = torch.randn(5, 128, generator=g)
    x[1, 32:64] = 0.0                                 # all-zero block -> scale 1, codes 0
    x[2, :32] *= 1e3
    x = x.numpy()
    q, s = oracle_lib.quantize_block32(x)
    assert s.shape == (5, 4)
    for r in range(5):
        for b in range(4):
            blk = x[r, 32 * b:32 * b + 32]
            assert s[r, b] == oracle_lib.pow2_scale(float(np.abs(blk).max()))
            for j in range(32):
                assert q[r, 32 * b + j] == oracle_lib.e4m3_encode(float(np.float32(blk[j]) / s[r, b]))
    assert s[1, 1] == 1.0 and not q[1, 32:64].any()
    # no saturation happens with a power-of-two scale >= amax/448
    dec = oracle_lib.e4m3_table()[q]
    assert np.all(np.abs(dec) <= 448.0)


# -------------------------------------------------------------------- GEMM
def _fr_tensor(A, B, sa, sb):
    M, K = A.shape
    N = B.shape[0]
    out = [[None] * N for _ in range(M)]
    alpha = np.float32(np.float32(sa) * np.float32(sb))
    for i in range(M):
        for j in range(N):
            acc = sum((dec_exact(int(A[i, k])) * dec_exact(int(B[j, k])) for k in range(K)), Fraction(0))
            out[i][j] = (Fraction(float(alpha)) * acc, acc)
    return out, alpha


def _fr_block(A, B, sfa, sfb):
    M, K = A.shape
    N = B.shape[0]
    out = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            tot = Fraction(0)
            for kb in range(K // 32):
                part = sum((dec_exact(int(A[i, k])) * dec_exact(int(B[j, k]))
                            for k in range(32 * kb, 32 * kb + 32)), Fraction(0))
                tot += Fraction(float(sfa[i, kb])) * Fraction(float(sfb[j, kb])) * part
            out[i][j] = tot
    return out


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C                      # no NaN codes
    return c


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 5, 32), (7, 2, 64), (9, 9, 64)])
def test_block_gemm_bruteforce_exact(oracle_lib, M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = _rand_codes(rng, (M, K))
    B = _rand_codes(rng, (N, K))
    sfa = (2.0 ** rng.integers(-8, 8, size=(M, K // 32))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-8, 8, size=(N, K // 32))).astype(np.float32)
    C, bound, exact = oracle_lib.gemm(A, B, sfa, sfb, block=True, out_kind=oracle_lib.OUT_F32,
                                      want_exact=True)
    Cb, _, _ = oracle_lib.gemm(A, B, sfa, sfb, block=True, out_kind=oracle_lib.OUT_BF16)
    ref = _fr_block(A, B, sfa, sfb)
    for i in range(M):
        for j in range(N):
            assert Fraction(exact[i, j]) == ref[i][j]                  # fp64 exact here
            assert Fraction(float(Cb[i, j])) == _bf16_exact(ref[i][j])  # direct RNE to bf16
            assert C[i, j] == np.float32(float(ref[i][j]))


def test_block_gemm_bruteforce_general_scales(oracle_lib):
    # literal fp32 amax/448-style scales (not powers of two) are accepted too
    rng = np.random.default_rng(9)
    A = _rand_codes(rng, (4, 64))
    B = _rand_codes(rng, (3, 64))
    sfa = rng.uniform(0.01, 3.0, size=(4, 2)).astype(np.float32)
    sfb = rng.uniform(0.01, 3.0, size=(3, 2)).astype(np.float32)
    _, bound, exact = oracle_lib.gemm(A, B, sfa, sfb, block=True, want_exact=True)
    ref = _fr_block(A, B, sfa, sfb)
    for i in range(4):
        for j in range(3):
            assert abs(Fraction(exact[i, j]) - ref[i][j]) <= abs(ref[i][j]) * Fraction(1, 2 ** 50)


@pytest.mark.parametrize("M,N,K", [(2, 3, 16), (5, 4, 48)])
def test_tensor_gemm_bruteforce_exact(oracle_lib, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = _rand_codes(rng, (M, K))
    B = _rand_codes(rng, (N, K))
    sa, sb = np.float32(0.37), np.float32(1.9e-3)
    C, _, exact = oracle_lib.gemm(A, B, np.array([sa]), np.array([sb]), block=False,
                                  out_kind=oracle_lib.OUT_F32, want_exact=True)
    ref, alpha = _fr_tensor(A, B, sa, sb)
    for i in range(M):
        for j in range(N):
            v, acc = ref[i][j]
            want = np.float32(float(v))                 # fl32(alpha * acc), exact product
            assert C[i, j] == want and exact[i, j] == float(want)


def test_identity_and_permutation_closed_form(oracle_lib):
    rng = np.random.default_rng(2)
    n = 64
    A = _rand_codes(rng, (n, n))
    eye = np.zeros((n, n), np.uint8)
    eye[np.arange(n), np.arange(n)] = 0x7E           # 448 = quantised 1.0 with sB = 1/448
    sa = np.float32(0.013)
    sb = np.float32(np.float32(1.0) / np.float32(448.0))
    C, _, _ = oracle_lib.gemm(A, eye, np.array([sa]), np.array([sb]), block=False,
                              out_kind=oracle_lib.OUT_F32)
    alpha = np.float32(sa * sb)
    dec = oracle_lib.e4m3_table()[A]
    want = (alpha.astype(np.float64) * (dec * 448.0)).astype(np.float32)
    assert np.array_equal(C, want)
    pi = rng.permutation(n)
    P = np.zeros((n, n), np.uint8)
    P[np.arange(n), pi] = 0x7E
    Cp, _, _ = oracle_lib.gemm(A, P, np.array([sa]), np.array([sb]), block=False,
                               out_kind=oracle_lib.OUT_F32)
    assert np.array_equal(Cp, want[:, pi])           # C[:, j] = alpha * 448 * dec(A[:, pi(j)])


def test_exhaustive_code_gemm(oracle_lib):
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    K = 256
    A = np.zeros((1, K), np.uint8)
    A[0, :len(codes)] = codes
    eye = np.zeros((K, K), np.uint8)
    eye[np.arange(K), np.arange(K)] = 0x38           # 1.0
    ones = np.ones((1, K // 32), np.float32)
    C, _, _ = oracle_lib.gemm(A, eye, ones, np.ones((K, K // 32), np.float32), block=True,
                              out_kind=oracle_lib.OUT_F32)
    tab = oracle_lib.e4m3_table()
    assert np.array_equal(C[0, :len(codes)], tab[codes].astype(np.float32))


def test_scaling_transpose_zero_laws(oracle_lib):
    rng = np.random.default_rng(8)
    A = _rand_codes(rng, (6, 96))
    B = _rand_codes(rng, (5, 96))
    sfa = (2.0 ** rng.integers(-4, 4, size=(6, 3))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-4, 4, size=(5, 3))).astype(np.float32)
    _, _, e1 = oracle_lib.gemm(A, B, sfa, sfb, True, want_exact=True)
    _, _, e2 = oracle_lib.gemm(A, B, sfa * 2, sfb, True, want_exact=True)
    _, _, et = oracle_lib.gemm(B, A, sfb, sfa, True, want_exact=True)
    _, _, ez = oracle_lib.gemm(np.zeros_like(A), B, sfa, sfb, True, want_exact=True)
    assert np.array_equal(e2, 2 * e1)
    assert np.array_equal(et, e1.T)
    assert not ez.any()


def test_tolerance_bound_uses_absolute_sums(oracle_lib):
    # a cancelling dot product: sum ab = 0 but sum |a||b| = K * 1
    K = 64
    A = np.full((1, K), 0x38, np.uint8)               # +1
    B = np.full((1, K), 0x38, np.uint8)
    B[0, ::2] = 0xB8                                   # -1 on even k
    ones = np.ones((1, 2), np.float32)
    C, bound, exact = oracle_lib.gemm(A, B, ones, ones, True, want_exact=True)
    assert exact[0, 0] == 0.0 and C[0, 0] == 0.0
    assert bound[0, 0] == pytest.approx(K * 2.0 ** -8 + 2.0 ** -133)


def test_sample_equals_full(oracle_lib):
    rng = np.random.default_rng(12)
    A = _rand_codes(rng, (20, 64))
    B = _rand_codes(rng, (17, 64))
    sfa = (2.0 ** rng.integers(-3, 3, size=(20, 2))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-3, 3, size=(17, 2))).astype(np.float32)
    C, bound, _ = oracle_lib.gemm(A, B, sfa, sfb, True)
    pi = rng.integers(0, 20, 50)
    pj = rng.integers(0, 17, 50)
    Cs, bs, _ = oracle_lib.gemm_sample(A, B, sfa, sfb, True, pi, pj)
    assert np.array_equal(Cs, C[pi, pj]) and np.array_equal(bs, bound[pi, pj])


def test_flop_count():
    import oracle
    assert oracle.gemm_flops(8192, 8192, 8192) == 2.0 * 8192 ** 3
    assert oracle.gemm_flops(128, 4096, 4096) == 4294967296.0


# ----------------------------------------------------------------- grouped
def _golden_raster():
    out = []
    for line in open(os.path.join(GOLDEN, "raster.txt")):
        if line.startswith("#") or not line.strip():
            continue
        out.append(line.split())
    return out


def test_raster_golden(oracle_lib):
    seen = 0
    for row in _golden_raster():
        if row[0] == "single":
            npm, npn, G = map(int, row[1:4])
            want = [tuple(map(int, x.split(","))) for x in row[4:]]
            got = [tuple(r) for r in oracle_lib.tile_map(npm * 128, npn * 256, 128, 256, G).tolist()]
            assert got == want
        else:
            counts = list(map(int, row[1].split(",")))
            N, BM, BN, G = map(int, row[2:6])
            want = [tuple(map(int, x.split(","))) + (0,) for x in row[6:]]
            got = [tuple(r) for r in oracle_lib.grouped_tile_map(counts, N, BM, BN, G).tolist()]
            assert got == want
        seen += 1
    assert seen == 3


@pytest.mark.parametrize("npm,npn,G", [(1, 1, 8), (64, 32, 8), (13, 7, 8), (5, 40, 3), (9, 1, 8)])
def test_raster_is_bijection(oracle_lib, npm, npn, G):
    tm = oracle_lib.tile_map(npm * 128, npn * 256, 128, 256, G)
    assert len({tuple(x) for x in tm.tolist()}) == npm * npn
    assert tm[:, 0].min() == 0 and tm[:, 0].max() == npm - 1
    assert tm[:, 1].min() == 0 and tm[:, 1].max() == npn - 1


def test_grouped_offsets_match_cumsum(oracle_lib):
    counts = np.array([120, 1, 3570, 0, 523, 15743, 4, 1], np.int32)
    off = oracle_lib.grouped_offsets(counts)
    assert off[0] == 0 and np.array_equal(off[1:], np.cumsum(counts))


def test_grouped_gemm_bruteforce(oracle_lib):
    rng = np.random.default_rng(21)
    counts = np.array([3, 0, 2, 1], np.int32)
    E, N, K = 4, 5, 64
    rows = int(counts.sum())
    A = _rand_codes(rng, (rows, K))
    B = _rand_codes(rng, (E, N, K))
    sfa = (2.0 ** rng.integers(-5, 5, size=(rows, K // 32))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-5, 5, size=(E, N, K // 32))).astype(np.float32)
    _, _, exact = oracle_lib.grouped_gemm(A, B, sfa, sfb, counts, want_exact=True)
    off = 0
    for e in range(E):
        for r in range(off, off + counts[e]):
            ref = _fr_block(A[r:r + 1], B[e], sfa[r:r + 1], sfb[e])
            for j in range(N):
                assert Fraction(exact[r, j]) == ref[0][j]
        off += counts[e]
