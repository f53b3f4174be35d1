"""Pins of the oracle's NVFP4 (E2M1 elements, 1x16 E4M3 block scales, one fp32
scale per tensor) against facts fixed without it: a worked example derived by
hand, closed forms, an exhaustive nearest-value search for the block scales,
the E2M1 rounding bound, and GEMM special cases that reduce to the pinned
E2M1 GEMM or to hand-computed values."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _lib(oracle_lib):
    yield


def test_worked_example():
    """Two blocks.  Block 1 holds 2688 = 6 x 448, so the tensor scale is 1 and
    its block scale 448 (E4M3 code 0x7E), 2688 / 448 = 6 -> code 7.  Block 0's
    amax is 7: t = 7 / 6 = 1.1667, whose nearest E4M3 value is 1.125 (code
    0x39; the neighbours are 1.125 and 1.25).  Its elements divided by 1.125,
    rounded to the nearest E2M1 value (ties to even), saturating at 6:
       0.5 -> 0.444 -> 0.5   1 -> 0.889 -> 1     1.5 -> 1.333 -> 1.5
       2 -> 1.778 -> 2       3 -> 2.667 -> 3     4 -> 3.556 -> 4
       6 -> 5.333 -> 6       -6 -> -6            0.25 -> 0.222 -> 0
       0.75 -> 0.667 -> 0.5  5 -> 4.444 -> 4     7 -> 6.222 -> 6 (saturated)
       -0.25 -> -0 (code 8)  0 -> 0              2.5 -> 2.222 -> 2
       -1 -> -0.889 -> -1"""
    x = np.zeros((1, 32), np.float32)
    x[0, :16] = [0.5, 1, 1.5, 2, 3, 4, 6, -6, 0.25, 0.75, 5, 7, -0.25, 0, 2.5, -1]
    x[0, 16] = 2688.0
    q, sf, g = oracle.quantize_nvfp4(x)
    assert g == 1.0
    assert sf.tolist() == [[0x39, 0x7E]]
    assert q[0, :16].tolist() == [1, 2, 3, 4, 5, 6, 7, 15, 0, 1, 6, 7, 8, 0, 4, 10]
    assert q[0, 16:].tolist() == [7] + [0] * 15


@pytest.mark.parametrize("c", [1e-3, 0.37, 1.0, 123.0, 3e4])
def test_constant_tensor(c):
    """Every |x| = c: g = fl32(c / 2688), each block's t is 448 up to one fp32
    rounding -> scale 448 (0x7E), and x / (448 g) = 6 up to rounding -> code 7
    (15 for -c)."""
    x = np.full((2, 32), c, np.float32)
    x[1] = -c
    q, sf, g = oracle.quantize_nvfp4(x)
    assert g == float(np.float32(c) / np.float32(2688))
    assert (sf == 0x7E).all()
    assert (q[0] == 7).all() and (q[1] == 15).all()


def test_zero_tensor_and_zero_block():
    x = np.zeros((1, 32), np.float32)
    q, sf, g = oracle.quantize_nvfp4(x)
    assert g == 1.0 and (sf == 0).all() and (q == 0).all()
    x[0, 20] = 3.0                      # block 0 all zero: scale 0, codes 0
    q, sf, g = oracle.quantize_nvfp4(x)
    assert sf[0, 0] == 0 and (q[0, :16] == 0).all()


def _e4m3_nonneg():
    t = oracle.e4m3_table()
    codes = [c for c in range(0x7F)]           # 0x00 .. 0x7E: +0 .. 448
    return np.array(codes), t[codes]


def test_block_scale_is_nearest_e4m3():
    """Exhaustive search over the 127 non-negative finite E4M3 values: the
    chosen scale is the nearest to t = amax_b / (6 g) (ties to the even
    code), with t evaluated in fp32 as the reading states."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.standard_normal((64, 1)) * 3)).astype(np.float32)
    q, sf, g = oracle.quantize_nvfp4(x)
    codes, vals = _e4m3_nonneg()
    g6 = np.float32(6) * np.float32(g)
    amax_b = np.abs(x).reshape(64, 16, 16).max(axis=2).astype(np.float32)
    t = (amax_b / g6).astype(np.float32).astype(np.float64)
    for (r, b), tv in np.ndenumerate(t):
        tv = min(tv, 448.0)                  # saturating
        d = np.abs(vals - tv)
        best = codes[d == d.min()]
        want = best[0] if best.size == 1 else best[best % 2 == 0][0]
        assert sf[r, b] == want, (r, b, tv, sf[r, b], want)


def test_elements_within_half_a_step():
    """|x / d - dec(q)| <= half the E2M1 spacing at that magnitude (0.25 below
    2, 0.5 below 4, 1 up to 6) for every element not saturated, d =
    dec(scale) g."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((32, 128)).astype(np.float32) * 5
    q, sf, g = oracle.quantize_nvfp4(x)
    dec = oracle.e2m1_table()[q]
    d = (oracle.nvfp4_scales(sf) * np.float32(g)).astype(np.float32)
    y = (x.reshape(32, 8, 16) / d[:, :, None]).reshape(32, 128).astype(np.float64)
    half = np.where(np.abs(y) < 2, 0.25, np.where(np.abs(y) < 4, 0.5, 1.0))
    ok = (np.abs(y - dec) <= half + 1e-12) | (np.abs(y) > 6)
    assert ok.all()


def test_gemm_unit_scales_is_e2m1_gemm():
    """All block scales 1.0 (E4M3 0x38) and gA = gB = 1: the E2M1 GEMM with
    per-tensor scales 1 (pinned in test_oracle_e2m1.py), bit for bit."""
    rng = np.random.default_rng(9)
    M, N, K = 24, 40, 96
    A = rng.integers(0, 16, (M, K)).astype(np.uint8)
    B = rng.integers(0, 16, (N, K)).astype(np.uint8)
    ones_a = np.full((M, K // 16), 0x38, np.uint8)
    ones_b = np.full((N, K // 16), 0x38, np.uint8)
    C, bound, exact = oracle.gemm_nvfp4(A, B, ones_a, ones_b, 1.0, 1.0, oracle.OUT_F32)
    one = np.ones(1, np.float32)
    C2, bound2, exact2 = oracle.gemm(A, B, one, one, False, oracle.OUT_F32, want_exact=True,
                                     a_fmt=oracle.E2M1, b_fmt=oracle.E2M1)
    assert np.array_equal(C, C2) and np.array_equal(exact, exact2)


def test_gemm_hand_value():
    """K = 32, one output: A = [1.0 x 16 | 2.0 x 16], B = 1.0 everywhere;
    block scales A (2.0, 0.5) = codes 0x40, 0x30, B (1.0, 4.0) = 0x38, 0x48;
    gA = 0.5, gB = 1:  0.5 (16 * 1 * 2*1 + 16 * 2 * 0.5*4) = 0.5 * 96 = 48."""
    A = np.array([[2] * 16 + [4] * 16], np.uint8)
    B = np.array([[2] * 32], np.uint8)
    C, _, exact = oracle.gemm_nvfp4(A, B, np.array([[0x40, 0x30]], np.uint8),
                                    np.array([[0x38, 0x48]], np.uint8), 0.5, 1.0, oracle.OUT_F32)
    assert exact[0, 0] == 48.0 and C[0, 0] == 48.0


def test_gemm_scale_linearity():
    """A block's scale code + 8 (one E4M3 binade up) doubles exactly the
    contribution of that block; gA = 2 doubles the whole result."""
    rng = np.random.default_rng(10)
    M, N, K = 8, 12, 64
    A = rng.integers(0, 16, (M, K)).astype(np.uint8)
    A[:, 16:] = 0                               # only block 0 of A is nonzero
    B = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sa = rng.integers(0x30, 0x50, (M, K // 16)).astype(np.uint8)
    sb = rng.integers(0x30, 0x50, (N, K // 16)).astype(np.uint8)
    _, _, e1 = oracle.gemm_nvfp4(A, B, sa, sb, 1.0, 1.0, oracle.OUT_F32)
    sa2 = sa.copy()
    sa2[:, 0] += 8
    _, _, e2 = oracle.gemm_nvfp4(A, B, sa2, sb, 1.0, 1.0, oracle.OUT_F32)
    assert np.array_equal(e2, 2 * e1)
    _, _, e3 = oracle.gemm_nvfp4(A, B, sa, sb, 2.0, 1.0, oracle.OUT_F32)
    assert np.array_equal(e3, 2 * e1)
