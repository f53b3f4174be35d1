"""Pins for the oracle's fused epilogue act(v + bias[j]): textbook values of
the standard normal CDF (GELU(x) = x Phi(x)), the odd-part identity
GELU(x) - GELU(-x) = x, ReLU's cases, and a brute-force GEMM in exact
rationals with bias and ReLU."""
import math
from fractions import Fraction

import numpy as np
import pytest

# Phi(x), standard normal CDF, from printed tables (10 significant digits)
PHI = {0.5: 0.6914624613, 1.0: 0.8413447461, 1.5: 0.9331927987, 2.0: 0.9772498681,
       3.0: 0.9986501020}


def test_gelu_textbook_values(oracle_lib):
    G = oracle_lib.ACT_GELU
    for x, phi in PHI.items():
        assert abs(oracle_lib.act(x, G) - x * phi) <= 1e-9 * x
        assert abs(oracle_lib.act(-x, G) - (-x) * (1.0 - phi)) <= 1e-9 * x
    assert oracle_lib.act(0.0, G) == 0.0
    assert oracle_lib.act(12.0, G) == 12.0 and oracle_lib.act(-40.0, G) == 0.0


def test_gelu_odd_part_identity(oracle_lib):
    G = oracle_lib.ACT_GELU
    for x in np.linspace(-6, 6, 97):
        assert abs(oracle_lib.act(x, G) - oracle_lib.act(-x, G) - x) <= 1e-14 * max(1.0, abs(x))


def test_relu_and_none(oracle_lib):
    R, N = oracle_lib.ACT_RELU, oracle_lib.ACT_NONE
    assert oracle_lib.act(-2.5, R) == 0.0 and oracle_lib.act(3.25, R) == 3.25
    assert math.isnan(oracle_lib.act(float("nan"), R))
    assert oracle_lib.act(-7.0, N) == -7.0


def _dec4(code):
    s = -1 if code & 0x80 else 1
    e, m = (code >> 3) & 15, code & 7
    if e == 0:
        return s * Fraction(m, 512)
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


@pytest.mark.parametrize("block", [True, False])
def test_gemm_bias_relu_bruteforce(oracle_lib, block):
    rng = np.random.default_rng(21 + block)
    M, N, K = 4, 5, 64
    A = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    B = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x30
    B[(B & 0x7F) == 0x7F] = 0x30
    if block:
        sfa = (2.0 ** rng.integers(-4, 4, size=(M, K // 32))).astype(np.float32)
        sfb = (2.0 ** rng.integers(-4, 4, size=(N, K // 32))).astype(np.float32)
    else:
        sfa, sfb = np.array([0.5], np.float32), np.array([0.25], np.float32)
    bias = rng.integers(-64, 64, size=N).astype(np.float32) * np.float32(0.5)
    C, bound, exact = oracle_lib.gemm(A, B, sfa, sfb, block, out_kind=oracle_lib.OUT_F32,
                                      want_exact=True, bias=bias, act_kind=oracle_lib.ACT_RELU)
    _, bound0, ex0 = oracle_lib.gemm(A, B, sfa, sfb, block, out_kind=oracle_lib.OUT_F32,
                                     want_exact=True)
    for i in range(M):
        for j in range(N):
            if block:
                v = sum(Fraction(float(sfa[i, kb])) * Fraction(float(sfb[j, kb])) *
                        sum((_dec4(int(A[i, k])) * _dec4(int(B[j, k]))
                             for k in range(32 * kb, 32 * kb + 32)), Fraction(0))
                        for kb in range(K // 32))
            else:   # fl32(fl32(sA sB) acc): exact here (acc has few significant bits)
                acc = sum((_dec4(int(A[i, k])) * _dec4(int(B[j, k])) for k in range(K)), Fraction(0))
                v = Fraction(float(np.float32(float(Fraction(0.125) * acc))))
            y = v + Fraction(float(bias[j]))
            want = y if y > 0 else Fraction(0)
            assert Fraction(exact[i, j]) == want
            assert C[i, j] == np.float32(float(want))
            # ReLU is 1-Lipschitz: the accumulation term is kept, the fp32 bias
            # term added (only the final-rounding ulp follows the new value)
            extra = 2.0 ** -20 * (abs(ex0[i, j]) + abs(float(bias[j])))
            assert bound[i, j] - extra - oracle_lib.bf16_ulp(float(C[i, j])) == pytest.approx(
                bound0[i, j] - oracle_lib.bf16_ulp(float(np.float32(ex0[i, j]))), rel=1e-12)
