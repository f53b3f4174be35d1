"""Pins for the oracle's literal block scales (s = fl32(amax / fmax) per 1x32
block, the workloads' "fp32 scale = block amax/448" taken literally): the
scale is the fp32 quotient itself, the block maximum lands on +-fmax (or the
largest code below it), codes agree with torch's float8 cast of x / s, and a
GEMM over such scales matches exact rational arithmetic up to fp64 rounding."""
from fractions import Fraction

import numpy as np
import pytest
import torch


@pytest.mark.parametrize("fmt,fmax,tdt", [(0, 448.0, torch.float8_e4m3fn),
                                          (1, 57344.0, torch.float8_e5m2)])
def test_literal_block_scales(oracle_lib, fmt, fmax, tdt):
    g = torch.Generator().manual_seed(17 + fmt)
    x = torch.randn(6, 128, generator=g) * torch.exp(torch.randn(6, 1, generator=g) * 3)
    x[2, 32:64] = 0.0
    xn = x.numpy()
    q, s = oracle_lib.quantize_block32(xn, fmt, literal=True)
    for r in range(6):
        for b in range(4):
            blk = xn[r, 32 * b:32 * b + 32]
            amax = np.float32(np.abs(blk).max())
            want = np.float32(amax / np.float32(fmax)) if amax > 0 else np.float32(1.0)
            assert s[r, b] == want
            y = (torch.from_numpy(blk.copy()) / torch.tensor(s[r, b])).clamp(-fmax, fmax)
            assert np.array_equal(q[r, 32 * b:32 * b + 32], y.to(tdt).view(torch.uint8).numpy())
            if amax > 0:
                dec = oracle_lib.e4m3_table() if fmt == 0 else oracle_lib.e5m2_table()
                assert np.abs(dec[q[r, 32 * b:32 * b + 32]]).max() >= fmax * 0.93
    assert s[2, 1] == 1.0 and not q[2, 32:64].any()


def test_literal_scale_gemm_bruteforce(oracle_lib):
    """Non-power-of-two scales: fp64 result within 2^-45 relative of the exact
    rational sum (the per-block scale products no longer keep sums exact)."""
    rng = np.random.default_rng(4)
    x = rng.normal(size=(3, 64)).astype(np.float32)
    w = rng.normal(size=(4, 64)).astype(np.float32)
    qa, sa = oracle_lib.quantize_block32(x, 0, literal=True)
    qb, sb = oracle_lib.quantize_block32(w, 0, literal=True)
    _, _, exact = oracle_lib.gemm(qa, qb, sa, sb, True, oracle_lib.OUT_F32, want_exact=True)
    tab = oracle_lib.e4m3_table()
    for i in range(3):
        for j in range(4):
            tot = Fraction(0)
            for kb in range(2):
                part = sum((Fraction(tab[qa[i, k]]) * Fraction(tab[qb[j, k]])
                            for k in range(32 * kb, 32 * kb + 32)), Fraction(0))
                tot += Fraction(float(sa[i, kb])) * Fraction(float(sb[j, kb])) * part
            assert abs(Fraction(exact[i, j]) - tot) <= abs(tot) * Fraction(1, 2 ** 45)
