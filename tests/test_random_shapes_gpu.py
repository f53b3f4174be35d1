"""Seeded random shapes through the public entry points: ragged M, N and K,
both scale modes, both output types and mixed formats, so the kernel chooser
takes every path (split-K clusters, single-CTA tiles, CTA pairs).  Each case
is compared element by element with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def _cases(n=24, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.choice([1, 7, 129, 255, 300, 513, 700, 1100, 1600]))
        N = int(8 * rng.integers(1, 1600 // 8))
        K = int(32 * rng.integers(1, 1280 // 32))
        block = bool(rng.integers(0, 2))
        fa, fb = int(rng.integers(0, 2)), int(rng.integers(0, 2))
        out_t = "f32" if rng.integers(0, 3) == 0 else "bf16"
        out.append((i, M, N, K, block, fa, fb, out_t))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c[1]}x{c[2]}x{c[3]}-b{int(c[4])}-f{c[5]}{c[6]}-{c[7]}")
def test_random_shape(case):
    i, M, N, K, block, fa, fb, out_t = case
    g = torch.Generator().manual_seed(100 + i)
    A = synth.with_outliers(synth.normal((M, K), seed=1000 + i), g)
    B = synth.normal((N, K), seed=2000 + i) * torch.exp(torch.randn(N, 1, generator=g))
    bs = 32 if block else 0
    qa, sa = fp8g.quantize(A.cuda(), bs, fmt=fa)
    qb, sb = fp8g.quantize(B.cuda(), bs, fmt=fb)
    qfn = oracle.quantize_block32 if block else oracle.quantize_tensor
    qa_o, sa_o = qfn(A.numpy(), fa)
    qb_o, sb_o = qfn(B.numpy(), fb)
    assert np.array_equal(qa.cpu().numpy(), qa_o) and np.array_equal(qb.cpu().numpy(), qb_o)
    dt = torch.bfloat16 if out_t == "bf16" else torch.float32
    C = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    o = fp8g.FP8G_OUT_BF16 if out_t == "bf16" else fp8g.FP8G_OUT_F32
    fn = fp8g.fp8_gemm_blockscaled_fmt if block else fp8g.fp8_gemm_fmt
    fn(qa, qb, sa, sb, C, o, fa, fb, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, block,
                                oracle.OUT_BF16 if out_t == "bf16" else oracle.OUT_F32,
                                a_fmt=fa, b_fmt=fb)
    plan = fp8g.fp8g_gemm_plan(int(block), M, N, K)
    assert_within(C.float().cpu().numpy(), ref, bound, f"case {case} plan {plan}")


def _pair_cases(n=6, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.integers(2400, 5000))
        N = int(8 * rng.integers(2400 // 8, 5000 // 8))
        K = int(32 * rng.integers(2, 40))
        out.append((i, M, N, K, bool(i % 2), int(rng.integers(0, 2)), int(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("case", _pair_cases(), ids=lambda c: f"{c[1]}x{c[2]}x{c[3]}-b{int(c[4])}-f{c[5]}{c[6]}")
def test_random_pair_shape_sampled(case):
    """Ragged shapes large enough for CTA pairs; 3000 sampled outputs plus the
    corners and the last row / column of every tile edge region."""
    i, M, N, K, block, fa, fb = case
    assert fp8g.fp8g_gemm_plan(int(block), M, N, K)["BM"] == 256
    A = synth.normal((M, K), seed=3000 + i)
    B = synth.normal((N, K), seed=4000 + i)
    bs = 32 if block else 0
    qa, sa = fp8g.quantize(A.cuda(), bs, fmt=fa)
    qb, sb = fp8g.quantize(B.cuda(), bs, fmt=fb)
    qfn = oracle.quantize_block32 if block else oracle.quantize_tensor
    qa_o, sa_o = qfn(A.numpy(), fa)
    qb_o, sb_o = qfn(B.numpy(), fb)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fn = fp8g.fp8_gemm_blockscaled_fmt if block else fp8g.fp8_gemm_fmt
    fn(qa, qb, sa, sb, C, 0, fa, fb, M, N, K)
    assert fp8g.fp8_gemm_status()[0] == 0
    Ch = C.float().cpu().numpy()
    assert not np.isnan(Ch).any()                      # every output written
    rng = np.random.default_rng(i)
    edge_r = np.array([0, M - 1, (M - 1) // 256 * 256, min(M - 1, (M - 1) // 256 * 256 + 255)])
    edge_c = np.array([0, N - 1, (N - 1) // 256 * 256, N - 2])
    pi = np.concatenate([rng.integers(0, M, 3000), np.repeat(edge_r, 4)])
    pj = np.concatenate([rng.integers(0, N, 3000), np.tile(edge_c, 4)])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, block, pi, pj, oracle.OUT_BF16,
                                       a_fmt=fa, b_fmt=fb)
    assert_within(Ch[pi, pj], ref, bound, f"pair case {case}")
