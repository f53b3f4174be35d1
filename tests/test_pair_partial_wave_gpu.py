"""CTA-pair shapes whose last wave is partial: 2304 x 2304 has 81 pair tiles
on 76 pairs, the last 5 in raster order (tile-column 8, tile-rows 4-8) on a
second round.  Full comparisons against the oracle (per-tensor; block-scaled
with bias + GELU), MXFP4 on the FP4-rate kernel sampled over those last
tiles, and identical bits from call to call."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within, quant_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def _pair_plan(block, M, N, K):
    plan = fp8g.fp8g_gemm_plan(block, M, N, K)
    assert plan["BM"] == 256 and plan["BN"] == 256
    return plan


def test_partial_wave_per_tensor_full():
    M = N = 2304
    K = 1024
    _pair_plan(0, M, N, K)
    A = synth.normal((M, K), seed=31)
    B = synth.normal((N, K), seed=32)
    qa, sa, qa_o, sa_o = quant_both(A, 0)
    qb, sb, qb_o, sb_o = quant_both(B, 0)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fp8g.fp8_gemm(qa, qb, sa, sb, C, fp8g.FP8G_OUT_F32, M, N, K)
    assert fp8g.fp8_gemm_status()[0] == 0
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, False, oracle.OUT_F32)
    assert_within(C.cpu().numpy(), ref, bound, "partial wave per-tensor")


def test_partial_wave_block_bias_gelu_full_and_deterministic():
    M = N = 2304
    K = 1024
    _pair_plan(1, M, N, K)
    A = synth.normal((M, K), seed=33)
    B = synth.normal((N, K), seed=34)
    qa, sa, qa_o, sa_o = quant_both(A, 32)
    qb, sb, qb_o, sb_o = quant_both(B, 32)
    bias = torch.from_numpy(np.random.default_rng(35).normal(0, 4, N).astype(np.float32))
    outs = []
    for _ in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        fp8g.fp8_gemm_blockscaled_ex(qa, qb, sa, sb, C, 0, 0, 0, bias.cuda(), fp8g.FP8G_ACT_GELU,
                                     M, N, K)
        assert fp8g.fp8_gemm_status()[0] == 0
        outs.append(C)
    assert torch.equal(outs[0], outs[1])
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle.OUT_BF16,
                                bias=bias.numpy(), act_kind=oracle.ACT_GELU)
    assert_within(outs[0].float().cpu().numpy(), ref, bound, "partial wave block + bias + GELU")


def test_partial_wave_mxfp4_sampled():
    """FP4-rate pairs, 2304 x 2304 x 2048 (8 FP4 stages)."""
    M = N = 2304
    K = 2048
    _pair_plan(1, M, N, K)
    F4 = fp8g.FP8G_E2M1
    A = synth.normal((M, K), seed=36)
    B = synth.normal((N, K), seed=37)
    qa, sa = fp8g.quantize(A.cuda(), 32, fmt=F4)
    qb, sb = fp8g.quantize(B.cuda(), 32, fmt=F4)
    qa_o, sa_o = oracle.quantize_block32(A.numpy(), F4)
    qb_o, sb_o = oracle.quantize_block32(B.numpy(), F4)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled_fmt(qa, qb, sa, sb, C, 0, F4, F4, M, N, K)
    assert fp8g.fp8_gemm_status()[0] == 0
    Ch = C.float().cpu().numpy()
    assert not np.isnan(Ch).any()
    # the last 5 tiles in raster order: tile-column 8, tile-rows 4-8
    rng = np.random.default_rng(38)
    pi = np.concatenate([rng.integers(1024, M, 2500), rng.integers(0, M, 500), [M - 1, 1024]])
    pj = np.concatenate([rng.integers(2048, N, 2500), rng.integers(0, N, 500), [N - 1, 2048]])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, True, pi, pj, oracle.OUT_BF16,
                                       a_fmt=F4, b_fmt=F4)
    assert_within(Ch[pi, pj], ref, bound, "partial wave MXFP4")
