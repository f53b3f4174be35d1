"""GPU parity of the literal-scale path: the quantiser with s = fl32(amax/fmax)
per 1x32 block bit-exact against the oracle, and the promotion GEMM (tensor
core partials per 32-wide K block, scaled and accumulated on CUDA cores)
within the tolerance for arbitrary fp32 scales, formats and the epilogue."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within

pytestmark = pytest.mark.gpu
LIT = 33


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def _quant_literal(x: torch.Tensor, fmt: int = 0):
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    s = torch.empty((rows, cols // 32), dtype=torch.float32, device="cuda")
    dtype = fp8g.FP8G_IN_BF16 if x.dtype == torch.bfloat16 else fp8g.FP8G_IN_F32
    fp8g.fp8g_quantize_rows(x.cuda(), dtype, rows, cols, None, rows, LIT, fmt, q, s)
    assert fp8g.fp8_gemm_status()[0] == 0
    qo, so = oracle.quantize_block32(x.float().numpy(), fmt, literal=True)
    assert np.array_equal(q.cpu().numpy(), qo), f"{int((q.cpu().numpy() != qo).sum())} mismatches"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    return q, s, qo, so


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [0, 1])
def test_literal_quantiser_bitexact(dtype, fmt):
    g = torch.Generator().manual_seed(fmt + 3)
    x = (torch.randn(200, 256, generator=g) * torch.exp(torch.randn(200, 1, generator=g) * 3))
    x[5, 64:96] = 0.0
    _quant_literal(x.to(dtype), fmt)


def _run(qa, sa, qb, sb, M, N, K, out="bf16", fa=0, fb=0, bias=None, act=0):
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
    b = torch.from_numpy(bias).cuda() if bias is not None else None
    fp8g.fp8_gemm_blockscaled_promote(qa, qb, sa, sb, C, o, fa, fb, b, act, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    return C.float().cpu().numpy()


@pytest.mark.parametrize("M,N,K,out", [(300, 392, 256, "bf16"), (1024, 1024, 1024, "f32"),
                                       (1, 8, 128, "bf16"), (129, 136, 4224, "bf16")])
def test_promote_literal_full(M, N, K, out):
    g = torch.Generator().manual_seed(M + K)
    A = synth.with_outliers(synth.normal((M, K), seed=M), g)
    B = synth.normal((N, K), seed=N) * torch.exp(torch.randn(N, 1, generator=g) * 2)
    qa, sa, qa_o, sa_o = _quant_literal(A)
    qb, sb, qb_o, sb_o = _quant_literal(B)
    C = _run(qa, sa, qb, sb, M, N, K, out)
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True,
                                oracle.OUT_BF16 if out == "bf16" else oracle.OUT_F32)
    assert_within(C, ref, bound, f"promote {M}x{N}x{K}")


def test_promote_arbitrary_signed_scales_formats_epilogue():
    """Scales of any sign and magnitude (not from a quantiser), E4M3 x E5M2,
    bias + GELU."""
    M, N, K = 384, 512, 512
    rng = np.random.default_rng(9)
    qa_o = rng.integers(0, 256, (M, K), dtype=np.uint8)
    qb_o = rng.integers(0, 256, (N, K), dtype=np.uint8)
    qa_o[(qa_o & 0x7F) == 0x7F] = 0x30
    qb_o[(qb_o & 0x7C) == 0x7C] = 0x31                    # no E5M2 inf / NaN
    sa_o = (rng.normal(size=(M, K // 32)) * 1e-2).astype(np.float32)
    sb_o = (rng.normal(size=(N, K // 32)) * 3e-3).astype(np.float32)
    bias = rng.normal(size=N).astype(np.float32)
    C = _run(torch.from_numpy(qa_o).cuda(), torch.from_numpy(sa_o).cuda(),
             torch.from_numpy(qb_o).cuda(), torch.from_numpy(sb_o).cuda(), M, N, K, "f32", 0, 1,
             bias, fp8g.FP8G_ACT_GELU)
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle.OUT_F32, a_fmt=0, b_fmt=1,
                                bias=bias, act_kind=oracle.ACT_GELU)
    assert_within(C, ref, bound, "promote signed scales")


def test_promote_large_sampled():
    M = N = 4096
    K = 2048
    A = synth.normal((M, K), seed=41)
    B = synth.normal((N, K), seed=42)
    qa, sa, qa_o, sa_o = _quant_literal(A)
    qb, sb, qb_o, sb_o = _quant_literal(B)
    C = _run(qa, sa, qb, sb, M, N, K)
    rng = np.random.default_rng(5)
    pi = np.concatenate([rng.integers(0, M, 3000), [0, M - 1]])
    pj = np.concatenate([rng.integers(0, N, 3000), [N - 1, 0]])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, True, pi, pj, oracle.OUT_BF16)
    assert_within(C[pi, pj], ref, bound, "promote 4096x4096x2048")


def test_promote_rejects_k_not_multiple_of_128():
    q = torch.zeros(128, 96, dtype=torch.uint8, device="cuda")
    s = torch.ones(128, 3, device="cuda")
    C = torch.empty(128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm_blockscaled_promote(q, torch.zeros(128, 96, dtype=torch.uint8, device="cuda"),
                                          s, s, C, 0, 0, 0, None, 0, 128, 128, 96)
    assert e.value.status == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("fa,fb,out", [(0, 1, "f32"), (1, 0, "bf16")])
def test_promote_tf32_route_full(fa, fb, out):
    """Shapes with a wave of 256 x 256 tiles take the TF32 route (operands
    dequantised with their fp32 scales, then the TF32 tensor-core GEMM on CTA
    pairs): ragged M and N, signed arbitrary scales, E4M3 x E5M2 either way,
    bias + GELU; the whole output against the oracle."""
    M, N, K = 2000, 2600, 640
    assert fp8g.fp8g_gemm_plan(0, M, N, K)["BM"] == 256          # the pair plan
    rng = np.random.default_rng(fa * 2 + fb)
    qa_o = rng.integers(0, 256, (M, K), dtype=np.uint8)
    qb_o = rng.integers(0, 256, (N, K), dtype=np.uint8)
    for q, f in ((qa_o, fa), (qb_o, fb)):
        if f == 0:
            q[(q & 0x7F) == 0x7F] = 0x30                            # no E4M3 NaN
        else:
            q[(q & 0x7C) == 0x7C] = 0x31                            # no E5M2 inf / NaN
    sa_o = (rng.normal(size=(M, K // 32)) * 1e-2).astype(np.float32)
    sb_o = (rng.normal(size=(N, K // 32)) * 3e-3).astype(np.float32)
    bias = rng.normal(size=N).astype(np.float32)
    C = _run(torch.from_numpy(qa_o).cuda(), torch.from_numpy(sa_o).cuda(),
             torch.from_numpy(qb_o).cuda(), torch.from_numpy(sb_o).cuda(), M, N, K, out, fa, fb,
             bias, fp8g.FP8G_ACT_GELU)
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True,
                                oracle.OUT_F32 if out == "f32" else oracle.OUT_BF16, a_fmt=fa,
                                b_fmt=fb, bias=bias, act_kind=oracle.ACT_GELU)
    assert_within(C, ref, bound, f"promote TF32 route {fa}x{fb}")


def test_promote_tf32_route_nan_propagates():
    """A NaN code on the TF32 route gives NaN exactly in its row / column."""
    M, N, K = 4096, 2048, 256
    qa = torch.full((M, K), 0x38, dtype=torch.uint8, device="cuda")   # 1.0
    qb = torch.full((N, K), 0x38, dtype=torch.uint8, device="cuda")
    qa[17, 100] = 0x7F                                                 # NaN
    s = torch.full((M, K // 32), 0.5, device="cuda")
    sb = torch.full((N, K // 32), 0.25, device="cuda")
    C = _run(qa, s, qb, sb, M, N, K, "f32")
    assert np.isnan(C[17]).all() and not np.isnan(np.delete(C, 17, axis=0)).any()
    assert (np.delete(C, 17, axis=0) == K * 0.5 * 0.25).all()          # exact sums
