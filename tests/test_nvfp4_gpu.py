"""GPU parity of NVFP4 (E2M1 elements two per byte, 1x16 E4M3 block scales, an
fp32 scale per tensor): the quantiser bit-exact against the oracle (codes,
scale codes, tensor scale; fp32 and bf16 sources); an exact product pinning
the scale layout of the kind::mxf4nvf4 MMA (four scale bytes per row per
MMA); GEMMs within the tolerance, whole and sampled, with bias + GELU."""
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


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.uint8)
    return (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)


def _quant(x: torch.Tensor):
    """Both sides; the GPU's packed codes, scale codes and tensor scale must
    equal the oracle's.  Returns the GPU tensors and the oracle's codes (one
    per byte), scale codes and g."""
    q, sf, g = fp8g.quantize_nvfp4(x.cuda())
    assert fp8g.fp8_gemm_status()[0] == 0
    qo, sfo, go = oracle.quantize_nvfp4(x.float().numpy())
    gg = float(g.cpu().numpy()[0])
    assert np.float32(gg).view(np.uint32) == np.float32(go).view(np.uint32), (gg, go)
    assert np.array_equal(sf.cpu().numpy(), sfo), f"{int((sf.cpu().numpy() != sfo).sum())} scale mismatches"
    qg = q.cpu().numpy()
    assert np.array_equal(qg, pack_e2m1(qo)), f"{int((qg != pack_e2m1(qo)).sum())} code mismatches"
    return (q, sf, g), (qo, sfo, go)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,cols", [(96, 256), (7, 64), (130, 1040)])
def test_nvfp4_quantiser_bitexact(dtype, rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 2)
    x[min(3, rows - 1), :16] = 0.0                 # an all-zero block
    x[min(4, rows - 1), 5] = float("nan")          # NaN: left out of the amaxes, code +6
    x[min(5, rows - 1), 17] = -1e-30
    _quant(x.to(dtype))


def test_nvfp4_scale_layout_exact():
    """B[j, k] = 1 at k = j mod K, else 0; random E4M3 block scales on both
    sides (0.5 .. 4), tensor scales 1: C[i, j] = dec(a(i, k)) sa(i, k/16)
    sb(j, k/16), one exact product per output (fp32 out).  Every scale byte of
    every 64-wide K group and every nibble decides some output."""
    M, N, K = 512, 768, 512
    rng = np.random.default_rng(3)
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cb = np.zeros((N, K), np.uint8)
    cb[np.arange(N), np.arange(N) % K] = 2              # E2M1 1.0
    sa = rng.integers(0x30, 0x49, (M, K // 16)).astype(np.uint8)
    sb = rng.integers(0x30, 0x49, (N, K // 16)).astype(np.uint8)
    one = torch.ones(1, device="cuda")
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fp8g.fp8_gemm_nvfp4(torch.from_numpy(pack_e2m1(ca)).cuda(), torch.from_numpy(pack_e2m1(cb)).cuda(),
                        torch.from_numpy(sa).cuda(), torch.from_numpy(sb).cuda(), one, one, C,
                        fp8g.FP8G_OUT_F32, None, fp8g.FP8G_ACT_NONE, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    k = np.arange(N) % K
    va = oracle.e2m1_table()[ca[:, k]]
    s_a = oracle.nvfp4_scales(sa)[:, k // 16]
    s_b = oracle.nvfp4_scales(sb)[np.arange(N), k // 16]
    want = (va * s_a * s_b[None, :]).astype(np.float32)
    got = C.cpu().numpy()
    assert np.array_equal(got, want), f"{int((got != want).sum())} mismatches"


def _gemm(M, N, K, seed, out="bf16", bias=False, act=0, sample=None):
    A = synth.normal((M, K), seed=seed)
    B = synth.normal((N, K), seed=seed + 1) * 2.0
    (qa, sa, ga), (qa_o, sa_o, ga_o) = _quant(A)
    (qb, sb, gb), (qb_o, sb_o, gb_o) = _quant(B)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
    bias_v = np.random.default_rng(seed).normal(0, 2, N).astype(np.float32) if bias else None
    C = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    fp8g.fp8_gemm_nvfp4(qa, qb, sa, sb, ga, gb, C, o,
                        torch.from_numpy(bias_v).cuda() if bias else None, act, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    Ch = C.float().cpu().numpy()
    ok = oracle.OUT_BF16 if out == "bf16" else oracle.OUT_F32
    if sample is None:
        assert bias_v is None and act == 0
        ref, bound, _ = oracle.gemm_nvfp4(qa_o, qb_o, sa_o, sb_o, ga_o, gb_o, ok)
        assert_within(Ch, ref, bound, f"NVFP4 {M}x{N}x{K}")
        return
    rng = np.random.default_rng(M + N)
    pi = np.concatenate([[0, M - 1, M - 1], rng.integers(0, M, sample)])
    pj = np.concatenate([[N - 1, 0, N - 1], rng.integers(0, N, sample)])
    ref, bound, _ = oracle.gemm_nvfp4_sample(qa_o, qb_o, sa_o, sb_o, ga_o, gb_o, pi, pj, ok,
                                             bias=bias_v, act_kind=act)
    assert_within(Ch[pi, pj], ref, bound, f"NVFP4 {M}x{N}x{K} sampled")


@pytest.mark.parametrize("M,N,K", [(300, 520, 512), (256, 256, 256), (1, 16, 256)])
def test_nvfp4_gemm_full(M, N, K):
    _gemm(M, N, K, seed=M + K)


def test_nvfp4_gemm_f32_full():
    _gemm(700, 384, 768, seed=5, out="f32")


def test_nvfp4_gemm_large_sampled():
    assert fp8g.fp8g_gemm_plan(1, 2304, 2560, 1024)["BM"] == 256
    _gemm(2304, 2560, 1024, seed=11, sample=4000)


def test_nvfp4_gemm_bias_gelu_sampled():
    _gemm(1024, 768, 512, seed=13, bias=True, act=fp8g.FP8G_ACT_GELU, sample=3000)
