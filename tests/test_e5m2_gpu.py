"""GPU parity of the E5M2 and mixed-format paths: the quantiser bit-exact
against the oracle's, and the GEMMs (per-tensor, block-scaled, grouped; split-K,
single-CTA and CTA-pair kernels) within the tolerance for every pairing of
operand formats."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within

pytestmark = pytest.mark.gpu
E4, E5 = 0, 1
PAIRS = [(E4, E5), (E5, E4), (E5, E5)]


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def _quant(x: torch.Tensor, block: int, fmt: int):
    qg, sg = fp8g.quantize(x.cuda(), block, fmt=fmt)
    if block == 32:
        qo, so = oracle.quantize_block32(x.numpy(), fmt)
    else:
        qo, so = oracle.quantize_tensor(x.numpy(), fmt)
    assert np.array_equal(qg.cpu().numpy(), qo), f"{int((qg.cpu().numpy() != qo).sum())} code mismatches"
    assert np.array_equal(sg.cpu().numpy().reshape(so.shape).view(np.uint32), so.view(np.uint32))
    return qg, sg, qo, so


@pytest.mark.parametrize("block", [0, 32])
@pytest.mark.parametrize("rows,cols", [(1, 32), (37, 96), (256, 4096)])
def test_quantize_e5m2_bitexact(block, rows, cols):
    g = torch.Generator().manual_seed(rows * cols + block)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 4)
    x = synth.with_outliers(x, g)
    if rows > 1:
        x[0, :32] = 0.0
        x[-1, 3] = float("nan")
        x[-1, 5] = 1e30
        x[-1, 6] = float("-inf")
    _quant(x, block, E5)


def _operands(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    A = synth.with_outliers(synth.normal((M, K), seed=seed), g)
    B = synth.normal((N, K), seed=seed + 1) * torch.exp(torch.randn(N, 1, generator=g))
    return A, B


def _run(qa, sa, qb, sb, fa, fb, block, out, M, N, K):
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
    if block:
        fp8g.fp8_gemm_blockscaled_fmt(qa, qb, sa, sb, C, o, fa, fb, M, N, K)
    else:
        fp8g.fp8_gemm_fmt(qa, qb, sa, sb, C, o, fa, fb, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    return C.float().cpu().numpy()


@pytest.mark.parametrize("fa,fb", PAIRS)
@pytest.mark.parametrize("block", [False, True])
@pytest.mark.parametrize("M,N,K", [(300, 392, 256),      # single CTAs, 128 x 128 (few tiles, short K)
                                   (300, 392, 2048),     # split-K clusters (16 K steps)
                                   (1536, 2048, 384)])   # single-CTA tiles
def test_gemm_formats_full(fa, fb, block, M, N, K):
    A, B = _operands(M, N, K, seed=M + 7 * fa + 3 * fb)
    bs = 32 if block else 0
    qa, sa, qa_o, sa_o = _quant(A, bs, fa)
    qb, sb, qb_o, sb_o = _quant(B, bs, fb)
    out = "bf16" if fa == fb else "f32"
    C = _run(qa, sa, qb, sb, fa, fb, block, out, M, N, K)
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, block,
                                oracle.OUT_BF16 if out == "bf16" else oracle.OUT_F32,
                                a_fmt=fa, b_fmt=fb)
    assert_within(C, ref, bound, f"fmt {fa}x{fb} block={block} {M}x{N}x{K}")


@pytest.mark.parametrize("fa,fb", PAIRS)
@pytest.mark.parametrize("block", [False, True])
def test_gemm_formats_pairs_sampled(fa, fb, block):
    """CTA-pair kernel (256 x 256 tiles): 3000 sampled outputs plus corners."""
    M, N, K = 4096, 4608, 512
    plan = fp8g.fp8g_gemm_plan(int(block), M, N, K)
    assert plan["BM"] == 256
    A, B = _operands(M, N, K, seed=11 + fa + 2 * fb)
    bs = 32 if block else 0
    qa, sa, qa_o, sa_o = _quant(A, bs, fa)
    qb, sb, qb_o, sb_o = _quant(B, bs, fb)
    C = _run(qa, sa, qb, sb, fa, fb, block, "bf16", M, N, K)
    rng = np.random.default_rng(fa * 2 + fb)
    pi = np.concatenate([rng.integers(0, M, 3000), [0, 0, M - 1, M - 1]])
    pj = np.concatenate([rng.integers(0, N, 3000), [0, N - 1, 0, N - 1]])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, block, pi, pj, oracle.OUT_BF16,
                                       a_fmt=fa, b_fmt=fb)
    assert_within(C[pi, pj], ref, bound, f"pairs fmt {fa}x{fb} block={block}")


@pytest.mark.parametrize("counts,N,K", [([130, 0, 5, 257], 264, 256),
                                          ([3, 250, 0, 129], 4160, 1120)])
def test_grouped_e5m2_weights(counts, N, K):
    """E4M3 activations against E5M2 expert weights (grouped, block-scaled);
    the second shape puts two tiles on some CTAs and takes two scale windows
    per tile (9 K steps, the last one partial)."""
    counts = np.array(counts, np.int32)
    E = counts.size
    w = synth.small_grouped(counts, N, K, seed=77)
    qa, sa, qa_o, sa_o = _quant(w.A, 32, E4)
    qb, sb, qb_o, sb_o = _quant(w.B.reshape(E * N, K), 32, E5)
    rows = int(counts.sum())
    C = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm_fmt(qa, qb.reshape(E, N, K), sa, sb.reshape(E, N, K // 32), C,
                              fp8g.FP8G_OUT_BF16, E4, E5, torch.from_numpy(counts).cuda(), E, N, K,
                              rows)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    off = 0
    Ch = C.float().cpu().numpy()
    for e, m in enumerate(counts.tolist()):
        if m:
            ref, bound, _ = oracle.gemm(qa_o[off:off + m], qb_o[e * N:(e + 1) * N],
                                        sa_o[off:off + m], sb_o[e * N:(e + 1) * N], True,
                                        oracle.OUT_BF16, a_fmt=E4, b_fmt=E5)
            assert_within(Ch[off:off + m], ref, bound, f"grouped expert {e}")
        off += m


def test_bad_format_rejected():
    q = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, device="cuda")
    C = torch.empty(128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm_fmt(q, q, s, s, C, 0, 5, 0, 128, 128, 128)
    assert e.value.status == fp8g.FP8G_ERR_INVALID_ARG
    x = torch.zeros(4, 32, device="cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8g_quantize(x, 4, 32, 32, 5, q, s)
    assert e.value.status == fp8g.FP8G_ERR_INVALID_ARG
