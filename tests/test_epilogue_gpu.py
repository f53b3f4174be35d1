"""GPU parity of the fused epilogue (bias + activation) on every kernel path:
split-K, single-CTA and CTA-pair tiles, per-tensor and block-scaled, grouped
with per-expert bias rows."""
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


def _quant(x, block):
    q, s = fp8g.quantize(x.cuda(), block)
    qo, so = (oracle.quantize_block32 if block == 32 else oracle.quantize_tensor)(x.numpy())
    assert np.array_equal(q.cpu().numpy(), qo)
    return q, s, qo, so


@pytest.mark.parametrize("act", [0, 1, 2])
@pytest.mark.parametrize("block", [False, True])
@pytest.mark.parametrize("M,N,K", [(300, 392, 256), (300, 392, 2048), (1536, 2048, 256)])
def test_epilogue_full(act, block, M, N, K):
    g = torch.Generator().manual_seed(M + act)
    A = synth.normal((M, K), seed=M + 1)
    B = synth.normal((N, K), seed=N + 2)
    bias = (torch.randn(N, generator=g) * 4).numpy().astype(np.float32)
    bs = 32 if block else 0
    qa, sa, qa_o, sa_o = _quant(A, bs)
    qb, sb, qb_o, sb_o = _quant(B, bs)
    out = "bf16" if act != 1 else "f32"
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
    bias_d = torch.from_numpy(bias).cuda()
    fn = fp8g.fp8_gemm_blockscaled_ex if block else fp8g.fp8_gemm_ex
    fn(qa, qb, sa, sb, C, o, 0, 0, bias_d, act, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, block,
                                oracle.OUT_BF16 if out == "bf16" else oracle.OUT_F32,
                                bias=bias, act_kind=act)
    assert_within(C.float().cpu().numpy(), ref, bound, f"act {act} block={block} {M}x{N}x{K}")


@pytest.mark.parametrize("act", [1, 2])
@pytest.mark.parametrize("block", [False, True])
def test_epilogue_pairs_sampled(act, block):
    M, N, K = 4096, 4608, 256
    A = synth.normal((M, K), seed=5)
    B = synth.normal((N, K), seed=6)
    bias = np.linspace(-3, 3, N).astype(np.float32)
    bs = 32 if block else 0
    qa, sa, qa_o, sa_o = _quant(A, bs)
    qb, sb, qb_o, sb_o = _quant(B, bs)
    assert fp8g.fp8g_gemm_plan(int(block), M, N, K)["BM"] == 256
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fn = fp8g.fp8_gemm_blockscaled_ex if block else fp8g.fp8_gemm_ex
    fn(qa, qb, sa, sb, C, 0, 0, 0, torch.from_numpy(bias).cuda(), act, M, N, K)
    assert fp8g.fp8_gemm_status()[0] == 0
    rng = np.random.default_rng(act)
    pi = np.concatenate([rng.integers(0, M, 3000), [0, M - 1]])
    pj = np.concatenate([rng.integers(0, N, 3000), [N - 1, 0]])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, block, pi, pj, oracle.OUT_BF16,
                                       bias=bias, act_kind=act)
    assert_within(C.float().cpu().numpy()[pi, pj], ref, bound, f"pairs act {act}")


def test_epilogue_grouped_per_expert_bias():
    counts = np.array([3000, 0, 70, 9000, 257], np.int32)
    E, N, K = counts.size, 2048, 256
    w = synth.small_grouped(counts, N, K, seed=31)
    bias = np.random.default_rng(3).normal(size=(E, N)).astype(np.float32)
    qa, sa, qa_o, sa_o = _quant(w.A, 32)
    qb, sb, qb_o, sb_o = _quant(w.B.reshape(E * N, K), 32)
    rows = int(counts.sum())
    C = torch.empty((rows, N), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm_ex(qa, qb.reshape(E, N, K), sa, sb.reshape(E, N, K // 32), C, 0, 0, 0,
                             torch.from_numpy(bias).cuda(), 2, torch.from_numpy(counts).cuda(), E,
                             N, K, rows)
    assert fp8g.fp8_gemm_status()[0] == 0
    Ch = C.float().cpu().numpy()
    offs = oracle.grouped_offsets(counts)
    rng = np.random.default_rng(8)
    for e in range(E):
        m = int(counts[e])
        if m == 0:
            continue
        pi = rng.integers(0, m, 400)
        pj = rng.integers(0, N, 400)
        ref, bound, _ = oracle.gemm_sample(qa_o[offs[e]:offs[e + 1]], qb_o[e * N:(e + 1) * N],
                                           sa_o[offs[e]:offs[e + 1]], sb_o[e * N:(e + 1) * N],
                                           True, pi, pj, oracle.OUT_BF16, bias=bias[e],
                                           act_kind=2)
        assert_within(Ch[offs[e] + pi, pj], ref, bound, f"grouped expert {e}")


@pytest.mark.parametrize("act", [1, 2])
def test_epilogue_grouped_single_cta_bias_f32(act):
    """The grouped 128 x 128 plan (scales converted in the kernel): per-expert
    bias and activation on fp32 output, ragged N and K, every element."""
    counts = np.array([3, 250, 0, 129], np.int32)
    E, N, K = counts.size, 1040, 1120
    rows = int(counts.sum())
    assert fp8g.fp8g_grouped_plan(N, K, rows, E)["BM"] == 128
    w = synth.small_grouped(counts, N, K, seed=33 + act)
    bias = np.random.default_rng(5 + act).normal(size=(E, N)).astype(np.float32)
    qa, sa, qa_o, sa_o = _quant(w.A, 32)
    qb, sb, qb_o, sb_o = _quant(w.B.reshape(E * N, K), 32)
    C = torch.full((rows, N), float("nan"), dtype=torch.float32, device="cuda")
    fp8g.fp8_grouped_gemm_ex(qa, qb.reshape(E, N, K), sa, sb.reshape(E, N, K // 32), C,
                             fp8g.FP8G_OUT_F32, 0, 0, torch.from_numpy(bias).cuda(), act,
                             torch.from_numpy(counts).cuda(), E, N, K, rows)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    Ch = C.cpu().numpy()
    offs = oracle.grouped_offsets(counts)
    for e in range(E):
        if counts[e] == 0:
            continue
        ref, bound, _ = oracle.gemm(qa_o[offs[e]:offs[e + 1]], qb_o[e * N:(e + 1) * N],
                                    sa_o[offs[e]:offs[e + 1]], sb_o[e * N:(e + 1) * N], True,
                                    oracle.OUT_F32, bias=bias[e], act_kind=act)
        assert_within(Ch[offs[e]:offs[e + 1]], ref, bound, f"grouped single-CTA expert {e}")


def test_epilogue_bad_act_rejected():
    q = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, device="cuda")
    C = torch.empty(128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm_ex(q, q, s, s, C, 0, 0, 0, None, 7, 128, 128, 128)
    assert e.value.status == fp8g.FP8G_ERR_INVALID_ARG
