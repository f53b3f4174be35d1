"""GPU parity of E2M1 (FP4) operands, stored two codes per byte (element 2j in
the low nibble of byte j): the quantiser bit-exact against the oracle's codes
packed the same way (power-of-two 1x32 scales: MXFP4; per-tensor; fp32 and
bf16 sources); the packed layout pinned through an identity product; GEMMs
with E2M1 on one or both sides within the tolerance on the split-K,
single-CTA, CTA-pair and grouped kernels."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within

pytestmark = pytest.mark.gpu
F4 = fp8g.FP8G_E2M1


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """One code per byte [r, c] -> two per byte [r, c/2], element 2j low."""
    c = codes.astype(np.uint8)
    return (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)


def _quant(x: torch.Tensor, block: int, fmt: int):
    """Quantise on both sides; GPU codes (packed for E2M1) must equal the
    oracle's codes (packed the same way).  Returns the GPU codes and scales
    and the oracle's one-code-per-byte codes and scales."""
    rows, cols = x.shape
    qcols = cols // 2 if fmt == F4 else cols
    q = torch.empty((rows, qcols), dtype=torch.uint8, device="cuda")
    s = torch.empty((rows, cols // 32) if block else (1,), dtype=torch.float32, device="cuda")
    dt = fp8g.FP8G_IN_BF16 if x.dtype == torch.bfloat16 else fp8g.FP8G_IN_F32
    fp8g.fp8g_quantize_rows(x.cuda(), dt, rows, cols, None, rows, block, fmt, q, s)
    assert fp8g.fp8_gemm_status()[0] == 0
    xf = x.float().numpy()
    qo, so = (oracle.quantize_block32 if block else oracle.quantize_tensor)(xf, fmt)
    want = pack_e2m1(qo) if fmt == F4 else qo
    qg = q.cpu().numpy()
    assert np.array_equal(qg, want), f"{int((qg != want).sum())} code byte mismatches"
    assert np.array_equal(s.cpu().numpy().reshape(so.shape).view(np.uint32), so.view(np.uint32))
    return q, s, qo, so


@pytest.mark.parametrize("block", [0, 32])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_e2m1_quantiser_bitexact(block, dtype):
    g = torch.Generator().manual_seed(block + 5)
    x = torch.randn(96, 256, generator=g) * torch.exp(torch.randn(96, 1, generator=g) * 2)
    x[3, :32] = 0.0
    x[4, 7] = -1e-30                                  # rounds to -0
    x[5, 9] = float("nan")
    x[6, 1] = float("inf")
    if block == 0:
        x[5, 9] = 1.0
        x[6, 1] = 2.0                                 # keep the per-tensor scale finite
    _quant(x.to(dtype), block, F4)


def test_e2m1_quantiser_gather_bf16():
    """Row gather + bf16 source + packed output in one pass; a ragged row
    count (not a multiple of any tile)."""
    g = torch.Generator().manual_seed(77)
    x = (torch.randn(50, 512, generator=g) * 3).to(torch.bfloat16)
    rows = torch.tensor([49, 0, 7, 7, 31, 12, 3], dtype=torch.int32)
    q = torch.empty((rows.numel(), 256), dtype=torch.uint8, device="cuda")
    s = torch.empty((rows.numel(), 16), dtype=torch.float32, device="cuda")
    fp8g.fp8g_quantize_rows(x.cuda(), fp8g.FP8G_IN_BF16, 50, 512, rows.cuda(), rows.numel(), 32,
                            F4, q, s)
    assert fp8g.fp8_gemm_status()[0] == 0
    qo, so = oracle.quantize_block32(x.float().numpy()[rows.numpy()], F4)
    assert np.array_equal(q.cpu().numpy(), pack_e2m1(qo))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


def test_e2m1_packed_layout_identity():
    """C = A I with per-tensor scales 1 and B the E4M3 identity (1.0 = 0x38):
    every output is one decoded E2M1 value, exact in fp32.  Pins the nibble
    order and the 16U4 tile layout against the oracle's decode table."""
    M = N = K = 256
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 16, (M, K)).astype(np.uint8)
    A = torch.from_numpy(pack_e2m1(codes)).cuda()
    B = torch.from_numpy((np.eye(N, K) * 0x38).astype(np.uint8)).cuda()
    one = torch.ones(1, device="cuda")
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fp8g.fp8_gemm_fmt(A, B, one, one, C, fp8g.FP8G_OUT_F32, F4, 0, M, N, K)
    assert fp8g.fp8_gemm_status()[0] == 0
    want = oracle.e2m1_table()[codes].astype(np.float32)
    got = C.cpu().numpy()
    assert np.array_equal(got, want), f"{int((got != want).sum())} mismatches"


def _gemm(fa, fb, block, M, N, K, sample=None):
    g = torch.Generator().manual_seed(M + N + fa)
    A = synth.normal((M, K), seed=M + fa)
    B = synth.normal((N, K), seed=N + fb) * torch.exp(torch.randn(N, 1, generator=g))
    bs = 32 if block else 0
    qa, sa, qa_o, sa_o = _quant(A, bs, fa)
    qb, sb, qb_o, sb_o = _quant(B, bs, fb)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fn = fp8g.fp8_gemm_blockscaled_fmt if block else fp8g.fp8_gemm_fmt
    fn(qa, qb, sa, sb, C, 0, fa, fb, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    Ch = C.float().cpu().numpy()
    if sample is None:
        ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, block, oracle.OUT_BF16,
                                    a_fmt=fa, b_fmt=fb)
        assert_within(Ch, ref, bound, f"E2M1 {fa}x{fb} block={block} {M}x{N}x{K}")
    else:
        rng = np.random.default_rng(M)
        pi, pj = rng.integers(0, M, sample), rng.integers(0, N, sample)
        ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, block, pi, pj,
                                           oracle.OUT_BF16, a_fmt=fa, b_fmt=fb)
        assert_within(Ch[pi, pj], ref, bound, f"E2M1 {fa}x{fb} block={block} {M}x{N}x{K}")


@pytest.mark.parametrize("fa,fb", [(F4, F4), (0, F4), (F4, 1)])
@pytest.mark.parametrize("block", [False, True])
@pytest.mark.parametrize("M,N,K", [(300, 392, 256), (300, 392, 2048), (1536, 2048, 384)])
def test_e2m1_gemm_full(fa, fb, block, M, N, K):
    _gemm(fa, fb, block, M, N, K)


@pytest.mark.parametrize("block", [False, True])
def test_e2m1_gemm_pairs_sampled(block):
    assert fp8g.fp8g_gemm_plan(int(block), 4096, 4608, 512)["BM"] == 256
    _gemm(F4, F4, block, 4096, 4608, 512, sample=3000)


def test_e2m1_promote_literal_scales():
    """E2M1 operands with literal fp32 1x32 scales (amax / 6) through the
    promotion kernel."""
    M, N, K = 260, 384, 512
    A = synth.normal((M, K), seed=91)
    B = synth.normal((N, K), seed=92)
    out = []
    for x, rows in ((A, M), (B, N)):
        q = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
        s = torch.empty((rows, K // 32), dtype=torch.float32, device="cuda")
        fp8g.fp8g_quantize_rows(x.cuda(), fp8g.FP8G_IN_F32, rows, K, None, rows,
                                fp8g.FP8G_BLOCK32_LITERAL, F4, q, s)
        qo, so = oracle.quantize_block32(x.numpy(), F4, literal=True)
        assert np.array_equal(q.cpu().numpy(), pack_e2m1(qo))
        assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
        out.append((q, s, qo, so))
    (qa, sa, qa_o, sa_o), (qb, sb, qb_o, sb_o) = out
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled_promote(qa, qb, sa, sb, C, 0, F4, F4, None, 0, M, N, K)
    assert fp8g.fp8_gemm_status()[0] == 0
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle.OUT_BF16, a_fmt=F4, b_fmt=F4)
    assert_within(C.float().cpu().numpy(), ref, bound, "E2M1 literal promote")


def test_e2m1_grouped():
    """Grouped MoE GEMM with E2M1 activations and E2M1 expert weights (the 3-D
    packed B map), ragged and empty experts."""
    counts = np.array([130, 0, 5, 257], np.int32)
    E, N, K = counts.size, 264, 256
    w = synth.small_grouped(counts, N, K, seed=41)
    qa, sa, qa_o, sa_o = _quant(w.A, 32, F4)
    qb, sb, qb_o, sb_o = _quant(w.B.reshape(E * N, K), 32, F4)
    rows = int(counts.sum())
    C = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm_fmt(qa, qb.reshape(E, N, K // 2), sa, sb.reshape(E, N, K // 32), C, 0,
                              F4, F4, torch.from_numpy(counts).cuda(), E, N, K, rows)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    # the oracle's grouped GEMM decodes its operands as E4M3: compare per
    # expert through the format-aware GEMM instead
    offs = oracle.grouped_offsets(counts)
    Ch = C.float().cpu().numpy()
    qb_o = qb_o.reshape(E, N, K)
    sb_o = sb_o.reshape(E, N, K // 32)
    for e in range(E):
        if counts[e] == 0:
            continue
        r0, r1 = offs[e], offs[e + 1]
        ref, bound, _ = oracle.gemm(qa_o[r0:r1], qb_o[e], sa_o[r0:r1], sb_o[e], True,
                                    oracle.OUT_BF16, a_fmt=F4, b_fmt=F4)
        assert_within(Ch[r0:r1], ref, bound, f"E2M1 grouped expert {e}")


# ---------------------------------------------------------------- FP4 rate
# MXFP4 (E2M1 x E2M1, 1x32 power-of-two scales) on CTA pairs with K % 256 == 0
# runs kind::mxf4: dense 4-bit operands, K = 64 per MMA, two scale bytes per
# row per MMA.  Pair shapes: at least a wave of 128 x 256 tiles.

def test_mxfp4_pair_scale_layout_exact():
    """B[j, k] = 1 at k = j mod K, else 0, with random power-of-two scales on
    both sides: C[i, j] = a(i, k) sfa(i, k/32) sfb(j, k/32) for k = j mod K,
    one exact product per output (fp32 out).  Every K block of every stage
    appears, so a wrong scale byte, K group or nibble fails bit-exactly."""
    M, N, K = 2048, 2560, 512
    assert fp8g.fp8g_gemm_plan(1, M, N, K)["BM"] == 256
    rng = np.random.default_rng(5)
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cb = np.zeros((N, K), np.uint8)
    cb[np.arange(N), np.arange(N) % K] = 2                       # E2M1 code 2 = 1.0
    sfa = np.exp2(rng.integers(-4, 5, (M, K // 32))).astype(np.float32)
    sfb = np.exp2(rng.integers(-4, 5, (N, K // 32))).astype(np.float32)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fp8g.fp8_gemm_blockscaled_fmt(torch.from_numpy(pack_e2m1(ca)).cuda(),
                                  torch.from_numpy(pack_e2m1(cb)).cuda(),
                                  torch.from_numpy(sfa).cuda(), torch.from_numpy(sfb).cuda(), C,
                                  fp8g.FP8G_OUT_F32, F4, F4, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    k = np.arange(N) % K
    want = (oracle.e2m1_table()[ca[:, k]] * sfa[:, k // 32] * sfb[np.arange(N), k // 32][None, :])
    got = C.cpu().numpy()
    assert np.array_equal(got, want.astype(np.float32)), f"{int((got != want).sum())} mismatches"


def _sampled(qa_o, qb_o, sa_o, sb_o, Ch, M, N, pts, what):
    rng = np.random.default_rng(M + N)
    edge_i = np.array([0, 1, 127, 128, 255, 256, M - 1, M - 2, M - 129])
    edge_j = np.array([0, 1, 127, 128, 255, 256, N - 1, N - 2, N - 129])
    pi = np.concatenate([np.repeat(edge_i, edge_j.size), rng.integers(0, M, pts)])
    pj = np.concatenate([np.tile(edge_j, edge_i.size), rng.integers(0, N, pts)])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, True, pi, pj, oracle.OUT_BF16,
                                       a_fmt=F4, b_fmt=F4)
    assert_within(Ch[pi, pj], ref, bound, what)


@pytest.mark.parametrize("M,N,K", [(2100, 2600, 768), (2048, 2560, 384)])
def test_mxfp4_pair_ragged_sampled(M, N, K):
    """Ragged M and N on pairs: K = 768 takes the FP4-rate kernel (3 stages);
    K = 384 (not a multiple of 256) the FP8-rate pair kernel with 4-bit loads."""
    assert fp8g.fp8g_gemm_plan(1, M, N, K)["BM"] == 256
    A = synth.normal((M, K), seed=M)
    B = synth.normal((N, K), seed=N) * 3.0
    qa, sa, qa_o, sa_o = _quant(A, 32, F4)
    qb, sb, qb_o, sb_o = _quant(B, 32, F4)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled_fmt(qa, qb, sa, sb, C, 0, F4, F4, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    _sampled(qa_o, qb_o, sa_o, sb_o, C.float().cpu().numpy(), M, N, 4000,
             f"MXFP4 pairs {M}x{N}x{K}")


def test_mxfp4_pair_full_f32():
    """A whole pair-shaped output against the oracle (fp32 out, one stage)."""
    M, N, K = 2304, 2304, 256
    assert fp8g.fp8g_gemm_plan(1, M, N, K)["BM"] == 256
    A = synth.normal((M, K), seed=8)
    B = synth.normal((N, K), seed=9)
    qa, sa, qa_o, sa_o = _quant(A, 32, F4)
    qb, sb, qb_o, sb_o = _quant(B, 32, F4)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fp8g.fp8_gemm_blockscaled_fmt(qa, qb, sa, sb, C, fp8g.FP8G_OUT_F32, F4, F4, M, N, K)
    assert fp8g.fp8_gemm_status()[0] == 0
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle.OUT_F32, a_fmt=F4, b_fmt=F4)
    assert_within(C.cpu().numpy(), ref, bound, "MXFP4 pairs full f32")


def test_mxfp4_grouped_pairs_sampled():
    """Grouped MoE GEMM on pairs at the FP4 rate: empty, one-row and ragged
    experts; offsets and tile map bit-exact; sampled outputs per expert."""
    counts = np.array([3000, 0, 70, 9000, 257, 1, 0, 129], np.int32)
    E, N, K = counts.size, 2048, 512
    rows = int(counts.sum())
    plan = fp8g.fp8g_grouped_plan(N, K, rows, E)
    assert plan["BM"] == 256
    w = synth.small_grouped(counts, N, K, seed=29)
    qa, sa, qa_o, sa_o = _quant(w.A, 32, F4)
    qb, sb, qb_o, sb_o = _quant(w.B.reshape(E * N, K), 32, F4)
    C = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    tmap = torch.full((plan["max_tiles"], 4), -1, dtype=torch.int32, device="cuda")
    fp8g.fp8_grouped_gemm_fmt(qa, qb.reshape(E, N, K // 2), sa, sb.reshape(E, N, K // 32), C, 0,
                              F4, F4, torch.from_numpy(counts).cuda(), E, N, K, rows, offs, tmap)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    offs_o = oracle.grouped_offsets(counts)
    assert np.array_equal(offs.cpu().numpy(), offs_o)
    want = oracle.grouped_tile_map(counts, N, plan["BM"], plan["BN"], plan["G"])
    assert np.array_equal(tmap.cpu().numpy()[:want.shape[0]], want)
    Ch = C.float().cpu().numpy()
    qb_o = qb_o.reshape(E, N, K)
    sb_o = sb_o.reshape(E, N, K // 32)
    rng = np.random.default_rng(30)
    for e in range(E):
        if counts[e] == 0:
            continue
        r0, r1 = int(offs_o[e]), int(offs_o[e + 1])
        m = r1 - r0
        pi = np.concatenate([[0, m - 1, min(255, m - 1), min(256, m - 1)], rng.integers(0, m, 300)])
        pj = rng.integers(0, N, pi.size)
        ref, bound, _ = oracle.gemm_sample(qa_o[r0:r1], qb_o[e], sa_o[r0:r1], sb_o[e], True, pi,
                                           pj, oracle.OUT_BF16, a_fmt=F4, b_fmt=F4)
        assert_within(Ch[r0 + pi, pj], ref, bound, f"MXFP4 grouped expert {e}")


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (129, 48, 128), (7, 264, 384)])
def test_e2m1_tiny_and_single_stage(M, N, K):
    """A single 128-wide K stage, one output row, N of one MMA width."""
    _gemm(F4, F4, True, M, N, K)
    _gemm(F4, 0, False, M, N, K)


def test_e2m1_grouped_zero_rows():
    """No routed rows at all: offsets all zero, nothing written, status OK."""
    E, N, K = 3, 128, 256
    qa = torch.zeros((1, K // 2), dtype=torch.uint8, device="cuda")
    qb = torch.zeros((E, N, K // 2), dtype=torch.uint8, device="cuda")
    sa = torch.ones((1, K // 32), device="cuda")
    sb = torch.ones((E, N, K // 32), device="cuda")
    C = torch.full((1, N), 5.0, dtype=torch.bfloat16, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    fp8g.fp8_grouped_gemm_fmt(qa, qb, sa, sb, C, 0, F4, F4, counts, E, N, K, 0, offs)
    assert fp8g.fp8_gemm_status()[0] == 0
    assert (offs.cpu().numpy() == 0).all()
    assert (C.float() == 5.0).all()


def test_mxfp4_pair_bias_relu_sampled():
    """The fused epilogue (per-column bias, ReLU) on the FP4-rate kernel."""
    M, N, K = 2304, 2560, 512
    assert fp8g.fp8g_gemm_plan(1, M, N, K)["BM"] == 256
    A = synth.normal((M, K), seed=51)
    B = synth.normal((N, K), seed=52)
    qa, sa, qa_o, sa_o = _quant(A, 32, F4)
    qb, sb, qb_o, sb_o = _quant(B, 32, F4)
    bias = np.random.default_rng(53).normal(0, 3, N).astype(np.float32)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled_ex(qa, qb, sa, sb, C, 0, F4, F4, torch.from_numpy(bias).cuda(),
                                 fp8g.FP8G_ACT_RELU, M, N, K)
    assert fp8g.fp8_gemm_status()[0] == 0
    rng = np.random.default_rng(54)
    pi = np.concatenate([[0, M - 1], rng.integers(0, M, 3000)])
    pj = np.concatenate([[N - 1, 0], rng.integers(0, N, 3000)])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, True, pi, pj, oracle.OUT_BF16,
                                       a_fmt=F4, b_fmt=F4, bias=bias, act_kind=oracle.ACT_RELU)
    assert_within(C.float().cpu().numpy()[pi, pj], ref, bound, "MXFP4 pairs bias + ReLU")
