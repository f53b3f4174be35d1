"""GPU parity of the FP6 operands E2M3 and E3M2, stored four codes per three
bytes (code i of a row in bits 6i .. 6i+5 of the row as a little-endian bit
string): the quantiser bit-exact against the oracle's codes packed the same
way (1x32 power-of-two scales: MXFP6; per-tensor; literal fp32 scales; fp32
and bf16 sources; row gather); the packing pinned through identity products
on either operand; GEMMs with FP6 on one or both sides, beside E4M3, E5M2
and E2M1, within the tolerance on the split-K, single-CTA, CTA-pair, grouped
and promotion kernels."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within

pytestmark = pytest.mark.gpu
E2M3, E3M2, F4 = fp8g.FP8G_E2M3, fp8g.FP8G_E3M2, fp8g.FP8G_E2M1


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def pack(codes: np.ndarray, fmt: int) -> np.ndarray:
    """One code per byte [r, c] -> the packed bytes of fmt."""
    c = codes.astype(np.uint32)
    if fmt == F4:
        return ((c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    if fmt not in (E2M3, E3M2):
        return codes.astype(np.uint8)
    v = (c[:, 0::4] & 0x3F) | ((c[:, 1::4] & 0x3F) << 6) | ((c[:, 2::4] & 0x3F) << 12) | \
        ((c[:, 3::4] & 0x3F) << 18)
    out = np.stack([v & 0xFF, (v >> 8) & 0xFF, (v >> 16) & 0xFF], axis=2)
    return out.reshape(codes.shape[0], -1).astype(np.uint8)


def table(fmt: int) -> np.ndarray:
    return {E2M3: oracle.fp6_table(E2M3), E3M2: oracle.fp6_table(E3M2), F4: oracle.e2m1_table(),
            1: oracle.e5m2_table()}.get(fmt, oracle.e4m3_table())


def _quant(x: torch.Tensor, block: int, fmt: int, rows_idx=None):
    """Quantise on both sides; the GPU's packed codes must equal the oracle's
    codes packed the same way, the scales bit for bit.  Returns the GPU codes
    and scales and the oracle's one-code-per-byte codes and scales."""
    x_rows, cols = x.shape
    n = x_rows if rows_idx is None else rows_idx.numel()
    q = torch.empty((n, fp8g.packed_cols(cols, fmt)), dtype=torch.uint8, device="cuda")
    s = torch.empty((n, cols // 32) if block else (1,), dtype=torch.float32, device="cuda")
    dt = fp8g.FP8G_IN_BF16 if x.dtype == torch.bfloat16 else fp8g.FP8G_IN_F32
    fp8g.fp8g_quantize_rows(x.cuda(), dt, x_rows, cols,
                            None if rows_idx is None else rows_idx.cuda(), n, block, fmt, q, s)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    xf = x.float().numpy() if rows_idx is None else x.float().numpy()[rows_idx.numpy()]
    if block:
        qo, so = oracle.quantize_block32(xf, fmt, literal=block == fp8g.FP8G_BLOCK32_LITERAL)
    else:
        qo, so = oracle.quantize_tensor(xf, fmt)
    want = pack(qo, fmt)
    qg = q.cpu().numpy()
    assert np.array_equal(qg, want), f"{int((qg != want).sum())} code byte mismatches"
    assert np.array_equal(s.cpu().numpy().reshape(so.shape).view(np.uint32), so.view(np.uint32))
    return q, s, qo, so


@pytest.mark.parametrize("fmt", [E2M3, E3M2])
@pytest.mark.parametrize("block", [0, 32, fp8g.FP8G_BLOCK32_LITERAL])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fp6_quantiser_bitexact(fmt, block, dtype):
    g = torch.Generator().manual_seed(block + fmt)
    x = torch.randn(96, 256, generator=g) * torch.exp(torch.randn(96, 1, generator=g) * 2)
    x[3, :32] = 0.0                                   # an all-zero block
    x[4, 7] = -1e-30                                  # rounds to -0
    x[7, 40:72] = torch.linspace(-0.3, 0.3, 32)       # subnormal codes under scale 1/4 .. 1
    if block != 0:
        x[5, 9] = float("nan")                        # largest positive code
        x[6, 1] = float("inf")
    _quant(x.to(dtype), block, fmt)


@pytest.mark.parametrize("fmt", [E2M3, E3M2])
def test_fp6_quantiser_gather_ragged(fmt):
    """Row gather + bf16 source + packed output; a row count that is no
    multiple of a tile and a row of 40 groups of 8 (240 bytes)."""
    g = torch.Generator().manual_seed(fmt + 70)
    x = (torch.randn(50, 320, generator=g) * 3).to(torch.bfloat16)
    rows = torch.tensor([49, 0, 7, 7, 31, 12, 3], dtype=torch.int32)
    _quant(x, 32, fmt, rows)


@pytest.mark.parametrize("fmt", [E2M3, E3M2])
@pytest.mark.parametrize("side", ["A", "B"])
def test_fp6_packed_layout_identity(fmt, side):
    """C = A I (or I B^T) with per-tensor scales 1 and the other operand the
    E4M3 identity (1.0 = 0x38): every output is one decoded FP6 value, exact in
    fp32.  Pins the packing and the 16U6 tile layout against the oracle's
    decode table, on the A and on the B operand."""
    M = N = K = 256
    rng = np.random.default_rng(11 + fmt)
    codes = rng.integers(0, 64, (M, K)).astype(np.uint8)
    P = torch.from_numpy(pack(codes, fmt)).cuda()
    I = torch.from_numpy((np.eye(N, K) * 0x38).astype(np.uint8)).cuda()
    one = torch.ones(1, device="cuda")
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    if side == "A":
        fp8g.fp8_gemm_fmt(P, I, one, one, C, fp8g.FP8G_OUT_F32, fmt, 0, M, N, K)
    else:
        fp8g.fp8_gemm_fmt(I, P, one, one, C, fp8g.FP8G_OUT_F32, 0, fmt, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    want = oracle.fp6_table(fmt)[codes].astype(np.float32)
    if side == "B":
        want = want.T
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
    what = f"FP6 {fa}x{fb} block={block} {M}x{N}x{K}"
    if sample is None:
        ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, block, oracle.OUT_BF16,
                                    a_fmt=fa, b_fmt=fb)
        assert_within(Ch, ref, bound, what)
    else:
        rng = np.random.default_rng(M)
        pi = np.concatenate([[0, M - 1, M - 1], rng.integers(0, M, sample)])
        pj = np.concatenate([[N - 1, 0, N - 1], rng.integers(0, N, sample)])
        ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, block, pi, pj,
                                           oracle.OUT_BF16, a_fmt=fa, b_fmt=fb)
        assert_within(Ch[pi, pj], ref, bound, what)


@pytest.mark.parametrize("fa,fb", [(E2M3, E2M3), (E3M2, E3M2), (E2M3, E3M2), (0, E3M2),
                                   (E3M2, F4), (E2M3, 1)])
@pytest.mark.parametrize("block", [False, True])
@pytest.mark.parametrize("M,N,K", [(300, 392, 256), (300, 392, 2048), (1536, 2048, 384)])
def test_fp6_gemm_full(fa, fb, block, M, N, K):
    _gemm(fa, fb, block, M, N, K)


@pytest.mark.parametrize("block", [False, True])
def test_fp6_gemm_pairs_sampled(block):
    assert fp8g.fp8g_gemm_plan(int(block), 4096, 4608, 512)["BM"] == 256
    _gemm(E2M3, E3M2, block, 4096, 4608, 512, sample=3000)


def test_fp6_grouped_ragged():
    """Grouped MoE GEMM with E2M3 activations and E3M2 expert weights (the
    3-D packed B map), ragged and empty experts."""
    counts = np.array([130, 0, 5, 257], np.int32)
    E, N, K = counts.size, 264, 256
    w = synth.small_grouped(counts, N, K, seed=43)
    qa, sa, qa_o, sa_o = _quant(w.A, 32, E2M3)
    qb, sb, qb_o, sb_o = _quant(w.B.reshape(E * N, K), 32, E3M2)
    rows = int(counts.sum())
    C = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm_fmt(qa, qb.reshape(E, N, 3 * K // 4), sa, sb.reshape(E, N, K // 32), C,
                              0, E2M3, E3M2, torch.from_numpy(counts).cuda(), E, N, K, rows)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    offs = oracle.grouped_offsets(counts)
    Ch = C.float().cpu().numpy()
    qb_o = qb_o.reshape(E, N, K)
    sb_o = sb_o.reshape(E, N, K // 32)
    for e in range(E):
        if counts[e] == 0:
            continue
        r0, r1 = offs[e], offs[e + 1]
        ref, bound, _ = oracle.gemm(qa_o[r0:r1], qb_o[e], sa_o[r0:r1], sb_o[e], True,
                                    oracle.OUT_BF16, a_fmt=E2M3, b_fmt=E3M2)
        assert_within(Ch[r0:r1], ref, bound, f"FP6 grouped expert {e}")


def test_fp6_promote_literal_scales():
    """E3M2 x E2M3 with literal fp32 1x32 scales (amax / 28, amax / 7.5)
    through the promotion kernel, with bias + GELU."""
    M, N, K = 260, 384, 512
    A = synth.normal((M, K), seed=93)
    B = synth.normal((N, K), seed=94)
    L = fp8g.FP8G_BLOCK32_LITERAL
    qa, sa, qa_o, sa_o = _quant(A, L, E3M2)
    qb, sb, qb_o, sb_o = _quant(B, L, E2M3)
    bias = np.random.default_rng(95).normal(0, 1, N).astype(np.float32)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled_promote(qa, qb, sa, sb, C, 0, E3M2, E2M3,
                                      torch.from_numpy(bias).cuda(), fp8g.FP8G_ACT_GELU, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle.OUT_BF16, a_fmt=E3M2,
                                b_fmt=E2M3, bias=bias, act_kind=oracle.ACT_GELU)
    assert_within(C.float().cpu().numpy(), ref, bound, "FP6 literal promote")


def test_fp6_grouped_pairs_sampled():
    """Grouped MoE GEMM on CTA pairs (the 3-D 16U6 map of B, expert-local
    256-row tiles) with E3M2 activations and E2M3 weights: empty, one-row and
    ragged experts; offsets and tile map bit-exact; sampled outputs per
    expert."""
    counts = np.array([3000, 0, 70, 9000, 257, 1, 0, 129], np.int32)
    E, N, K = counts.size, 2048, 512
    rows = int(counts.sum())
    plan = fp8g.fp8g_grouped_plan(N, K, rows, E)
    assert plan["BM"] == 256
    w = synth.small_grouped(counts, N, K, seed=31)
    qa, sa, qa_o, sa_o = _quant(w.A, 32, E3M2)
    qb, sb, qb_o, sb_o = _quant(w.B.reshape(E * N, K), 32, E2M3)
    C = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    tmap = torch.full((plan["max_tiles"], 4), -1, dtype=torch.int32, device="cuda")
    fp8g.fp8_grouped_gemm_fmt(qa, qb.reshape(E, N, 3 * K // 4), sa, sb.reshape(E, N, K // 32), C,
                              0, E3M2, E2M3, torch.from_numpy(counts).cuda(), E, N, K, rows, offs,
                              tmap)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    offs_o = oracle.grouped_offsets(counts)
    assert np.array_equal(offs.cpu().numpy(), offs_o)
    want = oracle.grouped_tile_map(counts, N, plan["BM"], plan["BN"], plan["G"])
    assert np.array_equal(tmap.cpu().numpy()[:want.shape[0]], want)
    Ch = C.float().cpu().numpy()
    qb_o = qb_o.reshape(E, N, K)
    sb_o = sb_o.reshape(E, N, K // 32)
    rng = np.random.default_rng(32)
    for e in range(E):
        if counts[e] == 0:
            continue
        r0, r1 = int(offs_o[e]), int(offs_o[e + 1])
        m = r1 - r0
        pi = np.concatenate([[0, m - 1, min(255, m - 1), min(256, m - 1)], rng.integers(0, m, 300)])
        pj = rng.integers(0, N, pi.size)
        ref, bound, _ = oracle.gemm_sample(qa_o[r0:r1], qb_o[e], sa_o[r0:r1], sb_o[e], True, pi,
                                           pj, oracle.OUT_BF16, a_fmt=E3M2, b_fmt=E2M3)
        assert_within(Ch[r0 + pi, pj], ref, bound, f"FP6 grouped pairs expert {e}")
