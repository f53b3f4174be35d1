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


# ---------------------------------------------------------------- grouped
# Expert e's rows of A times its own weight B[e], each B[e] quantised on its
# own (its own tensor scale gB[e]); A shares one tensor scale.  256 x 256
# tiles on CTA pairs for every shape, rastered in bands of 16 row tiles.

def _grouped(counts, N, K, seed, out="bf16", bias=False, act=0, sample=None):
    counts = np.asarray(counts, np.int32)
    E, rows = counts.size, int(counts.sum())
    w = synth.small_grouped(counts, N, K, seed=seed)
    (qa, sa, ga), (qa_o, sa_o, ga_o) = _quant(w.A)
    qbs, sbs, gbs, qb_o, sb_o, gb_o = [], [], [], [], [], []
    for e in range(E):
        # experts an order of magnitude apart: distinct tensor scales
        (q, s, g), (qo, so, go) = _quant(w.B[e] * float(4.0 ** (e % 3)))
        qbs.append(q), sbs.append(s), gbs.append(g), qb_o.append(qo), sb_o.append(so), gb_o.append(go)
    assert len({float(g) for g in gb_o}) > 1 or E == 1
    qb, sb, gb = torch.stack(qbs), torch.stack(sbs), torch.cat(gbs)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
    bias_v = np.random.default_rng(seed).normal(0, 2, (E, N)).astype(np.float32) if bias else None
    C = torch.full((rows, N), float("nan"), dtype=dt, device="cuda")
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    npn = (N + 255) // 256
    tmap = torch.full(((rows // 256 + E) * npn, 4), -1, dtype=torch.int32, device="cuda")
    fp8g.fp8_grouped_gemm_nvfp4(qa, qb, sa, sb, ga, gb, C, o,
                                torch.from_numpy(bias_v).cuda() if bias else None, act,
                                torch.from_numpy(counts).cuda(), E, N, K, rows, offs, tmap)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    offs_o = oracle.grouped_offsets(counts)
    assert np.array_equal(offs.cpu().numpy(), offs_o)
    want = oracle.grouped_tile_map(counts, N, 256, 256, 16)
    tm = tmap.cpu().numpy()
    assert np.array_equal(tm[:want.shape[0]], want) and (tm[want.shape[0]:] == -1).all()
    Ch = C.float().cpu().numpy()
    ok = oracle.OUT_BF16 if out == "bf16" else oracle.OUT_F32
    rng = np.random.default_rng(seed + 1)
    for e in range(E):
        if counts[e] == 0:
            continue
        r0, r1 = int(offs_o[e]), int(offs_o[e + 1])
        be = bias_v[e] if bias else None
        if sample is None:
            ref, bound, _ = oracle.gemm_nvfp4(qa_o[r0:r1], qb_o[e], sa_o[r0:r1], sb_o[e], ga_o,
                                              gb_o[e], ok, bias=be, act_kind=act)
            assert_within(Ch[r0:r1], ref, bound, f"NVFP4 grouped expert {e}")
            continue
        m = r1 - r0
        pi = np.concatenate([[0, m - 1, min(255, m - 1), min(256, m - 1)], rng.integers(0, m, sample)])
        pj = np.concatenate([[N - 1, 0, N - 1, 0], rng.integers(0, N, sample)])
        ref, bound, _ = oracle.gemm_nvfp4_sample(qa_o[r0:r1], qb_o[e], sa_o[r0:r1], sb_o[e], ga_o,
                                                 gb_o[e], pi, pj, ok, bias=be, act_kind=act)
        assert_within(Ch[r0 + pi, pj], ref, bound, f"NVFP4 grouped expert {e} sampled")


def test_nvfp4_grouped_ragged_full():
    """Empty, one-row and ragged experts, N past a 256 column tile; every
    output against the oracle."""
    _grouped([300, 0, 7, 1, 520, 256], 392, 512, seed=51)


def test_nvfp4_grouped_bias_relu_f32_full():
    _grouped([129, 640, 0, 33], 264, 768, seed=53, out="f32", bias=True, act=fp8g.FP8G_ACT_RELU)


def test_nvfp4_grouped_many_tiles_sampled():
    """More tiles than CTA pairs (persistent loop over experts)."""
    _grouped([3000, 0, 70, 9000, 257, 1, 0, 129], 2048, 512, seed=55, sample=300)


def test_nvfp4_grouped_zero_rows_and_bad_counts():
    """total_rows = 0: offsets all zero, no tile, nothing stored; counts that
    do not sum to total_rows: FP8G_ERR_INVALID_ARG through the status word and
    no tile runs."""
    E, N, K = 3, 256, 256
    B = torch.zeros((E, N, K // 2), dtype=torch.uint8, device="cuda")
    sb = torch.full((E, N, K // 16), 0x38, dtype=torch.uint8, device="cuda")
    sa = torch.full((1, K // 16), 0x38, dtype=torch.uint8, device="cuda")
    g = torch.ones(E, device="cuda")
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    tmap = torch.full((E, 4), -1, dtype=torch.int32, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    fp8g.fp8_grouped_gemm_nvfp4(None, B, sa, sb, g, g, None, fp8g.FP8G_OUT_BF16, None, 0, counts,
                                E, N, K, 0, offs, tmap)
    assert fp8g.fp8_gemm_status()[0] == 0
    assert (offs.cpu().numpy() == 0).all() and (tmap.cpu().numpy() == -1).all()
    A = torch.zeros((64, K // 2), dtype=torch.uint8, device="cuda")
    sa = torch.full((64, K // 16), 0x38, dtype=torch.uint8, device="cuda")
    C = torch.full((64, N), 3.0, dtype=torch.bfloat16, device="cuda")
    bad = torch.tensor([10, 20, 30], dtype=torch.int32, device="cuda")   # sums to 60, not 64
    fp8g.fp8_grouped_gemm_nvfp4(A, B, sa, sb, g, g, C, fp8g.FP8G_OUT_BF16, None, 0, bad, E, N, K,
                                64, None, None)
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_ERR_INVALID_ARG
    assert (C.float() == 3.0).all().item()
