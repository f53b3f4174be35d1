"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerance (per element): |C - C_ref| <= 2^-8 * sum_k |sA a_ik||sB b_jk| + 1 bf16
ulp(|C_ref|).  It covers fp32 accumulation in any order (K * 2^-24 << 2^-8 for
K <= 2^13) plus the output rounding.  Exact cases (identity / permutation /
exhaustive codes) are compared bit for bit; quantiser codes and scales are
always bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_codes_equal, assert_within, oracle_out, quant_both, run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    torch.cuda.init()
    yield


def _tensor_case(A, B, out):
    qa, sa, qa_o, sa_o = quant_both(A, 0)
    qb, sb, qb_o, sb_o = quant_both(B, 0)
    assert_codes_equal(qa, sa, qa_o, sa_o)
    assert_codes_equal(qb, sb, qb_o, sb_o)
    C = run_gemm(qa, sa, qb, sb, False, out)
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, False, oracle_out(out))
    return C, ref, bound


def _block_case(A, B, out):
    qa, sa, qa_o, sa_o = quant_both(A, 32)
    qb, sb, qb_o, sb_o = quant_both(B, 32)
    assert_codes_equal(qa, sa, qa_o, sa_o)
    assert_codes_equal(qb, sb, qb_o, sb_o)
    C = run_gemm(qa, sa, qb, sb, True, out)
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle_out(out))
    return C, ref, bound


# ---------------------------------------------------------------- quantiser
@pytest.mark.parametrize("rows,cols", [(256, 256), (300, 320), (1, 32), (7, 4096)])
def test_quantize_block32_bitexact(rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 3)
    if rows > 2 and cols >= 96:
        x[1, :32] = 0.0                                   # zero block
        x[2, 32:64] = 1e-40                               # subnormal block
        x[0, 5] = float("nan")
        x[0, 70] = float("inf")
        x[1, 40] = -0.0
    qg, sg, qo, so = quant_both(x, 32)
    assert_codes_equal(qg, sg, qo, so)


@pytest.mark.parametrize("rows,cols", [(256, 256), (100, 72), (3, 8)])
def test_quantize_tensor_bitexact(rows, cols):
    g = torch.Generator().manual_seed(rows * cols)
    x = torch.randn(rows, cols, generator=g) * 7
    x[0, 0] = float("nan")
    qg, sg, qo, so = quant_both(x, 0)
    assert_codes_equal(qg, sg, qo, so)


# --------------------------------------------------------------- per-tensor
def test_square256_bf16():
    w = synth.square_tensor(256, seed=0, out="bf16")
    C, ref, bound = _tensor_case(w.A, w.B, "bf16")
    assert_within(C, ref, bound, "256^3 per-tensor bf16")


def test_square1024_f32():
    w = synth.square_tensor(1024, seed=1, out="f32")
    C, ref, bound = _tensor_case(w.A, w.B, "f32")
    assert_within(C, ref, bound, "1024^3 per-tensor f32")


@pytest.mark.parametrize("kind", ["identity", "permutation"])
def test_exact_identity_permutation(kind):
    cases = synth.exact_cases(1024, seed=1)
    C, ref, _ = _tensor_case(cases["A"], cases[kind], "f32")
    assert np.array_equal(C.view(np.uint32), ref.view(np.uint32)), f"{kind}: not bit-exact"


@pytest.mark.parametrize("M,N,K,out", [(200, 264, 384, "bf16"), (1, 8, 16, "bf16"),
                                       (130, 520, 48, "f32"), (257, 8, 272, "bf16"),
                                       (129, 4, 1040, "f32")])
def test_tensor_ragged(M, N, K, out):
    A = synth.normal((M, K), seed=M)
    B = synth.normal((N, K), seed=N + 1000)
    C, ref, bound = _tensor_case(A, B, out)
    assert_within(C, ref, bound, f"per-tensor {M}x{N}x{K} {out}")


# ------------------------------------------------------------- block-scaled
def test_skinny_128x4096x4096_full():
    w = synth.skinny_block()
    C, ref, bound = _block_case(w.A, w.B, "bf16")
    assert_within(C, ref, bound, "skinny 128x4096x4096")


@pytest.mark.parametrize("M,N,K,out", [(300, 392, 320, "bf16"), (129, 136, 128, "f32"),
                                       (64, 1024, 4096, "bf16"), (1, 8, 32, "bf16"),
                                       (384, 512, 2048, "f32")])
def test_block_ragged(M, N, K, out):
    g = torch.Generator().manual_seed(M * 7 + N)
    A = synth.with_outliers(synth.normal((M, K), seed=M), g)
    B = synth.normal((N, K), seed=N) * torch.exp(torch.randn(N, 1, generator=g) * 2)
    C, ref, bound = _block_case(A, B, out)
    assert_within(C, ref, bound, f"block {M}x{N}x{K} {out}")


def test_block_exhaustive_codes_exact():
    """Every finite E4M3 code goes through the block-scaled MMA: A's rows hold
    all 254 finite codes (rotated per row), B = identity (code 1.0), scales 1."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    K = 256
    M = 128
    A = np.zeros((M, K), np.uint8)
    for i in range(M):
        A[i, :codes.size] = np.roll(codes, i)
    eye = np.zeros((K, K), np.uint8)
    eye[np.arange(K), np.arange(K)] = 0x38
    sfa = np.ones((M, K // 32), np.float32)
    sfb = np.ones((K, K // 32), np.float32)
    C = run_gemm(torch.from_numpy(A).cuda(), torch.from_numpy(sfa).cuda(),
                 torch.from_numpy(eye).cuda(), torch.from_numpy(sfb).cuda(), True, "f32")
    ref, _, _ = oracle.gemm(A, eye, sfa, sfb, True, oracle.OUT_F32)
    assert np.array_equal(C.view(np.uint32), ref.view(np.uint32))


def test_block_scale_layout_exact():
    """Distinct power-of-two scales per (row, K-block) on both operands with
    single-nonzero dot products make every output exact: any mix-up of the
    scale-factor layout (row, K-block, operand) changes a value."""
    M, N, K = 256, 512, 512
    rng = np.random.default_rng(5)
    A = np.zeros((M, K), np.uint8)
    B = np.zeros((N, K), np.uint8)
    ka = rng.integers(0, K, size=M)
    A[np.arange(M), ka] = rng.integers(0x30, 0x50, size=M)
    # B row j has one nonzero, at the K position of A row (j % M)
    B[np.arange(N), ka[np.arange(N) % M]] = rng.integers(0x30, 0x50, size=N)
    sfa = (2.0 ** rng.integers(-20, 20, size=(M, K // 32))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-20, 20, size=(N, K // 32))).astype(np.float32)
    C = run_gemm(torch.from_numpy(A).cuda(), torch.from_numpy(sfa).cuda(),
                 torch.from_numpy(B).cuda(), torch.from_numpy(sfb).cuda(), True, "f32")
    ref, _, _ = oracle.gemm(A, B, sfa, sfb, True, oracle.OUT_F32)
    assert np.array_equal(C.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("n", [4096, 8192])
def test_large_block_sampled(n):
    """Full-size large block-scaled GEMM, run exactly as the bench runs it;
    2048 sampled outputs (plus the four corners) against the oracle."""
    w = synth.large_block(n, seed=3)
    C, qa_o, sa_o, qb_o, sb_o = _block_full(w)
    rng = np.random.default_rng(n)
    pi = np.concatenate([rng.integers(0, n, 2048), [0, 0, n - 1, n - 1]])
    pj = np.concatenate([rng.integers(0, n, 2048), [0, n - 1, 0, n - 1]])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, True, pi, pj, oracle.OUT_BF16)
    assert_within(C[pi, pj], ref, bound, f"{n}^3 block sampled")


def _block_full(w):
    qa, sa, qa_o, sa_o = quant_both(w.A, 32)
    qb, sb, qb_o, sb_o = quant_both(w.B, 32)
    assert_codes_equal(qa, sa, qa_o, sa_o)
    assert_codes_equal(qb, sb, qb_o, sb_o)
    C = run_gemm(qa, sa, qb, sb, True, w.out)
    return C, qa_o, sa_o, qb_o, sb_o


# ------------------------------------------------------------------- errors
@pytest.mark.parametrize("M,N,K,bad_b,path", [
    (256, 256, 256, False, "inline"),    # single CTAs, in-kernel check
    (200, 392, 320, True, "inline"),     # single CTAs, K/32 odd
    (256, 256, 2048, False, "split"),    # split-K: in-kernel check
    (200, 392, 2080, True, "split"),     # split-K, K/32 odd
    (2048, 2048, 256, True, "pack")])    # packing kernel's check
def test_scale_format_error_recorded(M, N, K, bad_b, path):
    qa = torch.zeros(M, K, dtype=torch.uint8, device="cuda")
    qb = torch.zeros(N, K, dtype=torch.uint8, device="cuda")
    sfa = torch.ones(M, K // 32, device="cuda")
    sfb = torch.ones(N, K // 32, device="cuda")
    if bad_b:
        sfb[N - 1, K // 32 - 1] = -2.0                # negative
    else:
        sfa[3, 2] = 0.75                              # not a power of two
    plan = fp8g.fp8g_gemm_plan(1, M, N, K)
    few = plan["BM"] == 128 and plan["BN"] == 128  # one CTA per 128 x 128 tile: scales inline
    assert path == ("split" if plan["split_k"] > 1 else "inline" if few else "pack"), plan
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled(qa, qb, sfa, sfb, C, fp8g.FP8G_OUT_BF16, M, N, K)
    st, _ = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_ERR_SCALE_FORMAT
    st, _ = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_OK                         # read clears


def test_host_checks_reject_without_launch():
    qa = torch.zeros(128, 64, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, device="cuda")
    C = torch.empty(128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm(qa, qa, s, s, C, 0, 128, 128, 40)        # K % 16 != 0
    assert e.value.status == fp8g.FP8G_ERR_ALIGNMENT
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm(qa.data_ptr() + 1, qa, s, s, C, 0, 128, 128, 64)
    assert e.value.status == fp8g.FP8G_ERR_ALIGNMENT
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm_blockscaled(qa, qa, s, s, C, 0, 128, 128, 48)  # K % 32 != 0
    assert e.value.status == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_OK


def test_plan_reports_tiles():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = fp8g.fp8g_gemm_plan(1, 8192, 8192, 8192)
    assert p["BM"] in (128, 256) and p["BN"] in (128, 256) and p["G"] == 16 and p["split_k"] == 1
    assert 1 <= p["grid"] <= sms
    s = fp8g.fp8g_gemm_plan(1, 128, 4096, 4096)          # few tiles: K split over a cluster
    assert 2 <= s["split_k"] <= 8 and s["grid"] % s["split_k"] == 0 and s["grid"] <= sms
    assert s["BN"] * (s["grid"] // s["split_k"]) >= 4096


@pytest.mark.parametrize("K", [128, 256, 384, 1024, 2048, 2080, 2432, 4096])
def test_few_tiles_split_k_or_single_cta(K):
    """Few tiles: from 16 K steps K is split over a cluster (ragged K-block
    counts per rank: 17 and 19 steps over 4); below, one CTA per 128 x 128
    tile (block-scaled: scales converted in the kernel, no packing)."""
    M, N = 130, 392
    g = torch.Generator().manual_seed(K)
    A = synth.normal((M, K), seed=K)
    B = synth.normal((N, K), seed=K + 1) * torch.exp(torch.randn(N, 1, generator=g))
    steps = -(-K // 128)
    for block in (0, 1):
        plan = fp8g.fp8g_gemm_plan(block, M, N, K)
        if steps >= 16:
            assert plan["split_k"] >= 2, plan
        else:
            assert plan["split_k"] == 1 and plan["BM"] == 128 and plan["BN"] == 128, plan
    C, ref, bound = _block_case(A, B, "bf16")
    assert_within(C, ref, bound, f"few tiles block {M}x{N}x{K}")
    C, ref, bound = _tensor_case(A, B, "f32")
    assert_within(C, ref, bound, f"few tiles per-tensor {M}x{N}x{K}")


def test_split_k_clusters_all_resident():
    """M=128, N=4864: 38 tiles of 128 x 128.  Clusters of four would need 38
    co-resident clusters; GB300 holds 36 of this kernel's four-CTA clusters
    (a cluster stays inside one GPC), so the plan takes 38 pairs (76 CTAs)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 128, 4864, 4096
    p = fp8g.fp8g_gemm_plan(1, M, N, K)
    if sms == 152:
        assert p["split_k"] == 2 and p["grid"] == 76
    A = synth.normal((M, K), seed=48)
    B = synth.normal((N, K), seed=49)
    qa, sa, qa_o, sa_o = quant_both(A, 32)
    qb, sb, qb_o, sb_o = quant_both(B, 32)
    C = run_gemm(qa, sa, qb, sb, True, "bf16")
    rng = np.random.default_rng(48)
    pi = rng.integers(0, M, 3000)
    pj = rng.integers(0, N, 3000)
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, True, pi, pj, oracle.OUT_BF16)
    assert_within(C[pi, pj], ref, bound, "split-K 128x4864x4096")


# ------------------------------------------------- per-tensor on CTA pairs
def test_tensor_pair_chosen_for_large():
    p = fp8g.fp8g_gemm_plan(0, 4096, 4608, 512)
    assert p["BM"] == 256 and p["BN"] == 256 and p["split_k"] == 1 and p["grid"] % 2 == 0


def test_tensor_pair_sampled():
    M, N, K = 4096, 4608, 512
    A = synth.normal((M, K), seed=41)
    B = synth.normal((N, K), seed=42) * 3
    qa, sa, qa_o, sa_o = quant_both(A, 0)
    qb, sb, qb_o, sb_o = quant_both(B, 0)
    assert_codes_equal(qa, sa, qa_o, sa_o)
    assert_codes_equal(qb, sb, qb_o, sb_o)
    C = run_gemm(qa, sa, qb, sb, False, "bf16")
    rng = np.random.default_rng(7)
    pi = np.concatenate([rng.integers(0, M, 4096), [0, 255, 256, M - 1, 127, 128]])
    pj = np.concatenate([rng.integers(0, N, 4096), [N - 1, 0, 255, 256, 4607, 4352]])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, False, pi, pj, oracle.OUT_BF16)
    assert_within(C[pi, pj], ref, bound, "pair per-tensor sampled")


def test_tensor_pair_ragged_full():
    M, N, K = 2000, 3000, 640           # partial 256-row and 256-column pair tiles
    assert fp8g.fp8g_gemm_plan(0, M, N, K)["BM"] == 256
    A = synth.normal((M, K), seed=43)
    B = synth.normal((N, K), seed=44)
    C, ref, bound = _tensor_case(A, B, "f32")
    assert_within(C, ref, bound, "pair per-tensor ragged")


@pytest.mark.parametrize("kind", ["identity", "permutation"])
def test_tensor_pair_exact(kind):
    n = 4096
    A = synth.normal((n, n), seed=45)
    B = synth.identity(n) if kind == "identity" else synth.permutation_matrix(n, 46)
    qa, sa, qa_o, sa_o = quant_both(A, 0)
    qb, sb, qb_o, sb_o = quant_both(B, 0)
    assert_codes_equal(qb, sb, qb_o, sb_o)
    C = run_gemm(qa, sa, qb, sb, False, "f32")
    rng = np.random.default_rng(8)
    pi = rng.integers(0, n, 8192)
    pj = rng.integers(0, n, 8192)
    if kind == "permutation":
        # include the nonzero entry of sampled rows: B[j, pi(j)] = 1
        perm = np.argmax(qb_o.reshape(n, n) != 0, axis=1)
        pj[::2] = np.argsort(perm)[rng.integers(0, n, 4096)]
    ref, _, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, False, pi, pj, oracle.OUT_F32)
    got = C[pi, pj]
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"{kind}: not bit-exact"


def test_block_pair_scale_layout_exact():
    """Block-scaled GEMM large enough for CTA pairs: distinct power-of-two
    scales per (row, K block) on both operands and single-product outputs make
    every sampled value exact, so any mix-up of which CTA holds which scale
    rows changes a value."""
    n, K = 4096, 256
    assert fp8g.fp8g_gemm_plan(1, n, n, K)["BM"] == 256
    rng = np.random.default_rng(17)
    ka = rng.integers(0, K, size=n)
    A = np.zeros((n, K), np.uint8)
    B = np.zeros((n, K), np.uint8)
    A[np.arange(n), ka] = rng.integers(0x30, 0x50, size=n)
    perm = rng.permutation(n)
    B[np.arange(n), ka[perm]] = rng.integers(0x30, 0x50, size=n)   # B row j pairs with A row perm[j]
    sfa = (2.0 ** rng.integers(-20, 20, size=(n, K // 32))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-20, 20, size=(n, K // 32))).astype(np.float32)
    C = run_gemm(torch.from_numpy(A).cuda(), torch.from_numpy(sfa).cuda(),
                 torch.from_numpy(B).cuda(), torch.from_numpy(sfb).cuda(), True, "f32")
    pj = np.concatenate([np.arange(n), rng.integers(0, n, 4096)])
    pi = np.concatenate([perm, rng.integers(0, n, 4096)])
    ref, _, _ = oracle.gemm_sample(A, B, sfa, sfb, True, pi, pj, oracle.OUT_F32)
    got = C[pi, pj]
    bad = np.flatnonzero(got.view(np.uint32) != ref.view(np.uint32))
    assert bad.size == 0, f"{bad.size} mismatches, e.g. {[(pi[b], pj[b], got[b], ref[b]) for b in bad[:4]]}"


def test_block_pair_bf16_ragged_edges():
    """bf16 output of the block-scaled CTA-pair kernel with ragged M and N:
    the last tile's columns 2368.. lie past N = 2368, and the odd CTA of the
    last row of tiles starts at row 2432, past M = 2404.  Every element within
    the tolerance, and the rows after C untouched."""
    M, N, K = 2404, 2368, 512
    assert fp8g.fp8g_gemm_plan(1, M, N, K)["BM"] == 256
    A = synth.normal((M, K), seed=91)
    B = synth.normal((N, K), seed=92)
    qa, sa, qa_o, sa_o = quant_both(A, 32)
    qb, sb, qb_o, sb_o = quant_both(B, 32)
    C_big = torch.full((M + 8, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = C_big[:M]
    fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C, fp8g.FP8G_OUT_BF16, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle.OUT_BF16)
    assert_within(C.float().cpu().numpy(), ref, bound, "pair bf16, ragged edges")
    assert torch.isnan(C_big[M:].float()).all()


def test_block_single_cta_256_tiles():
    """A block-scaled shape with between half a wave and a wave of 128x256
    tiles runs on single CTAs with 256-wide tiles (no split, no pair)."""
    M, N, K = 2048, 2048 - 8, 1024
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = fp8g.fp8g_gemm_plan(1, M, N, K)
    assert plan["BM"] == 128 and plan["BN"] == 256 and plan["split_k"] == 1, (plan, sms)
    g = torch.Generator().manual_seed(9)
    A = synth.with_outliers(synth.normal((M, K), seed=51), g)
    B = synth.normal((N, K), seed=52) * torch.exp(torch.randn(N, 1, generator=g))
    qa, sa, qa_o, sa_o = quant_both(A, 32)
    qb, sb, qb_o, sb_o = quant_both(B, 32)
    assert_codes_equal(qa, sa, qa_o, sa_o)
    assert_codes_equal(qb, sb, qb_o, sb_o)
    C = run_gemm(qa, sa, qb, sb, True, "bf16")
    rng = np.random.default_rng(10)
    pi = np.concatenate([rng.integers(0, M, 4096), [0, M - 1, 127, 128]])
    pj = np.concatenate([rng.integers(0, N, 4096), [N - 1, 0, 255, 256]])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, True, pi, pj, oracle.OUT_BF16)
    assert_within(C[pi, pj], ref, bound, "block single-CTA 256-wide")


def test_kernel_timing_hook():
    """The library's kernel timing records one duration per GEMM call, each
    shorter than the whole call (which also packs the scales)."""
    M = N = K = 2048
    A = synth.normal((M, K), seed=71)
    B = synth.normal((N, K), seed=72)
    qa, sa, _, _ = quant_both(A, 32)
    qb, sb, _, _ = quant_both(B, 32)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    fp8g.fp8g_kernel_timing_begin(4)
    with pytest.raises(fp8g.Fp8gError):
        fp8g.fp8g_kernel_timing_begin(4)                 # already recording
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(6):
        fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C, 0, M, N, K)
    e1.record()
    torch.cuda.synchronize()
    ms = fp8g.fp8g_kernel_timing_end(8)
    assert len(ms) == 4 and all(0 < t for t in ms)
    assert sum(ms) < e0.elapsed_time(e1)
    assert fp8g.fp8_gemm_status()[0] == 0
    with pytest.raises(fp8g.Fp8gError):
        fp8g.fp8g_kernel_timing_end(1)                   # not recording
