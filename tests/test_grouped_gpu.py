"""GPU parity of the grouped (MoE) block-scaled GEMM: outputs within the
tolerance, problem offsets and tile map bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_codes_equal, assert_within, quant_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def _quant_grouped(w):
    E, N, K = w.B.shape
    qa, sa, qa_o, sa_o = quant_both(w.A, 32)
    qb, sb, qb_o, sb_o = quant_both(w.B.reshape(E * N, K), 32)
    assert_codes_equal(qa, sa, qa_o, sa_o)
    assert_codes_equal(qb, sb, qb_o, sb_o)
    return (qa, sa, qb.reshape(E, N, K), sb.reshape(E, N, K // 32),
            qa_o, sa_o, qb_o.reshape(E, N, K), sb_o.reshape(E, N, K // 32))


def _run_grouped(qa, sa, qb, sb, counts, out="bf16"):
    E, N, K = qb.shape
    rows = int(counts.sum())
    plan = fp8g.fp8g_grouped_plan(N, K, rows, E)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = torch.full((max(rows, 1), N), float("nan"), dtype=dt, device="cuda")
    counts_d = torch.from_numpy(counts.astype(np.int32)).cuda()
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    tmap = torch.full((max(plan["max_tiles"], 1), 4), -1, dtype=torch.int32, device="cuda")
    o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
    fp8g.fp8_grouped_gemm(qa, qb, sa, sb, C, o, counts_d, E, N, K, rows, offs, tmap)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    return C[:rows].float().cpu().numpy(), offs.cpu().numpy(), tmap.cpu().numpy(), plan


@pytest.mark.parametrize("counts,N,K", [
    ([130, 0, 5, 257], 264, 256),
    ([1, 1, 4, 0, 0, 300, 2, 128], 512, 384),
    ([0, 0, 3], 136, 128),
    ([129], 256, 4160),
])
def test_grouped_small_full(counts, N, K):
    counts = np.array(counts, np.int32)
    w = synth.small_grouped(counts, N, K, seed=int(counts.sum()) + N)
    qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o = _quant_grouped(w)
    C, offs, tmap, plan = _run_grouped(qa, sa, qb, sb, counts)
    ref, bound, _ = oracle.grouped_gemm(qa_o, qb_o, sa_o, sb_o, counts, oracle.OUT_BF16)
    assert_within(C, ref, bound, f"grouped {counts.tolist()} N={N} K={K}")
    assert np.array_equal(offs, oracle.grouped_offsets(counts))
    want = oracle.grouped_tile_map(counts, N, plan["BM"], plan["BN"], plan["G"])
    assert np.array_equal(tmap[:want.shape[0]], want)
    assert (tmap[want.shape[0]:] == -1).all()


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_grouped_single_cta_several_tiles_per_cta(out):
    """128 x 128 tiles that convert their own scales, more tiles than SMs (so
    CTAs take two, the second one's scale windows converted while the first
    drains), a ragged N (4160 = 32.5 tiles), K of 9 steps (a window of 8 and
    one of 1) ending in a half K step (1120 = 8.75 x 128), and an expert of 3
    rows beside empty ones."""
    counts = np.array([3, 250, 0, 129], np.int32)
    N, K = 4160, 1120
    rows = int(counts.sum())
    plan = fp8g.fp8g_grouped_plan(N, K, rows, counts.size)
    assert plan["BM"] == 128 and plan["BN"] == 128
    tiles = int(sum(-(-c // 128) for c in counts)) * (-(-N // 128))
    assert tiles > torch.cuda.get_device_properties(0).multi_processor_count
    w = synth.small_grouped(counts, N, K, seed=41)
    qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o = _quant_grouped(w)
    C, offs, tmap, plan = _run_grouped(qa, sa, qb, sb, counts, out)
    ref, bound, _ = oracle.grouped_gemm(qa_o, qb_o, sa_o, sb_o, counts,
                                        oracle.OUT_BF16 if out == "bf16" else oracle.OUT_F32)
    assert_within(C, ref, bound, f"grouped single-CTA {counts.tolist()} N={N} K={K} {out}")
    assert np.array_equal(offs, oracle.grouped_offsets(counts))
    want = oracle.grouped_tile_map(counts, N, plan["BM"], plan["BN"], plan["G"])
    assert want.shape[0] == tiles
    assert np.array_equal(tmap[:tiles], want)


def test_grouped_single_cta_many_short_tiles():
    """64 experts of 0..20 rows (many empty), N = 2048, K = 256: about five
    tiles per CTA whose 2 K steps are fewer than the ring's stages, so every
    tile's scales go in one window and each drain follows the next tile's
    conversion."""
    rng = np.random.default_rng(47)
    counts = rng.integers(0, 21, 64).astype(np.int32)
    counts[rng.random(64) < 0.25] = 0
    N, K = 2048, 256
    rows = int(counts.sum())
    plan = fp8g.fp8g_grouped_plan(N, K, rows, counts.size)
    assert plan["BM"] == 128 and plan["BN"] == 128
    tiles = int((counts > 0).sum()) * (N // 128)
    assert tiles >= 4 * torch.cuda.get_device_properties(0).multi_processor_count
    w = synth.small_grouped(counts, N, K, seed=48)
    qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o = _quant_grouped(w)
    C, offs, tmap, plan = _run_grouped(qa, sa, qb, sb, counts)
    ref, bound, _ = oracle.grouped_gemm(qa_o, qb_o, sa_o, sb_o, counts, oracle.OUT_BF16)
    assert_within(C, ref, bound, "grouped single-CTA, 64 experts")
    assert np.array_equal(offs, oracle.grouped_offsets(counts))
    want = oracle.grouped_tile_map(counts, N, plan["BM"], plan["BN"], plan["G"])
    assert want.shape[0] == tiles
    assert np.array_equal(tmap[:tiles], want)


@pytest.mark.parametrize("where", ["A", "B_late"])
def test_grouped_single_cta_bad_scale_recorded(where):
    """A scale that is not a power of two, read by a single-CTA grouped tile,
    records FP8G_ERR_SCALE_FORMAT: in a routed row of A, or in B's last K
    step of an expert whose tiles come second on their CTAs."""
    counts = np.array([3, 250, 0, 129], np.int32)
    N, K = 4160, 1120
    rows = int(counts.sum())
    w = synth.small_grouped(counts, N, K, seed=43)
    qa, sa, qb, sb, _, _, _, _ = _quant_grouped(w)
    _run_grouped(qa, sa, qb, sb, counts)        # clean: status 0 (asserted there)
    if where == "A":
        sa = sa.clone()
        sa[2, 17] = 3.0                          # expert 0's last row
    else:
        sb = sb.clone()
        sb[3, N - 1, K // 32 - 1] = -0.5         # tiles 163, 164: second on CTAs 11, 12
    C = torch.empty((rows, N), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm(qa, qb, sa, sb, C, fp8g.FP8G_OUT_BF16,
                          torch.from_numpy(counts).cuda(), counts.size, N, K, rows)
    st, _ = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_ERR_SCALE_FORMAT
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_OK


def test_grouped_equals_per_expert_gemms():
    """The grouped GEMM equals one block-scaled GEMM per expert.  The single
    GEMMs of these small shapes run their own plan (one CTA per 128 x 128
    tile, scales converted in the kernel), so both are held to the oracle's
    bound: |grouped - single| <= 2 bound."""
    counts = np.array([200, 0, 77, 130], np.int32)
    N, K = 392, 512
    w = synth.small_grouped(counts, N, K, seed=3)
    qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o = _quant_grouped(w)
    C, _, _, _ = _run_grouped(qa, sa, qb, sb, counts)
    _, bound, _ = oracle.grouped_gemm(qa_o, qb_o, sa_o, sb_o, counts, oracle.OUT_BF16)
    off = 0
    for e, m in enumerate(counts.tolist()):
        if m == 0:
            continue
        Ce = torch.empty(m, N, dtype=torch.bfloat16, device="cuda")
        fp8g.fp8_gemm_blockscaled(qa[off:off + m], qb[e], sa[off:off + m], sb[e], Ce,
                                  fp8g.FP8G_OUT_BF16, m, N, K)
        d = np.abs(Ce.float().cpu().numpy().astype(np.float64) - C[off:off + m])
        assert (d <= 2 * bound[off:off + m]).all()
        off += m
    assert fp8g.fp8_gemm_status()[0] == 0


def test_grouped_pair_ragged_sampled():
    """Enough rows for 256 x 256 tiles on CTA pairs, with experts that are
    empty, one row, ragged against 128 and 256, and consecutive."""
    counts = np.array([3000, 0, 70, 9000, 257, 1, 0, 129], np.int32)
    N, K = 2048, 512
    rows = int(counts.sum())
    plan = fp8g.fp8g_grouped_plan(N, K, rows, counts.size)
    assert plan["BM"] == 256
    w = synth.small_grouped(counts, N, K, seed=23)
    qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o = _quant_grouped(w)
    C, offs, tmap, plan = _run_grouped(qa, sa, qb, sb, counts)
    assert np.array_equal(offs, oracle.grouped_offsets(counts))
    want = oracle.grouped_tile_map(counts, N, plan["BM"], plan["BN"], plan["G"])
    assert np.array_equal(tmap[:want.shape[0]], want)
    rng = np.random.default_rng(24)
    offs_o = oracle.grouped_offsets(counts)
    # every expert's first and last row, tile boundaries, plus random rows
    edge = [offs_o[e] for e in range(counts.size) if counts[e]] + \
           [offs_o[e + 1] - 1 for e in range(counts.size) if counts[e]] + \
           [offs_o[0] + 255, offs_o[0] + 256, offs_o[3] + 127, offs_o[3] + 128]
    pi = np.concatenate([np.array(edge), rng.integers(0, rows, 3000)]).astype(np.int64)
    pj = rng.integers(0, N, pi.size)
    expert = np.searchsorted(offs_o, pi, side="right") - 1
    got = C[pi, pj]
    ref = np.empty(pi.size, np.float32)
    bound = np.empty(pi.size, np.float64)
    for e in np.unique(expert):
        sel = np.flatnonzero(expert == e)
        r, b, _ = oracle.gemm_sample(qa_o, qb_o[e], sa_o, sb_o[e], True, pi[sel], pj[sel],
                                     oracle.OUT_BF16)
        ref[sel] = r
        bound[sel] = b
    assert_within(got, ref, bound, "grouped pair ragged")


def test_grouped_empty_expert_scales_not_read():
    """The weights of an expert without rows are not read: a malformed weight
    scale there changes nothing (no status, same outputs), while the same
    scale in an expert with rows records FP8G_ERR_SCALE_FORMAT."""
    counts = np.array([0, 200, 0, 70], np.int32)
    N, K = 256, 512
    w = synth.small_grouped(counts, N, K, seed=81)
    qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o = _quant_grouped(w)
    C0, _, _, _ = _run_grouped(qa, sa, qb, sb, counts)
    sb_bad = sb.clone()
    sb_bad[0, 5, 3] = 0.75       # not a power of two, in empty expert 0
    sb_bad[2, N - 1, 0] = -4.0   # negative, in empty expert 2
    C1, _, _, _ = _run_grouped(qa, sa, qb, sb_bad, counts)
    assert np.array_equal(C0, C1)
    sb_bad[1, 7, 1] = 0.75       # expert 1 has rows
    rows = int(counts.sum())
    C = torch.empty((rows, N), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm(qa, qb, sa, sb_bad, C, fp8g.FP8G_OUT_BF16,
                          torch.from_numpy(counts).cuda(), counts.size, N, K, rows)
    st, _ = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_ERR_SCALE_FORMAT
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_OK


def test_grouped_counts_mismatch_is_reported():
    counts = np.array([10, 20], np.int32)
    N, K = 128, 128
    qa = torch.zeros(31, K, dtype=torch.uint8, device="cuda")      # sum(counts) = 30 != 31
    qb = torch.zeros(2, N, K, dtype=torch.uint8, device="cuda")
    sa = torch.ones(31, K // 32, device="cuda")
    sb = torch.ones(2, N, K // 32, device="cuda")
    C = torch.full((31, N), 5.0, dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm(qa, qb, sa, sb, C, 0, torch.from_numpy(counts).cuda(), 2, N, K, 31)
    st, _ = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_ERR_INVALID_ARG
    assert (C.float() == 5.0).all()                                 # nothing written


def test_moe_full_size_sampled():
    """The MoE workload at full size (8 experts, N=14336, K=4096, 32768 routed
    rows with Zipf counts incl. empty experts): offsets and tile map bit-exact,
    4096 sampled outputs against the oracle."""
    w = synth.moe_grouped()
    counts = w.counts
    qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o = _quant_grouped(w)
    C, offs, tmap, plan = _run_grouped(qa, sa, qb, sb, counts)
    E, N, K = qb_o.shape
    assert np.array_equal(offs, oracle.grouped_offsets(counts))
    want = oracle.grouped_tile_map(counts, N, plan["BM"], plan["BN"], plan["G"])
    assert np.array_equal(tmap[:want.shape[0]], want)
    rng = np.random.default_rng(4)
    rows = int(counts.sum())
    pi = rng.integers(0, rows, 4096)
    pj = rng.integers(0, N, 4096)
    offs_o = oracle.grouped_offsets(counts)
    expert = np.searchsorted(offs_o, pi, side="right") - 1
    got = np.empty(pi.size, np.float32)
    ref = np.empty(pi.size, np.float32)
    bound = np.empty(pi.size, np.float64)
    for e in np.unique(expert):
        sel = np.flatnonzero(expert == e)
        r, b, _ = oracle.gemm_sample(qa_o, qb_o[e], sa_o, sb_o[e], True, pi[sel], pj[sel],
                                     oracle.OUT_BF16)
        ref[sel] = r
        bound[sel] = b
        got[sel] = C[pi[sel], pj[sel]]
    assert_within(got, ref, bound, "MoE sampled")
