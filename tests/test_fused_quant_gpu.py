"""fp8_grouped_gemm_quant: the grouped (MoE) GEMM from fp32 / bf16 token
activations.  With FP8G_QUANT_FUSED the 1x32 E4M3 quantisation of the routed
rows runs inside the GEMM kernel when the plan runs single-CTA tiles (few
routed rows); otherwise, and by default, as a gather-quantise pass before the
GEMM.

Parity: the codes and scales the call reports are bit-exact against the
oracle's quantiser on the gathered rows; the outputs are within the
block-scaled tolerance of the oracle's GEMM of those codes, per expert; and
they equal, bit for bit, the two-call path (fp8g_quantize_rows, then
fp8_grouped_gemm_scatter), which runs the same GEMM on the same codes."""
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


def _route(T, E, seed):
    """Top-2 routing (two distinct experts per token, Zipf-skewed), rows in
    expert order: (counts, token of each routed row, row of C = 2 t + slot)."""
    rng = np.random.default_rng(seed)
    w = rng.zipf(1.5, size=E).astype(np.float64)
    p = w / w.sum()
    pairs = np.array([rng.choice(E, 2, replace=False, p=p) for _ in range(T)])
    rows = sorted((pairs[t, s], t, s) for t in range(T) for s in range(2))
    counts = np.bincount([r[0] for r in rows], minlength=E).astype(np.int32)
    tok = np.array([r[1] for r in rows], np.int32)
    crow = np.array([2 * r[1] + r[2] for r in rows], np.int32)
    return counts, tok, crow


def _weights(E, N, K, seed):
    B = synth.normal((E, N, K), seed=seed, std=0.02)
    qb, sb = fp8g.quantize(B.reshape(E * N, K).cuda(), 32)
    qb_o, sb_o = oracle.quantize_block32(B.reshape(E * N, K).numpy())
    assert np.array_equal(qb.cpu().numpy(), qb_o)
    assert np.array_equal(sb.cpu().numpy().reshape(sb_o.shape).view(np.uint32), sb_o.view(np.uint32))
    return (qb.reshape(E, N, K), sb.reshape(E, N, K // 32), qb_o.reshape(E, N, K),
            sb_o.reshape(E, N, K // 32))


def _fused(X, tok, qb, sb, counts, N, K, crow=None, c_rows=0, bias=None, act=0, copies=True,
           out=fp8g.FP8G_OUT_BF16, flags=fp8g.FP8G_QUANT_FUSED):
    E = counts.size
    rows = int(counts.sum())
    dt = fp8g.FP8G_IN_BF16 if X.dtype == torch.bfloat16 else fp8g.FP8G_IN_F32
    C = torch.full((c_rows if crow is not None else rows, N), float("nan"),
                   dtype=torch.bfloat16 if out == fp8g.FP8G_OUT_BF16 else torch.float32,
                   device="cuda")
    qa = torch.full((rows, K), 0xEE, dtype=torch.uint8, device="cuda") if copies else None
    sa = torch.full((rows, K // 32), -1.0, device="cuda") if copies else None
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    plan = fp8g.fp8g_grouped_plan(N, K, rows, E)
    tmap = torch.full((4 * plan["max_tiles"],), -1, dtype=torch.int32, device="cuda")
    fp8g.fp8_grouped_gemm_quant(X.cuda(), dt, X.shape[0], torch.from_numpy(tok).cuda(), qb, sb, C,
                                out, fp8g.FP8G_E4M3,
                                None if bias is None else torch.from_numpy(bias).cuda(), act,
                                torch.from_numpy(counts).cuda(), E, N, K, rows,
                                None if crow is None else torch.from_numpy(crow).cuda(), c_rows,
                                qa, sa, offs, tmap, flags)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    return C, qa, sa, offs.cpu().numpy(), tmap.cpu().numpy(), plan


def _two_calls(X, tok, qb, sb, counts, N, K, crow=None, c_rows=0, bias=None, act=0):
    E = counts.size
    rows = int(counts.sum())
    dt = fp8g.FP8G_IN_BF16 if X.dtype == torch.bfloat16 else fp8g.FP8G_IN_F32
    qa = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    sa = torch.empty((rows, K // 32), device="cuda")
    fp8g.fp8g_quantize_rows(X.cuda(), dt, X.shape[0], K, torch.from_numpy(tok).cuda(), rows, 32,
                            fp8g.FP8G_E4M3, qa, sa)
    C = torch.full((c_rows if crow is not None else rows, N), float("nan"),
                   dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm_scatter(qa, qb, sa, sb, C, 0, 0, 0,
                                  None if bias is None else torch.from_numpy(bias).cuda(), act,
                                  torch.from_numpy(counts).cuda(), E, N, K, rows,
                                  None if crow is None else torch.from_numpy(crow).cuda(),
                                  c_rows if crow is not None else rows)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    return C


def _oracle_codes(X, tok):
    return oracle.quantize_block32(X.float().numpy()[tok])       # bf16 -> fp32 is exact


def _check_codes(qa, sa, qo, so):
    q = qa.cpu().numpy()
    assert np.array_equal(q, qo), f"{int((q != qo).sum())} code mismatches"
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), so.view(np.uint32)), "scale mismatch"


def _oracle_out(qo, so, qb_o, sb_o, counts, crow, c_rows, bias, act):
    N = qb_o.shape[1]
    offs = oracle.grouped_offsets(counts)
    ref = np.zeros((c_rows, N), np.float32)
    bound = np.zeros((c_rows, N), np.float64)
    for e in range(counts.size):
        a, b = offs[e], offs[e + 1]
        if a == b:
            continue
        r, bd, _ = oracle.gemm(qo[a:b], qb_o[e], so[a:b], sb_o[e], True, oracle.OUT_BF16,
                               bias=None if bias is None else bias[e], act_kind=act)
        ref[crow[a:b]] = r
        bound[crow[a:b]] = bd
    return ref, bound


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_fused_quantiser_full(dtype):
    """Few routed rows (single-CTA plan, so the quantisation runs inside the
    GEMM): ragged experts, bias + ReLU, scatter to (token, slot) rows."""
    T, E, N, K = 300, 4, 768, 544           # K: four full 128-wide steps and a 32-wide tail
    counts, tok, crow = _route(T, E, seed=31)
    rows = int(counts.sum())
    g = torch.Generator().manual_seed(32)
    X = torch.randn(T, K, generator=g) * torch.exp(torch.randn(T, 1, generator=g) * 2)
    X[3, :32] = 0.0                          # an all-zero block: scale 1, codes 0
    X[5, 40] = 1e4                           # one outlier sets its block's scale
    X = X.to(dtype)
    qb, sb, qb_o, sb_o = _weights(E, N, K, seed=33)
    bias = np.random.default_rng(34).normal(size=(E, N)).astype(np.float32)
    assert fp8g.fp8g_grouped_plan(N, K, rows, E)["BM"] == 128
    C, qa, sa, offs, tmap, plan = _fused(X, tok, qb, sb, counts, N, K, crow, 2 * T, bias,
                                         fp8g.FP8G_ACT_RELU)
    qo, so = _oracle_codes(X, tok)
    _check_codes(qa, sa, qo, so)
    assert np.array_equal(offs, oracle.grouped_offsets(counts))
    want = oracle.grouped_tile_map(counts, N, plan["BM"], plan["BN"], plan["G"])
    assert np.array_equal(tmap[:want.size], want.reshape(-1))
    ref, bound = _oracle_out(qo, so, qb_o, sb_o, counts, crow, 2 * T, bias, oracle.ACT_RELU)
    x = C.float().cpu().numpy()
    assert_within(x, ref, bound, f"fused quantiser {dtype}")
    two = _two_calls(X, tok, qb, sb, counts, N, K, crow, 2 * T, bias, fp8g.FP8G_ACT_RELU)
    assert np.array_equal(x.view(np.uint32), two.float().cpu().numpy().view(np.uint32))
    # no copies asked for, and the default two-kernel path: the same bits
    for copies, flags in ((False, fp8g.FP8G_QUANT_FUSED), (True, 0), (False, 0)):
        C2 = _fused(X, tok, qb, sb, counts, N, K, crow, 2 * T, bias, fp8g.FP8G_ACT_RELU,
                    copies=copies, flags=flags)[0]
        assert torch.equal(C2.view(torch.int16), C.view(torch.int16)), (copies, flags)


def test_fused_entry_with_many_rows_takes_two_passes():
    """Enough routed rows for 256-row tiles on CTA pairs: the call quantises in
    a pass of its own, then runs the pair GEMM; same codes, same bits as the
    two calls, sampled outputs against the oracle."""
    T, E, N, K = 4096, 2, 1024, 512
    counts, tok, crow = _route(T, E, seed=41)
    rows = int(counts.sum())
    assert fp8g.fp8g_grouped_plan(N, K, rows, E)["BM"] == 256
    X = synth.normal((T, K), seed=42).to(torch.bfloat16)
    qb, sb, qb_o, sb_o = _weights(E, N, K, seed=43)
    C, qa, sa, _, _, _ = _fused(X, tok, qb, sb, counts, N, K)
    qo, so = _oracle_codes(X, tok)
    _check_codes(qa, sa, qo, so)
    two = _two_calls(X, tok, qb, sb, counts, N, K)
    assert torch.equal(C.view(torch.int16), two.view(torch.int16))
    C3 = _fused(X, tok, qb, sb, counts, N, K, copies=False)[0]       # pool temporary
    assert torch.equal(C3.view(torch.int16), C.view(torch.int16))
    rng = np.random.default_rng(44)
    pi = rng.integers(0, rows, 2048)
    pj = rng.integers(0, N, 2048)
    offs = oracle.grouped_offsets(counts)
    expert = np.searchsorted(offs, pi, side="right") - 1
    x = C.float().cpu().numpy()
    for e in np.unique(expert):
        sel = np.flatnonzero(expert == e)
        r, b, _ = oracle.gemm_sample(qo, qb_o[e], so, sb_o[e], True, pi[sel], pj[sel],
                                     oracle.OUT_BF16)
        assert_within(x[pi[sel], pj[sel]], r, b, f"two-pass expert {e}")


def test_fused_decode_moe_full_size_sampled():
    """The decode-shaped MoE at full expert size: 8 experts of [14336, 4096],
    128 tokens routed top-2 (256 rows, Zipf counts) from bf16 activations, the
    launch the bench times (single-CTA plan, fused quantiser): every code and
    scale bit-exact, 4096 sampled outputs against the oracle."""
    X, idx, w = synth.moe_tokens(tokens=128)
    X = X.to(torch.bfloat16)
    counts = w.counts
    E, N, K = w.B.shape
    rows = int(counts.sum())
    assert rows == 256 and fp8g.fp8g_grouped_plan(N, K, rows, E)["BM"] == 128
    qb, sb = fp8g.quantize(w.B.reshape(E * N, K).cuda(), 32)
    qb_o, sb_o = oracle.quantize_block32(w.B.reshape(E * N, K).numpy())
    assert np.array_equal(qb.cpu().numpy(), qb_o)
    tok = idx.numpy()
    C, qa, sa, offs, _, _ = _fused(X, tok, qb.reshape(E, N, K), sb.reshape(E, N, K // 32), counts,
                                   N, K)
    qo, so = _oracle_codes(X, tok)
    _check_codes(qa, sa, qo, so)
    rng = np.random.default_rng(45)
    pi = np.concatenate([rng.integers(0, rows, 4096), [0, rows - 1]])
    pj = np.concatenate([rng.integers(0, N, 4096), [N - 1, 0]])
    oo = oracle.grouped_offsets(counts)
    expert = np.searchsorted(oo, pi, side="right") - 1
    x = C.float().cpu().numpy()
    qb_o = qb_o.reshape(E, N, K)
    sb_o = sb_o.reshape(E, N, K // 32)
    for e in np.unique(expert):
        sel = np.flatnonzero(expert == e)
        r, b, _ = oracle.gemm_sample(qo, qb_o[e], so, sb_o[e], True, pi[sel], pj[sel],
                                     oracle.OUT_BF16)
        assert_within(x[pi[sel], pj[sel]], r, b, f"decode MoE expert {e}")


def test_fused_bad_source_row_recorded():
    """A routed row naming a token outside X records FP8G_ERR_INVALID_ARG with
    the routed row as detail; that row quantises as zeros, nothing outside X is
    read, and the other rows are unaffected."""
    T, E, N, K = 64, 2, 256, 256
    counts = np.array([70, 58], np.int32)
    tok = (np.arange(128) % T).astype(np.int32)
    tok[77] = T + 9
    X = synth.normal((T, K), seed=51)
    qb, sb, _, _ = _weights(E, N, K, seed=52)
    C = torch.full((128, N), 5.0, dtype=torch.bfloat16, device="cuda")
    qa = torch.full((128, K), 0xEE, dtype=torch.uint8, device="cuda")
    sa = torch.full((128, K // 32), -1.0, device="cuda")
    fp8g.fp8_grouped_gemm_quant(X.cuda(), fp8g.FP8G_IN_F32, T, torch.from_numpy(tok).cuda(), qb,
                                sb, C, 0, 0, None, 0, torch.from_numpy(counts).cuda(), E, N, K,
                                128, None, 0, qa, sa, None, None, fp8g.FP8G_QUANT_FUSED)
    st, detail = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_ERR_INVALID_ARG and detail == 77
    assert (qa[77] == 0).all() and (sa[77] == 1.0).all() and (C[77].float() == 0.0).all()
    good = np.delete(np.arange(128), 77)
    qo, so = oracle.quantize_block32(X.numpy()[tok[good]])
    assert np.array_equal(qa.cpu().numpy()[good], qo)


def test_fused_zero_rows():
    E, N, K = 3, 256, 128
    qb, sb, _, _ = _weights(E, N, K, seed=61)
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    X = torch.zeros(4, K, device="cuda")
    C = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm_quant(X, fp8g.FP8G_IN_F32, 4, None, qb, sb, C, 0, 0, None, 0, counts, E,
                                N, K, 0, None, 0, None, None, offs, None, fp8g.FP8G_QUANT_FUSED)
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_OK
    assert (offs.cpu() == 0).all()
