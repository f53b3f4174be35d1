"""GPU parity of the MoE data movement around the grouped GEMM: the
gathering activation quantiser (fp32 or bf16 tokens -> expert-ordered FP8
rows + scales, bit-exact against the oracle's quantiser on the gathered
rows) and the grouped GEMM's row scatter back to (token, slot) order."""
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


def _gather_quant(x: torch.Tensor, idx: np.ndarray, block: int, fmt: int):
    """GPU gather-quantise of x[idx] vs the oracle's quantiser on x[idx] (fp32 values)."""
    n, cols = idx.size, x.shape[1]
    q = torch.empty((n, cols), dtype=torch.uint8, device="cuda")
    s = torch.empty((n, cols // 32) if block == 32 else (1,), dtype=torch.float32, device="cuda")
    dtype = fp8g.FP8G_IN_BF16 if x.dtype == torch.bfloat16 else fp8g.FP8G_IN_F32
    fp8g.fp8g_quantize_rows(x.cuda(), dtype, x.shape[0], cols, torch.from_numpy(idx).cuda(), n,
                            block, fmt, q, s)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    xg = x.float().numpy()[idx]                                  # bf16 -> fp32 is exact
    qo, so = (oracle.quantize_block32 if block == 32 else oracle.quantize_tensor)(xg, fmt)
    assert np.array_equal(q.cpu().numpy(), qo), f"{int((q.cpu().numpy() != qo).sum())} mismatches"
    assert np.array_equal(s.cpu().numpy().reshape(so.shape).view(np.uint32), so.view(np.uint32))
    return q, s, qo, so


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("block", [0, 32])
@pytest.mark.parametrize("fmt", [0, 1])
def test_gather_quantize_bitexact(dtype, block, fmt):
    g = torch.Generator().manual_seed(block + fmt)
    T, K = 300, 256
    x = (torch.randn(T, K, generator=g) * torch.exp(torch.randn(T, 1, generator=g))).to(dtype)
    rng = np.random.default_rng(7)
    idx = np.concatenate([rng.permutation(T), rng.integers(0, T, 77)]).astype(np.int32)
    _gather_quant(x, idx, block, fmt)


def test_gather_quantize_identity_equals_plain():
    x = synth.normal((64, 128), seed=3)
    q, s, _, _ = _gather_quant(x, np.arange(64, dtype=np.int32), 32, 0)
    qp, sp = fp8g.quantize(x.cuda(), 32)
    assert torch.equal(q, qp) and torch.equal(s, sp)


def test_gather_quantize_bad_row_recorded():
    x = torch.ones(8, 32, device="cuda")
    idx = torch.tensor([0, 9, 3], dtype=torch.int32, device="cuda")
    q = torch.full((3, 32), 0x55, dtype=torch.uint8, device="cuda")
    s = torch.zeros(3, 1, device="cuda")
    fp8g.fp8g_quantize_rows(x, fp8g.FP8G_IN_F32, 8, 32, idx, 3, 32, 0, q, s)
    st, detail = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_ERR_INVALID_ARG and detail == 1
    assert (q[1] == 0).all() and s[1].item() == 1.0              # zeros, nothing read
    assert (q[0] != 0).all() and (q[2] != 0).all()


def _route(T, E, seed):
    """Top-2 routing: each token to two distinct experts (seeded), rows in
    expert order.  Returns (counts, token of each routed row, C row = 2 t + slot)."""
    rng = np.random.default_rng(seed)
    w = rng.zipf(1.5, size=E).astype(np.float64)
    p = w / w.sum()
    pairs = np.array([rng.choice(E, 2, replace=False, p=p) for _ in range(T)])
    rows = [(e, t, s) for t in range(T) for s in range(2) for e in [pairs[t, s]]]
    rows.sort(key=lambda r: (r[0], r[1], r[2]))
    counts = np.bincount([r[0] for r in rows], minlength=E).astype(np.int32)
    tok = np.array([r[1] for r in rows], np.int32)
    crow = np.array([2 * r[1] + r[2] for r in rows], np.int32)
    return counts, tok, crow


@pytest.mark.parametrize("T,E,N,K", [(512, 4, 384, 256), (3000, 8, 2048, 512)])
def test_moe_gather_gemm_scatter(T, E, N, K):
    counts, tok, crow = _route(T, E, seed=T)
    x = synth.normal((T, K), seed=T + 1).to(torch.bfloat16)
    qa, sa, qa_o, sa_o = _gather_quant(x, tok, 32, 0)
    B = synth.normal((E, N, K), seed=T + 2, std=0.02)
    qb, sb = fp8g.quantize(B.reshape(E * N, K).cuda(), 32)
    qb_o, sb_o = oracle.quantize_block32(B.reshape(E * N, K).numpy())
    assert np.array_equal(qb.cpu().numpy(), qb_o)
    rows = int(counts.sum())
    C = torch.full((2 * T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    bias = np.random.default_rng(1).normal(size=(E, N)).astype(np.float32)
    fp8g.fp8_grouped_gemm_scatter(qa, qb.reshape(E, N, K), sa, sb.reshape(E, N, K // 32), C, 0,
                                  0, 0, torch.from_numpy(bias).cuda(), fp8g.FP8G_ACT_RELU,
                                  torch.from_numpy(counts).cuda(), E, N, K, rows,
                                  torch.from_numpy(crow).cuda(), 2 * T)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    Ch = C.float().cpu().numpy()
    offs = oracle.grouped_offsets(counts)
    ref = np.empty((2 * T, N), np.float32)
    bound = np.empty((2 * T, N), np.float64)
    for e in range(E):
        a, b = offs[e], offs[e + 1]
        if a == b:
            continue
        r, bd, _ = oracle.gemm(qa_o[a:b], qb_o[e * N:(e + 1) * N], sa_o[a:b],
                               sb_o[e * N:(e + 1) * N], True, oracle.OUT_BF16, bias=bias[e],
                               act_kind=oracle.ACT_RELU)
        ref[crow[a:b]] = r
        bound[crow[a:b]] = bd
    assert_within(Ch, ref, bound, f"MoE gather/GEMM/scatter T={T}")


def test_scatter_bad_row_recorded():
    counts = np.array([128], np.int32)
    N, K = 128, 128
    qa = torch.zeros(128, K, dtype=torch.uint8, device="cuda")
    qb = torch.zeros(1, N, K, dtype=torch.uint8, device="cuda")
    sa = torch.ones(128, K // 32, device="cuda")
    sb = torch.ones(1, N, K // 32, device="cuda")
    crow = torch.arange(128, dtype=torch.int32, device="cuda")
    crow[5] = 500                                               # outside C's 128 rows
    C = torch.full((128, N), 3.0, dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_grouped_gemm_scatter(qa, qb, sa, sb, C, 0, 0, 0, None, 0,
                                  torch.from_numpy(counts).cuda(), 1, N, K, 128, crow, 128)
    st, detail = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_ERR_INVALID_ARG and detail == 5
    assert (C[5].float() == 3.0).all() and (C[4].float() == 0.0).all()
