"""Parity of the widened workloads at the sizes the bench times them, built
and launched by the bench's own code (bench.make_inputs, bench.run_once): the
GPU quantisation bit-exact against the oracle's own quantisation of the same
synthetic data, then 2048 sampled outputs plus the four corners against the
oracle.  (The FP8 workloads at full size: test_gemm_gpu.py,
test_grouped_gpu.py.)"""
import numpy as np
import pytest
import torch

import bench
import oracle
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def pack(codes: np.ndarray, fmt: int) -> np.ndarray:
    """One code per byte -> the library's packed bytes of format fmt."""
    c = codes.astype(np.uint32)
    if fmt == fp8g.FP8G_E2M1:
        return ((c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    if fmt in (fp8g.FP8G_E2M3, fp8g.FP8G_E3M2):
        v = (c[:, 0::4] & 0x3F) | ((c[:, 1::4] & 0x3F) << 6) | ((c[:, 2::4] & 0x3F) << 12) | \
            ((c[:, 3::4] & 0x3F) << 18)
        return np.stack([v & 0xFF, (v >> 8) & 0xFF, (v >> 16) & 0xFF], 2).reshape(c.shape[0], -1) \
            .astype(np.uint8)
    return codes


def _run(name):
    wl = bench.WORKLOADS[name]
    w, t = bench.make_inputs(wl, torch.device("cuda"))
    assert fp8g.fp8_gemm_status()[0] == 0
    dt = torch.float32 if w.out == "f32" else torch.bfloat16
    rows = (t["qa"] if "qa" in t else t["tmp_qa"]).shape[0]
    C = torch.full((rows, wl["N"]), float("nan"), dtype=dt, device="cuda")
    bench.run_once(fp8g, wl, w, t, C, torch.cuda.current_stream())
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"status {st} detail {detail}"
    return wl, w, t, C.float().cpu().numpy()


def _same(gpu: torch.Tensor, want: np.ndarray, what: str):
    g = gpu.cpu().numpy().reshape(want.shape)
    if want.dtype == np.float32:
        g, want = g.view(np.uint32), want.view(np.uint32)
    assert np.array_equal(g, want), f"{what}: {int((g != want).sum())} mismatches"


def _points(M, N, seed):
    rng = np.random.default_rng(seed)
    pi = np.concatenate([rng.integers(0, M, 2048), [0, 0, M - 1, M - 1]])
    pj = np.concatenate([rng.integers(0, N, 2048), [0, N - 1, 0, N - 1]])
    return pi, pj


@pytest.mark.parametrize("name", ["tensor8192", "mixed8192", "literal8192", "mxfp4_8192",
                                  "mxfp6_8192"])
def test_workload_sampled(name):
    wl, w, t, C = _run(name)
    fa, fb = wl.get("a_fmt", 0), wl.get("b_fmt", 0)
    block = wl["kind"] != "tensor"
    out = []
    for x, fmt, q, s in ((w.A, fa, t["qa"], t["sa"]), (w.B, fb, t["qb"], t["sb"])):
        if not block:
            qo, so = oracle.quantize_tensor(x.numpy(), fmt)
        else:
            qo, so = oracle.quantize_block32(x.numpy(), fmt, literal=bool(wl.get("literal")))
        _same(q, pack(qo, fmt), f"{name} codes")
        _same(s, so, f"{name} scales")
        out.append((qo, so))
    (qa_o, sa_o), (qb_o, sb_o) = out
    pi, pj = _points(wl["M"], wl["N"], 8192)
    ok = oracle.OUT_F32 if w.out == "f32" else oracle.OUT_BF16
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, block, pi, pj, ok, a_fmt=fa,
                                       b_fmt=fb)
    assert_within(C[pi, pj], ref, bound, f"{name} sampled")


def test_workload_nvfp4_sampled():
    wl, w, t, C = _run("nvfp4_8192")
    out = []
    for x, q, s, g in ((w.A, t["qa"], t["sa"], t["ga"]), (w.B, t["qb"], t["sb"], t["gb"])):
        qo, so, go = oracle.quantize_nvfp4(x.numpy())
        _same(q, pack(qo, fp8g.FP8G_E2M1), "nvfp4 codes")
        _same(s, so, "nvfp4 scale codes")
        _same(g, np.array([go], np.float32), "nvfp4 tensor scale")
        out.append((qo, so, go))
    (qa_o, sa_o, ga_o), (qb_o, sb_o, gb_o) = out
    pi, pj = _points(wl["M"], wl["N"], 4)
    ref, bound, _ = oracle.gemm_nvfp4_sample(qa_o, qb_o, sa_o, sb_o, ga_o, gb_o, pi, pj,
                                             oracle.OUT_BF16)
    assert_within(C[pi, pj], ref, bound, "nvfp4_8192 sampled")


def test_workload_moe_nvfp4_sampled():
    """The MoE workload in NVFP4 (8 experts, N=14336, K=4096, 32768 routed
    rows with Zipf counts): A's and every expert's quantisation bit-exact,
    outputs sampled over all rows."""
    wl, w, t, C = _run("moe_nvfp4")
    qa_o, sa_o, ga_o = oracle.quantize_nvfp4(w.A.numpy())
    _same(t["qa"], pack(qa_o, fp8g.FP8G_E2M1), "moe A codes")
    _same(t["sa"], sa_o, "moe A scale codes")
    _same(t["ga"], np.array([ga_o], np.float32), "moe gA")
    E = w.B.shape[0]
    experts = []
    for e in range(E):
        qo, so, go = oracle.quantize_nvfp4(w.B[e].numpy())
        _same(t["qb"][e], pack(qo, fp8g.FP8G_E2M1), f"expert {e} codes")
        _same(t["sb"][e], so, f"expert {e} scale codes")
        _same(t["gb"][e:e + 1], np.array([go], np.float32), f"expert {e} gB")
        experts.append((qo, so, go))
    rows = int(w.counts.sum())
    offs = oracle.grouped_offsets(w.counts)
    pi, pj = _points(rows, wl["N"], 5)
    expert = np.searchsorted(offs, pi, side="right") - 1
    for e in np.unique(expert):
        sel = np.flatnonzero(expert == e)
        r0, r1 = int(offs[e]), int(offs[e + 1])
        qb_o, sb_o, gb_o = experts[e]
        ref, bound, _ = oracle.gemm_nvfp4_sample(qa_o[r0:r1], qb_o, sa_o[r0:r1], sb_o, ga_o, gb_o,
                                                 pi[sel] - r0, pj[sel], oracle.OUT_BF16)
        assert_within(C[pi[sel], pj[sel]], ref, bound, f"moe_nvfp4 expert {e}")


def _grouped_sampled(name, qa_o, sa_o, qb_o, sb_o, counts, C, seed):
    rows = int(counts.sum())
    N = qb_o.shape[1]
    offs = oracle.grouped_offsets(counts)
    pi, pj = _points(rows, N, seed)
    expert = np.searchsorted(offs, pi, side="right") - 1
    for e in np.unique(expert):
        sel = np.flatnonzero(expert == e)
        r0, r1 = int(offs[e]), int(offs[e + 1])
        ref, bound, _ = oracle.gemm_sample(qa_o[r0:r1], qb_o[e], sa_o[r0:r1], sb_o[e],
                                           True, pi[sel] - r0, pj[sel], oracle.OUT_BF16)
        assert_within(C[pi[sel], pj[sel]], ref, bound, f"{name} problem {e}")


def test_workload_skinny_x8_sampled():
    """Eight independent skinny products (128 x 4096 x 4096, the skinny
    recipe) in one grouped call: every code and scale bit-exact, sampled
    outputs of every product against the oracle."""
    wl, w, t, C = _run("skinny_x8")
    E, N, K = w.B.shape
    qa_o, sa_o = oracle.quantize_block32(w.A.numpy())
    qb_o, sb_o = oracle.quantize_block32(w.B.reshape(E * N, K).numpy())
    _same(t["qa"], qa_o, "skinny_x8 A codes")
    _same(t["sa"], sa_o, "skinny_x8 A scales")
    _same(t["qb"], qb_o, "skinny_x8 B codes")
    _same(t["sb"], sb_o, "skinny_x8 B scales")
    _grouped_sampled("skinny_x8", qa_o, sa_o, qb_o.reshape(E, N, K), sb_o.reshape(E, N, K // 32),
                     w.counts, C, 6)


def test_workload_decode_bf16_sampled():
    """The decode-shaped MoE from bf16 tokens as the bench runs it, through
    the fused quantiser, the one-call and the two-call paths: the same bits, and
    sampled outputs against the oracle's quantisation of the gathered tokens
    and its GEMM."""
    import synth
    wl, w, t, C = _run("decode_bf16_fused")
    wl2, _, t2, C2 = _run("decode_bf16_2call")
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32))
    C1 = _run("decode_bf16")[3]
    assert np.array_equal(C1.view(np.uint32), C2.view(np.uint32))
    X, idx, _ = synth.moe_tokens(seed=wl["seed"], tokens=wl["tokens"])
    qa_o, sa_o = oracle.quantize_block32(X.to(torch.bfloat16).float().numpy()[idx.numpy()])
    _same(t2["tmp_qa"], qa_o, "decode A codes (two calls)")
    _same(t2["tmp_sa"], sa_o, "decode A scales (two calls)")
    E, N, K = w.B.shape
    qb_o, sb_o = oracle.quantize_block32(w.B.reshape(E * N, K).numpy())
    _same(t["qb"], qb_o, "decode B codes")
    _grouped_sampled("decode_bf16", qa_o, sa_o, qb_o.reshape(E, N, K), sb_o.reshape(E, N, K // 32),
                     w.counts, C, 7)

