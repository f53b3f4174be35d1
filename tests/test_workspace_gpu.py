"""The block-scaled entry points repack the scales into a stream-ordered
temporary from the library pool on every call.  These tests change shapes,
alternate streams, replace a destroyed stream, capture calls into a CUDA
graph and release the pool with fp8g_shutdown; every result is checked
against the oracle or against an eager call of the same kernel."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within, quant_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


def _case(M, N, K, seed):
    A = synth.normal((M, K), seed=seed)
    B = synth.normal((N, K), seed=seed + 1)
    qa, sa, qa_o, sa_o = quant_both(A, 32)
    qb, sb, qb_o, sb_o = quant_both(B, 32)
    return (qa, sa, qb, sb), (qa_o, sa_o, qb_o, sb_o)


def _check(C, ref_in, M, N, what, pts=1500):
    qa_o, sa_o, qb_o, sb_o = ref_in
    rng = np.random.default_rng(M + N)
    pi = np.concatenate([[0, M - 1], rng.integers(0, M, pts)])
    pj = np.concatenate([[N - 1, 0], rng.integers(0, N, pts)])
    ref, bound, _ = oracle.gemm_sample(qa_o, qb_o, sa_o, sb_o, True, pi, pj, oracle.OUT_BF16)
    assert_within(C.float().cpu().numpy()[pi, pj], ref, bound, what)


# single-CTA and CTA-pair shapes whose packed scales differ in size
SHAPES = [(512, 384, 256), (2304, 2304, 512), (1024, 768, 1024), (4096, 4608, 512)]


def test_shapes_alternate_streams():
    cases = [(_case(M, N, K, 100 + i), (M, N, K)) for i, (M, N, K) in enumerate(SHAPES)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for rep in range(2):
        for i, ((gpu_in, _), (M, N, K)) in enumerate(cases):
            s = s1 if (i + rep) % 2 == 0 else s2
            with torch.cuda.stream(s):      # the NaN fill, then the GEMM, on s
                C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
                qa, sa, qb, sb = gpu_in
                fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C, 0, M, N, K, s)
            outs.append((C, i))
    torch.cuda.synchronize()
    assert fp8g.fp8_gemm_status()[0] == 0
    for C, i in outs:
        M, N, K = cases[i][1]
        _check(C, cases[i][0][1], M, N, f"stream reuse {M}x{N}x{K}")


def test_replaced_stream_and_back_to_back_calls():
    (gpu_in, ref_in) = _case(2304, 2304, 512, 7)
    qa, sa, qb, sb = gpu_in
    M = N = 2304
    K = 512
    s = torch.cuda.Stream()
    C1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C1, 0, M, N, K, s)
    del s                                 # destroyed with work possibly pending
    s = torch.cuda.Stream()
    Cs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for C in Cs:                          # back-to-back calls
        fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C, 0, M, N, K, s)
    torch.cuda.synchronize()
    assert fp8g.fp8_gemm_status()[0] == 0
    _check(C1, ref_in, M, N, "first stream")
    for C in Cs:
        assert torch.equal(C, C1)         # same kernel, same inputs: identical bits


def test_graph_capture_matches_eager():
    (gpu_in, ref_in) = _case(2304, 2304, 512, 9)
    qa, sa, qb, sb = gpu_in
    M = N = 2304
    K = 512
    C_eager = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C_eager, 0, M, N, K)
    torch.cuda.synchronize()
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C, 0, M, N, K, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert fp8g.fp8_gemm_status()[0] == 0
    assert torch.equal(C, C_eager)
    _check(C, ref_in, M, N, "graph replay")


def test_graph_capture_grouped_from_tokens_two_calls():
    """The grouped GEMM from bf16 tokens (quantiser, scale packing and GEMM,
    each kernel placed while its predecessor finishes) captured twice back to
    back in one graph: replays give the eager bits, for both calls."""
    counts = np.array([300, 0, 5, 211], np.int32)
    E, N, K = counts.size, 512, 1024
    rows = int(counts.sum())
    tokens = 320
    g_ = torch.Generator().manual_seed(91)
    X = torch.randn(tokens, K, generator=g_).to(torch.bfloat16).cuda()
    idx = torch.randint(0, tokens, (rows,), generator=g_, dtype=torch.int32).cuda()
    w = synth.small_grouped(counts, N, K, seed=92)
    qb, sb = fp8g.quantize(w.B.reshape(E * N, K).cuda(), 32)
    qb, sb = qb.reshape(E, N, K), sb.reshape(E, N, K // 32)
    dc = torch.from_numpy(counts).cuda()

    def call(C, stream):
        fp8g.fp8_grouped_gemm_quant(X, fp8g.FP8G_IN_BF16, tokens, idx, qb, sb, C,
                                    fp8g.FP8G_OUT_BF16, fp8g.FP8G_E4M3, None, fp8g.FP8G_ACT_NONE,
                                    dc, E, N, K, rows, stream=stream)

    C_eager = torch.empty((rows, N), dtype=torch.bfloat16, device="cuda")
    call(C_eager, None)
    torch.cuda.synchronize()
    assert fp8g.fp8_gemm_status()[0] == 0
    Cs = [torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for C in Cs:
                call(C, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert fp8g.fp8_gemm_status()[0] == 0
    for C in Cs:
        assert torch.equal(C, C_eager)


def test_shutdown_releases_and_calls_continue():
    (gpu_in, ref_in) = _case(1024, 768, 1024, 11)
    qa, sa, qb, sb = gpu_in
    M, N, K = 1024, 768, 1024
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C, 0, M, N, K)
    fp8g.fp8g_shutdown()
    C2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C2, 0, M, N, K)
    torch.cuda.synchronize()
    assert fp8g.fp8_gemm_status()[0] == 0
    assert torch.equal(C, C2)
    _check(C2, ref_in, M, N, "after shutdown")
