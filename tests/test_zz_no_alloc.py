"""The allocation-free block-scaled GEMM entry point.

fp8_gemm_blockscaled_noalloc is for callers that cannot let the library
allocate device memory (a fixed device-memory budget, an allocator that owns
every device byte, a path where allocation calls are not allowed).  It keeps
the repacked scales in a fixed array inside the library instead of a pool
temporary, so its results must equal fp8_gemm_blockscaled's.  Two calls in a
row on different inputs check that nothing left in the shared array from the
previous call leaks into the next one.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import synth
import fp8_block_scaled_06_gb300 as fp8g

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    A = synth.with_outliers(synth.normal((M, K), seed=seed), g)
    B = synth.normal((N, K), seed=seed + 1000) * torch.exp(torch.randn(N, 1, generator=g) * 2)
    qa, sa = fp8g.quantize(A.cuda(), 32)
    qb, sb = fp8g.quantize(B.cuda(), 32)
    return qa, sa, qb, sb


def test_noalloc_matches_blockscaled_two_calls(fp8g):
    # two different shapes back to back, the second with ragged M / N / K tails
    for (M, N, K, out), seed in (((512, 768, 1024, "bf16"), 11), ((300, 392, 320, "f32"), 12)):
        qa, sa, qb, sb = _operands(M, N, K, seed)
        dt = torch.bfloat16 if out == "bf16" else torch.float32
        o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
        ref = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        got = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, ref, o, M, N, K)
        fp8g.fp8_gemm_blockscaled_noalloc(qa, qb, sa, sb, got, o, M, N, K)
        st, detail = fp8g.fp8_gemm_status()
        assert st == 0, f"device status {st} detail {detail}"
        r = ref.float().cpu().numpy()
        x = got.float().cpu().numpy()
        assert not np.isnan(x).any()
        # same kernels, same accumulation order: identical bits
        assert np.array_equal(r.view(np.uint32), x.view(np.uint32))


def test_noalloc_rejects_shapes_over_its_limit(fp8g):
    # (ceil(M/128) + 2 ceil(N/256)) * ceil(K/128) * 512 > 8 MiB -> refused before launch
    qa = torch.zeros(16, 16, dtype=torch.uint8, device="cuda")
    s = torch.ones(16, device="cuda")
    C = torch.empty(16, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm_blockscaled_noalloc(qa, qa, s, s, C, 0, 32768, 32768, 32768)
    assert e.value.status == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_OK
