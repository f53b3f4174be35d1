"""The allocation-free block-scaled GEMM entry point.

fp8_gemm_blockscaled_noalloc is for callers that cannot let the library
allocate device memory (a fixed device-memory budget, an allocator that owns
every device byte, a path where allocation calls are not allowed).  It keeps
the repacked scales in a fixed 16 MiB array inside the library instead of a
pool temporary.

Every shape here takes a kernel that reads repacked scales (plan split_k == 1:
the CTA-pair kernel and the single-CTA 256-wide kernel; split-K shapes convert
their scales inside the GEMM and never touch the array), so the array is
written by the packing kernel and read by the GEMM on every call.  Each output
is compared element by element with the oracle (the tolerance of every parity
test) and bit for bit with fp8_gemm_blockscaled.  The calls run back to back,
the largest first, so a later, smaller call finds the previous call's packed
scales in the array beyond what it rewrites.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_codes_equal, assert_within, oracle_out, quant_both

pytestmark = pytest.mark.gpu

# (M, N, K, out, seed, kernel): CTA pairs take 256-row tiles, the single-CTA
# kernel 128 x 256 tiles whose B scales are packed replicated (4 KB per
# 256 rows and K step)
CASES = [
    (4096, 4096, 512, "bf16", 11, "pair"),
    (2048, 2040, 1024, "f32", 12, "single"),
    (2000, 3000, 640, "bf16", 13, "pair"),     # ragged M, N tails and K
]


def _operands(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    A = synth.with_outliers(synth.normal((M, K), seed=seed), g)
    B = synth.normal((N, K), seed=seed + 1000) * torch.exp(torch.randn(N, 1, generator=g) * 2)
    qa, sa, qa_o, sa_o = quant_both(A, 32)
    qb, sb, qb_o, sb_o = quant_both(B, 32)
    assert_codes_equal(qa, sa, qa_o, sa_o)
    assert_codes_equal(qb, sb, qb_o, sb_o)
    return qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o


def _scratch_bytes(M, N, K, pair):
    """Repacked scale bytes of one call (A's chunks + B's chunks)."""
    kg = -(-K // 128)
    rows_b = 2 * -(-N // 256)
    return (-(-M // 128) + rows_b * (1 if pair else 4)) * kg * 512


def test_noalloc_packs_into_its_array_and_matches(fp8g, oracle_lib):
    for M, N, K, out, seed, kernel in CASES:
        plan = fp8g.fp8g_gemm_plan(1, M, N, K)
        assert plan["split_k"] == 1, (M, N, K, plan)          # the packing path runs
        assert plan["BM"] == (256 if kernel == "pair" else 128) and plan["BN"] == 256
        assert _scratch_bytes(M, N, K, kernel == "pair") <= 16 << 20
        qa, sa, qb, sb, qa_o, sa_o, qb_o, sb_o = _operands(M, N, K, seed)
        dt = torch.bfloat16 if out == "bf16" else torch.float32
        o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
        got = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        fp8g.fp8_gemm_blockscaled_noalloc(qa, qb, sa, sb, got, o, M, N, K)
        st, detail = fp8g.fp8_gemm_status()
        assert st == 0, f"device status {st} detail {detail}"
        ref_lib = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, ref_lib, o, M, N, K)
        assert fp8g.fp8_gemm_status()[0] == 0
        x = got.float().cpu().numpy()
        ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle_out(out))
        assert_within(x, ref, bound, f"noalloc {kernel} {M}x{N}x{K} {out}")
        # same kernels, same accumulation order as the pool-backed call
        r = ref_lib.float().cpu().numpy()
        assert np.array_equal(r.view(np.uint32), x.view(np.uint32))


def test_noalloc_rejects_shapes_over_its_limit(fp8g):
    # M = N = 4096 on CTA pairs: (32 + 32) * ceil(K/128) * 512 bytes of packed
    # scales; K = 66048 needs 516 * 32 KiB > 16 MiB.  The operands have their
    # true sizes (about 0.65 GB in all), so no argument points at a buffer
    # smaller than the shape says.
    M = N = 4096
    K = 66048
    plan = fp8g.fp8g_gemm_plan(1, M, N, K)
    assert plan["split_k"] == 1 and plan["BM"] == 256
    assert _scratch_bytes(M, N, K, True) > 16 << 20
    qa = torch.zeros(M, K, dtype=torch.uint8, device="cuda")
    qb = torch.zeros(N, K, dtype=torch.uint8, device="cuda")
    s = torch.ones(M, K // 32, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm_blockscaled_noalloc(qa, qb, s, s, C, 0, M, N, K)
    assert e.value.status == fp8g.FP8G_ERR_UNSUPPORTED_SHAPE
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_OK
    assert bool((C == 7.0).all())                            # nothing was launched
    del qa, qb, s, C
    torch.cuda.empty_cache()
