"""Failure detection on the GPU without a fault: a device-side wait that can
never complete ends after its limit with FP8G_ERR_TIMEOUT in the status word
(read by the host), and the context stays usable afterwards."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp8_block_scaled_06_gb300 as fp8g
from gpu_util import assert_within, quant_both, run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fp8g, oracle_lib):
    yield


@pytest.mark.parametrize("limit_us", [500, 3000])
def test_wait_runs_out_and_is_reported(limit_us):
    fp8g.fp8_gemm_status()                                   # clear
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    fp8g.fp8g_wait_selftest(limit_us)
    e1.record()
    torch.cuda.synchronize()
    st, detail = fp8g.fp8_gemm_status()
    assert st == fp8g.FP8G_ERR_TIMEOUT and detail == 0xDEAD
    ms = e0.elapsed_time(e1)
    assert limit_us / 1000 * 0.95 <= ms < limit_us / 1000 + 100   # it waited, then gave up
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_OK         # read clears


def test_context_usable_after_timeout():
    fp8g.fp8g_wait_selftest(200)
    assert fp8g.fp8_gemm_status()[0] == fp8g.FP8G_ERR_TIMEOUT
    A = synth.normal((256, 512), seed=61)
    B = synth.normal((384, 512), seed=62)
    qa, sa, qa_o, sa_o = quant_both(A, 32)
    qb, sb, qb_o, sb_o = quant_both(B, 32)
    C = run_gemm(qa, sa, qb, sb, True, "bf16")               # asserts status OK
    ref, bound, _ = oracle.gemm(qa_o, qb_o, sa_o, sb_o, True, oracle.OUT_BF16)
    assert_within(C, ref, bound, "GEMM after a timeout")


def test_selftest_rejects_bad_limits():
    for bad in (0, 10_000_001):
        with pytest.raises(fp8g.Fp8gError) as e:
            fp8g.fp8g_wait_selftest(bad)
        assert e.value.status == fp8g.FP8G_ERR_INVALID_ARG
