"""Helpers for the GPU parity tests: each side quantises with its own code
(the CUDA quantiser kernel vs the oracle's C quantiser), codes and scales are
compared bit for bit, then each side's GEMM runs on its own inputs."""
import numpy as np
import torch

import oracle
import fp8_block_scaled_06_gb300 as fp8g


def quant_both(x: torch.Tensor, block: int):
    """x: CPU fp32 [rows, cols]. Returns (gpu codes, gpu scales, oracle codes, oracle scales)."""
    qg, sg = fp8g.quantize(x.cuda(), block)
    if block == 32:
        qo, so = oracle.quantize_block32(x.numpy())
    else:
        qo, so = oracle.quantize_tensor(x.numpy())
    return qg, sg, qo, so


def assert_codes_equal(qg, sg, qo, so):
    qg_h = qg.cpu().numpy()
    sg_h = sg.cpu().numpy().reshape(so.shape)
    assert np.array_equal(qg_h, qo), f"{int((qg_h != qo).sum())} code mismatches"
    assert np.array_equal(sg_h.view(np.uint32), so.view(np.uint32)), "scale mismatch"


def assert_within(C_gpu: np.ndarray, C_ref: np.ndarray, bound: np.ndarray, what: str = ""):
    """|C - C_ref| <= 2^-8 sum|sA a||sB b| + 1 bf16 ulp(|C_ref|), NaN where the reference is NaN."""
    C_gpu = C_gpu.astype(np.float64)
    C_ref = C_ref.astype(np.float64)
    nan_ref = np.isnan(C_ref)
    assert np.array_equal(np.isnan(C_gpu), nan_ref), f"{what}: NaN pattern differs"
    d = np.abs(C_gpu - C_ref)
    ok = (d <= bound) | nan_ref
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        info = [(tuple(i), C_gpu[tuple(i)], C_ref[tuple(i)], bound[tuple(i)]) for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance, e.g. {info}")


def run_gemm(qa, sa, qb, sb, block: bool, out: str):
    M, K = qa.shape
    N = qb.shape[0]
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    C = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    o = fp8g.FP8G_OUT_BF16 if out == "bf16" else fp8g.FP8G_OUT_F32
    if block:
        fp8g.fp8_gemm_blockscaled(qa, qb, sa, sb, C, o, M, N, K)
    else:
        fp8g.fp8_gemm(qa, qb, sa, sb, C, o, M, N, K)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"device status {st} ({fp8g.fp8g_status_string(st)}), detail {detail}"
    return C.float().cpu().numpy()


def oracle_out(out: str) -> int:
    return oracle.OUT_BF16 if out == "bf16" else oracle.OUT_F32
