"""FP8 GEMM throughput on GB300: TFLOPS and fraction of the roofline.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload large8192|large4096|skinny|moe|square256|square1024|tensor8192|
                            mixed8192|literal8192|mxfp4_8192|mxfp6_8192|nvfp4_8192|
                            moe_nvfp4|moe_bf16|moe_bf16_2call|decode_bf16|
                            decode_bf16_fused|decode_bf16_2call|skinny_x8|moe_2x2048]

One step = one GEMM call (the whole hot path: tile scheduling, TMA ring,
scale staging, tcgen05 MMA, epilogue) over one batch of synthetic input
already resident in HBM.  Operand quantisation is data preparation and is
not timed (it is its own kernel and its own metric), except in the MoE
workloads from bf16 tokens (*_bf16*), whose step quantises the routed rows
(fused into the GEMM, or as a pass of its own).  The default workload is
the large block-scaled GEMM M=N=K=8192 (1x32 scales along K, N(0,1) with 0.1%
x50 outliers, bf16 out), the shape the >= 70%-of-peak target is quoted on.

L2: the timed steps rotate over several copies of the inputs whose total is
larger than 2x the L2, so every step reads its operands from HBM.

Multi-GPU (torchrun, one rank per GPU): replicas only — every rank runs the
same GEMM on its own GPU, no collective on the data path; value = total FLOPs
of all ranks / max-over-ranks time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

WORKLOADS = {
    "large8192": dict(kind="block", M=8192, N=8192, K=8192, seed=3),
    "large4096": dict(kind="block", M=4096, N=4096, K=4096, seed=3),
    "skinny": dict(kind="block", M=128, N=4096, K=4096, seed=2),
    "moe": dict(kind="grouped", M=32768, N=14336, K=4096, seed=4),
    # eight independent skinny products (128 x 4096 x 4096 each, the skinny
    # recipe) in one grouped call: the skinny shape batched into one launch
    "skinny_x8": dict(kind="grouped", M=1024, N=4096, K=4096, seed=2, batch=8),
    # reduced MoE for profiling captures: 2 experts of the MoE's size, 2048
    # tokens top-2 (2048 routed rows each), about 0.25 GB on the device
    "moe_2x2048": dict(kind="grouped", M=4096, N=14336, K=4096, seed=4, experts=2, tokens=2048),
    "square256": dict(kind="tensor", M=256, N=256, K=256, seed=0),
    "square1024": dict(kind="tensor", M=1024, N=1024, K=1024, seed=1),
    "tensor8192": dict(kind="tensor", M=8192, N=8192, K=8192, seed=3),
    # E4M3 activations x E5M2 weights, block-scaled (the mixed-format path)
    "mixed8192": dict(kind="block", M=8192, N=8192, K=8192, seed=3, b_fmt=1),
    # literal fp32 block scales amax/448 (promotion GEMM)
    "literal8192": dict(kind="block", M=8192, N=8192, K=8192, seed=3, literal=True),
    # E2M1 x E2M1 with power-of-two 1x32 scales (MXFP4), two codes per byte
    "mxfp4_8192": dict(kind="block", M=8192, N=8192, K=8192, seed=3, a_fmt=2, b_fmt=2),
    # E2M3 x E2M3 with power-of-two 1x32 scales (MXFP6), four codes per 3 bytes
    "mxfp6_8192": dict(kind="block", M=8192, N=8192, K=8192, seed=3, a_fmt=3, b_fmt=3),
    # NVFP4: E2M1 with 1x16 E4M3 block scales and an fp32 scale per tensor
    "nvfp4_8192": dict(kind="nvfp4", M=8192, N=8192, K=8192, seed=3, a_fmt=2, b_fmt=2),
    # the MoE workload in NVFP4 (each expert's weight with its own tensor scale)
    "moe_nvfp4": dict(kind="grouped_nvfp4", M=32768, N=14336, K=4096, seed=4, a_fmt=2, b_fmt=2),
    # MoE from bf16 token activations, the routed rows' 1x32 E4M3 quantisation
    # inside the timed step: fp8_grouped_gemm_quant (one call; "fused": with
    # FP8G_QUANT_FUSED, the quantiser inside the GEMM kernel where the plan
    # runs single-CTA tiles) against fp8g_quantize_rows + fp8_grouped_gemm
    # (two calls).  The full MoE size runs 256-row tiles (never fused);
    # 128 tokens (decoding: 256 routed rows) run single-CTA tiles.
    "moe_bf16": dict(kind="grouped_quant", M=32768, N=14336, K=4096, seed=4, tokens=16384,
                     path="1call"),
    "moe_bf16_2call": dict(kind="grouped_quant", M=32768, N=14336, K=4096, seed=4,
                           tokens=16384, path="2call"),
    "decode_bf16": dict(kind="grouped_quant", M=256, N=14336, K=4096, seed=4, tokens=128,
                        path="1call"),
    "decode_bf16_fused": dict(kind="grouped_quant", M=256, N=14336, K=4096, seed=4, tokens=128,
                              path="fused"),
    "decode_bf16_2call": dict(kind="grouped_quant", M=256, N=14336, K=4096, seed=4, tokens=128,
                              path="2call"),
}
FMT_NAMES = ["e4m3", "e5m2", "e2m1", "e2m3", "e3m2"]
# bytes per element of each format in memory (E2M1: two codes per byte; FP6:
# four codes per three bytes)
FMT_BYTES = [1.0, 1.0, 0.5, 0.75, 0.75]
METRIC = "FP8 GEMM TFLOPS and % of GB300 roofline (tensor peak or HBM) at 1 GPU"


def bf16_peak_for(peaks: dict, region_s: float):
    """(sustained?, bf16 TFLOP/s) for a timed region of region_s seconds: one
    of a second or more is a long step at the power cap, measured against the
    sustained rate (bf16 GEMMs back to back for seconds); a shorter one runs
    in the burst, against the burst rate."""
    sustained = region_s >= 1.0
    return sustained, (peaks["bf16_sus"] if sustained else peaks["bf16"])


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 10 ms with the host
    time of each sample, so that the record can be cut to the window in which
    the GPU ran the timed calls."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 10

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []   # (host perf_counter time, csv line)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.perf_counter(), ln.strip()))

    def stop(self, t0: float | None = None, t_region: float | None = None,
             t1: float | None = None, tail_ms: float = 0.0) -> dict:
        """Summary of the samples taken in [t0, t1] (host times; all samples if
        t0 is None); [t0, t_region] is the timed region itself."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._t.join(timeout=2)
        return self.summarize(self.lines, t0, t_region, t1, tail_ms)

    @classmethod
    def summarize(cls, lines, t0=None, t_region=None, t1=None, tail_ms: float = 0.0) -> dict:
        sm, smax, reasons, power, in_region = [], None, set(), [], 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for th, ln in lines:
            if t0 is not None and not (t0 <= th <= t1):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            if t0 is not None and th <= t_region:
                in_region += 1
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
               "reasons": sorted(reasons), "samples": len(sm),
               "power_w_max": max(power) if power else None}
        if t0 is not None:
            out["samples_in_timed_region"] = in_region
            out["window"] = (f"every {cls.INTERVAL_MS} ms over the timed region "
                             f"({(t_region - t0) * 1e3:.1f} ms) and a {tail_ms:.0f}-ms run of "
                             f"the same calls queued right behind it")
        return out


def make_inputs(wl: dict, device):
    """Synthetic operands (CPU, seeded) -> quantised on the GPU by the library."""
    import synth
    import fp8_block_scaled_06_gb300 as fp8g

    if wl["kind"] == "grouped":
        w = (synth.skinny_batch(wl["batch"], seed=wl["seed"]) if "batch" in wl else
             synth.moe_grouped(seed=wl["seed"], experts=wl.get("experts", 8),
                               tokens=wl.get("tokens", 16384)))
        E, N, K = w.B.shape
        qa, sa = fp8g.quantize(w.A.to(device), 32)
        qb, sb = fp8g.quantize(w.B.reshape(E * N, K).to(device), 32)
        qb = qb.reshape(E, N, K)
        sb = sb.reshape(E, N, K // 32)
        counts = torch.from_numpy(w.counts).to(device)
        return w, dict(qa=qa, sa=sa, qb=qb, sb=sb, counts=counts)
    if wl["kind"] == "grouped_quant":
        X, idx, w = synth.moe_tokens(seed=wl["seed"], tokens=wl["tokens"])
        E, N, K = w.B.shape
        qb, sb = fp8g.quantize(w.B.reshape(E * N, K).to(device), 32)
        rows = int(w.counts.sum())
        # tmp_*: the two-call path's quantised rows (outputs of its first call)
        return w, dict(X=X.to(torch.bfloat16).to(device), idx=idx.to(device),
                       qb=qb.reshape(E, N, K), sb=sb.reshape(E, N, K // 32),
                       counts=torch.from_numpy(w.counts).to(device),
                       tmp_qa=torch.empty((rows, K), dtype=torch.uint8, device=device),
                       tmp_sa=torch.empty((rows, K // 32), dtype=torch.float32, device=device))
    if wl["kind"] == "grouped_nvfp4":
        w = synth.moe_grouped(seed=wl["seed"], experts=wl.get("experts", 8),
                              tokens=wl.get("tokens", 16384))
        qa, sa, ga = fp8g.quantize_nvfp4(w.A.to(device))
        qbs = [fp8g.quantize_nvfp4(w.B[e].to(device)) for e in range(w.B.shape[0])]
        qb, sb, gb = (torch.stack([q[0] for q in qbs]), torch.stack([q[1] for q in qbs]),
                      torch.cat([q[2] for q in qbs]))
        counts = torch.from_numpy(w.counts).to(device)
        return w, dict(qa=qa, sa=sa, ga=ga, qb=qb, sb=sb, gb=gb, counts=counts)
    if wl["kind"] == "nvfp4":
        w = synth.large_block(wl["M"], seed=wl["seed"])
        qa, sa, ga = fp8g.quantize_nvfp4(w.A.to(device))
        qb, sb, gb = fp8g.quantize_nvfp4(w.B.to(device))
        return w, dict(qa=qa, sa=sa, ga=ga, qb=qb, sb=sb, gb=gb)
    if wl["kind"] == "tensor":
        w = synth.square_tensor(wl["M"], seed=wl["seed"], out="f32" if wl["M"] == 1024 else "bf16")
        bs = 0
    elif wl["M"] == 128:
        w = synth.skinny_block(seed=wl["seed"])
        bs = 32
    else:
        w = synth.large_block(wl["M"], seed=wl["seed"])
        bs = 32
    if wl.get("literal"):
        bs = fp8g.FP8G_BLOCK32_LITERAL
    qa, sa = fp8g.quantize(w.A.to(device), bs, fmt=wl.get("a_fmt", 0))
    qb, sb = fp8g.quantize(w.B.to(device), bs, fmt=wl.get("b_fmt", 0))
    return w, dict(qa=qa, sa=sa, qb=qb, sb=sb)


def algorithmic_bytes(wl: dict, w) -> int:
    """Bytes the call must move: each operand read once, C written once.
    Grouped: only the weights (and scales) of experts that receive rows are
    read; the counts and, from tokens, the routing index are read once."""
    M, N, K = wl["M"], wl["N"], wl["K"]
    out_b = 4 if w.out == "f32" else 2
    ea, eb = FMT_BYTES[wl.get("a_fmt", 0)], FMT_BYTES[wl.get("b_fmt", 0)]
    counts = getattr(w, "counts", None)
    E_all = w.B.shape[0] if w.B.dim() == 3 else 1
    # experts whose weights are read (all of them when the counts are unknown)
    E_used = int((np.asarray(counts) > 0).sum()) if counts is not None else E_all
    if wl["kind"] == "grouped":
        E = E_used
        return int(M * K * ea + E * N * K * eb + 4 * (M * K // 32 + E * N * K // 32) +
                   M * N * out_b + 4 * E_all)
    if wl["kind"] == "grouped_quant":   # bf16 routed rows read once; int32 routing index
        E = E_used
        return int(M * K * 2 + 4 * M + E * N * K * eb + 4 * E * N * K // 32 +
                   M * N * out_b + 4 * E_all)
    if wl["kind"] == "grouped_nvfp4":   # E4M3 scale bytes per 16; fp32 gA and E gB
        E = E_used
        return int(M * K * ea + E * N * K * eb + (M + E * N) * K // 16 + 4 * (1 + E) +
                   M * N * out_b + 4 * E_all)
    if wl["kind"] == "nvfp4":   # E4M3 scale bytes per 16 elements + two fp32 tensor scales
        return int(M * K * ea + N * K * eb + (M + N) * K // 16 + 8 + M * N * out_b)
    sf = 8 if wl["kind"] == "tensor" else 4 * (M * K // 32 + N * K // 32)
    return int(M * K * ea + N * K * eb + sf + M * N * out_b)


def run_once(fp8g, wl, w, t, C, stream):
    out = fp8g.FP8G_OUT_F32 if w.out == "f32" else fp8g.FP8G_OUT_BF16
    if wl["kind"] == "grouped_quant":
        E, N, K = t["qb"].shape
        rows = t["tmp_qa"].shape[0]
        if wl["path"] != "2call":
            fp8g.fp8_grouped_gemm_quant(t["X"], fp8g.FP8G_IN_BF16, t["X"].shape[0], t["idx"],
                                        t["qb"], t["sb"], C, out, fp8g.FP8G_E4M3, None,
                                        fp8g.FP8G_ACT_NONE, t["counts"], E, N, K, rows,
                                        flags=fp8g.FP8G_QUANT_FUSED if wl["path"] == "fused" else 0,
                                        stream=stream)
        else:
            fp8g.fp8g_quantize_rows(t["X"], fp8g.FP8G_IN_BF16, t["X"].shape[0], K, t["idx"], rows,
                                    32, fp8g.FP8G_E4M3, t["tmp_qa"], t["tmp_sa"], stream)
            fp8g.fp8_grouped_gemm(t["tmp_qa"], t["qb"], t["tmp_sa"], t["sb"], C, out,
                                  t["counts"], E, N, K, rows, None, None, stream)
    elif wl["kind"] == "grouped":
        E, N, K = t["qb"].shape
        fp8g.fp8_grouped_gemm(t["qa"], t["qb"], t["sa"], t["sb"], C, out, t["counts"], E, N, K,
                              t["qa"].shape[0], None, None, stream)
    elif wl["kind"] == "grouped_nvfp4":
        E, N, K2 = t["qb"].shape
        fp8g.fp8_grouped_gemm_nvfp4(t["qa"], t["qb"], t["sa"], t["sb"], t["ga"], t["gb"], C, out,
                                    None, fp8g.FP8G_ACT_NONE, t["counts"], E, N, 2 * K2,
                                    t["qa"].shape[0], None, None, stream)
    elif wl["kind"] == "nvfp4":
        fp8g.fp8_gemm_nvfp4(t["qa"], t["qb"], t["sa"], t["sb"], t["ga"], t["gb"], C, out, None,
                            fp8g.FP8G_ACT_NONE, wl["M"], wl["N"], wl["K"], stream)
    elif wl["kind"] == "tensor":
        fp8g.fp8_gemm(t["qa"], t["qb"], t["sa"], t["sb"], C, out, wl["M"], wl["N"], wl["K"], stream)
    elif wl.get("literal"):
        fp8g.fp8_gemm_blockscaled_promote(t["qa"], t["qb"], t["sa"], t["sb"], C, out,
                                          wl.get("a_fmt", 0), wl.get("b_fmt", 0), None,
                                          fp8g.FP8G_ACT_NONE, wl["M"], wl["N"], wl["K"], stream)
    elif "a_fmt" in wl or "b_fmt" in wl:
        fp8g.fp8_gemm_blockscaled_fmt(t["qa"], t["qb"], t["sa"], t["sb"], C, out,
                                      wl.get("a_fmt", 0), wl.get("b_fmt", 0), wl["M"], wl["N"],
                                      wl["K"], stream)
    else:
        fp8g.fp8_gemm_blockscaled(t["qa"], t["qb"], t["sa"], t["sb"], C, out, wl["M"], wl["N"],
                                  wl["K"], stream)


def gemm_alone(fp8g, wl, t, C, stream, prepare=False):
    """The grouped GEMM of a call from tokens on its quantised rows: the
    two-call path's second call; the one-call path runs the same GEMM kernel
    after its quantiser (prepare=True first writes the quantised rows, which
    the one-call path keeps to itself).  None for other workloads."""
    if wl["kind"] != "grouped_quant" or wl["path"] not in ("1call", "2call"):
        return None
    E, N, K = t["qb"].shape
    if prepare:
        fp8g.fp8g_quantize_rows(t["X"], fp8g.FP8G_IN_BF16, t["X"].shape[0], K, t["idx"],
                                t["tmp_qa"].shape[0], 32, fp8g.FP8G_E4M3, t["tmp_qa"],
                                t["tmp_sa"], stream)
        return True
    out = fp8g.FP8G_OUT_BF16 if C.dtype == torch.bfloat16 else fp8g.FP8G_OUT_F32
    fp8g.fp8_grouped_gemm(t["tmp_qa"], t["qb"], t["tmp_sa"], t["sb"], C, out, t["counts"], E, N,
                          K, t["tmp_qa"].shape[0], None, None, stream)
    return True


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# of the dominant kernel, from the ncu captures summarised in profiles/.
# Valid only for the kernel source those captures measured: an entry leaves
# this table when its kernel changes, and workloads without a capture of the
# current kernel report null.
TRAFFIC_BYTES = {"large8192": 257_933_312 + 117_130_752,
                 "mxfp4_8192": 107_267_584 + 95_654_144,
                 "nvfp4_8192": 113_694_976 + 97_257_984,
                 "mxfp6_8192": 167_501_824 + 110_660_864}


def fp4_rate(fp8g, wl) -> bool:
    """Whether the call runs the FP4-rate MMA: E2M1 x E2M1 block-scaled on CTA
    pairs with K % 256 == 0 (the library's own selection rule)."""
    if wl["kind"] in ("nvfp4", "grouped_nvfp4"):
        return True                 # kind::mxf4nvf4 on CTA pairs for every shape
    if wl.get("a_fmt", 0) != 2 or wl.get("b_fmt", 0) != 2 or wl["K"] % 256:
        return False
    if wl["kind"] == "grouped":
        return fp8g.fp8g_grouped_plan(wl["N"], wl["K"], wl["M"], 8)["BM"] == 256
    if wl["kind"] != "block" or wl.get("literal"):
        return False
    return fp8g.fp8g_gemm_plan(1, wl["M"], wl["N"], wl["K"])["BM"] == 256


def tf32_route(fp8g, wl) -> bool:
    """Whether a literal-scale call takes the TF32 route (the library's rule:
    1-byte codes on a shape with a wave of 256 x 256 tiles): two dequantising
    passes, then a kind::tf32 GEMM."""
    return (bool(wl.get("literal")) and wl.get("a_fmt", 0) in (0, 1) and
            wl.get("b_fmt", 0) in (0, 1) and
            fp8g.fp8g_gemm_plan(0, wl["M"], wl["N"], wl["K"])["BM"] == 256)


def launches_per_call(fp8g, wl) -> int:
    """Kernels one call launches: the GEMM, plus the scale-packing kernel on the
    block-scaled plans that take packed scales (split-K, single CTAs on 128 x
    128 tiles and grouped 128 x 128 tiles convert the scales themselves), plus
    the quantiser of the routed rows (grouped calls from tokens)."""
    if wl["kind"] == "tensor":
        return 1
    if wl["kind"] in ("nvfp4", "grouped_nvfp4"):
        return 2
    if wl["kind"] == "grouped":
        # 128 x 128 tiles convert their own scales; CTA pairs take them packed
        return 1 if fp8g.fp8g_grouped_plan(wl["N"], wl["K"], wl["M"], 8)["BM"] == 128 else 2
    if wl["kind"] == "grouped_quant":
        # 128 x 128 tiles: quantiser + GEMM, or (fused) B's scale packing +
        # GEMM; CTA pairs: quantiser, scale packing, GEMM
        return 2 if fp8g.fp8g_grouped_plan(wl["N"], wl["K"], wl["M"], 8)["BM"] == 128 else 3
    if wl.get("literal"):
        return 3 if tf32_route(fp8g, wl) else 1
    plan = fp8g.fp8g_gemm_plan(1, wl["M"], wl["N"], wl["K"])
    return 1 if plan["BM"] == 128 and plan["BN"] == 128 else 2


def e2e_pipelined(fp8g, wl, w, t, C, device, steps, lanes=1):
    """Per-step milliseconds of the end-to-end loop (see the caller).  With
    lanes > 1 each step's copies are split into contiguous chunks over that
    many streams per direction (measured on GB300: 4 lanes were slower, 1086
    against 1197 TFLOPS on the 8192^3 workload; the host link, not one copy
    engine, is the limit)."""
    host = {k: v.cpu().pin_memory() for k, v in t.items() if not k.startswith("tmp_")}
    nbuf = 2
    dev_in = [{k: torch.empty_like(v) for k, v in t.items()} for _ in range(nbuf)]
    dev_C = [C] + [torch.empty_like(C) for _ in range(nbuf - 1)]
    host_C = [torch.empty(C.shape, dtype=C.dtype).pin_memory() for _ in range(nbuf)]
    s_in = [torch.cuda.Stream(device) for _ in range(lanes)]
    s_gemm = torch.cuda.Stream(device)
    s_out = [torch.cuda.Stream(device) for _ in range(lanes)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done = [[ev() for _ in range(lanes)] for _ in range(nbuf)]
    gemm_done = [ev() for _ in range(nbuf)]
    out_done = [[ev() for _ in range(lanes)] for _ in range(nbuf)]
    first = [True] * nbuf

    def chunks(a, b):
        """Matching contiguous pieces of two same-shape tensors, ~lanes per pair."""
        fa, fb = a.reshape(-1), b.reshape(-1)
        n = fa.numel()
        step_ = max(1, -(-n // lanes))
        return [(fa[o:o + step_], fb[o:o + step_]) for o in range(0, n, step_)]

    def step(i):
        b = i % nbuf
        pieces = [p for k in host for p in chunks(dev_in[b][k], host[k])]
        for j, s_ in enumerate(s_in):
            with torch.cuda.stream(s_):
                if not first[b]:
                    s_.wait_event(gemm_done[b])
                for dst, src in pieces[j::lanes]:
                    dst.copy_(src, non_blocking=True)
                in_done[b][j].record(s_)
        for j in range(lanes):
            s_gemm.wait_event(in_done[b][j])
            if not first[b]:
                s_gemm.wait_event(out_done[b][j])
        run_once(fp8g, wl, w, dev_in[b], dev_C[b], s_gemm)
        gemm_done[b].record(s_gemm)
        outs = chunks(host_C[b], dev_C[b])
        for j, s_ in enumerate(s_out):
            with torch.cuda.stream(s_):
                s_.wait_event(gemm_done[b])
                for dst, src in outs[j::lanes]:
                    dst.copy_(src, non_blocking=True)
                out_done[b][j].record(s_)
        first[b] = False

    t0 = time.perf_counter()
    for i in range(2 * nbuf):  # warm-up
        step(i)
    torch.cuda.synchronize(device)
    est = (time.perf_counter() - t0) / (2 * nbuf)
    # 50 pipelined steps (the pipeline's fill and drain, one step's copies
    # each, then weigh 1/50 on the result), fewer for a step above 40 ms
    n = max(20, min(50, int(2.0 / max(est, 1e-6))))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    start = torch.cuda.Stream(device)
    e0.record(start)
    for s_ in s_in:
        s_.wait_stream(start)
    for i in range(n):
        step(i)
    end = torch.cuda.Stream(device)
    for s_ in s_in + s_out + [s_gemm]:
        end.wait_stream(s_)
    e1.record(end)
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / n, n


def oracle_inputs(wl, w):
    """The oracle's own quantisation of the workload (done once, untimed)."""
    import oracle
    if wl["kind"] == "grouped_quant":   # the bf16 tokens, gathered
        import synth
        X, idx, _ = synth.moe_tokens(seed=wl["seed"], tokens=wl["tokens"])
        w = synth.Workload(w.name, w.M, w.N, w.K, True, w.out,
                           X.to(torch.bfloat16).float()[idx.long()], w.B, w.counts)
    if wl["kind"] in ("grouped", "grouped_quant"):
        E, N, K = w.B.shape
        qa, sa = oracle.quantize_block32(w.A.numpy())
        qb, sb = oracle.quantize_block32(w.B.reshape(E * N, K).numpy())
        offs = oracle.grouped_offsets(w.counts)
        e = int(np.argmax(w.counts))                 # the largest expert
        return dict(A=qa[offs[e]:offs[e + 1]], sa=sa[offs[e]:offs[e + 1]],
                    B=qb.reshape(E, N, K)[e], sb=sb.reshape(E, N, K // 32)[e], block=True,
                    N=N, K=K, desc=f"rows of expert {e} (all {N} columns)")
    if wl["kind"] == "grouped_nvfp4":
        N, K = wl["N"], wl["K"]
        offs = oracle.grouped_offsets(w.counts)
        e = int(np.argmax(w.counts))                 # the largest expert
        qa, sa, ga = oracle.quantize_nvfp4(w.A.numpy())
        qb, sb, gb = oracle.quantize_nvfp4(w.B[e].numpy())
        return dict(A=qa[offs[e]:offs[e + 1]], sa=sa[offs[e]:offs[e + 1]], B=qb, sb=sb, ga=ga,
                    gb=gb, nv=True, block=True, N=N, K=K,
                    desc=f"rows of expert {e} (all {N} columns)")
    if wl["kind"] == "nvfp4":
        qa, sa, ga = oracle.quantize_nvfp4(w.A.numpy())
        qb, sb, gb = oracle.quantize_nvfp4(w.B.numpy())
        return dict(A=qa, sa=sa, B=qb, sb=sb, ga=ga, gb=gb, nv=True, block=True, N=wl["N"],
                    K=wl["K"], desc=f"rows of A (all {wl['N']} columns)")
    block = wl["kind"] != "tensor"
    if wl.get("literal"):
        qa, sa = oracle.quantize_block32(w.A.numpy(), wl.get("a_fmt", 0), literal=True)
        qb, sb = oracle.quantize_block32(w.B.numpy(), wl.get("b_fmt", 0), literal=True)
    else:
        qfn = oracle.quantize_block32 if block else oracle.quantize_tensor
        qa, sa = qfn(w.A.numpy(), wl.get("a_fmt", 0))
        qb, sb = qfn(w.B.numpy(), wl.get("b_fmt", 0))
    return dict(A=qa, sa=sa, B=qb, sb=sb, block=block, N=wl["N"], K=wl["K"],
                a_fmt=wl.get("a_fmt", 0), b_fmt=wl.get("b_fmt", 0),
                desc=f"rows of A (all {wl['N']} columns)")


def cpu_baseline(oi: dict, budget_s: float = 12.0):
    """The oracle GEMM as it stands, on this host's cores, over a bounded row
    sample sized to take about budget_s seconds."""
    import oracle
    threads = os.cpu_count() or 1
    N, K, block = oi["N"], oi["K"], oi["block"]
    total_rows = oi["A"].shape[0]
    rows = 1
    spent = 0.0
    while True:
        r = min(rows, total_rows)
        a = np.ascontiguousarray(oi["A"][:r])
        s = np.ascontiguousarray(oi["sa"][:r]) if block else oi["sa"]
        t0 = time.perf_counter()
        if oi.get("nv"):
            oracle.gemm_nvfp4(a, oi["B"], s, oi["sb"], oi["ga"], oi["gb"], oracle.OUT_BF16,
                              threads=threads)
        else:
            oracle.gemm(a, oi["B"], s, oi["sb"], block, oracle.OUT_BF16, threads=threads,
                        a_fmt=oi.get("a_fmt", 0), b_fmt=oi.get("b_fmt", 0))
        dt = time.perf_counter() - t0
        spent += dt
        flops = 2.0 * r * N * K
        if dt > budget_s / 4 or r == total_rows or spent > budget_s:
            break
        rows = int(min(total_rows, max(rows * 2, rows * (budget_s / 3) / max(dt, 1e-3))))
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": f"{r} {oi['desc']}, K={K}: {flops:.3e} FLOP in {dt:.3f} s"}


def config_of(name: str, wl: dict, out: str, world: int) -> dict:
    """The workload's description: the same dict on both arms of the bench."""
    return {"workload": name, "M": wl["M"], "N": wl["N"], "K": wl["K"],
            "formats": FMT_NAMES[wl.get("a_fmt", 0)] + " x " + FMT_NAMES[wl.get("b_fmt", 0)],
            "scales": ("1x32 along K, literal fp32 amax/448" if wl.get("literal") else
                       {"block": "1x32 along K, power of two",
                        "grouped": "1x32 along K, power of two",
                        "grouped_quant": "1x32 along K, power of two; A quantised from bf16 "
                                         "tokens inside the step" + {
                                             "1call": " (one call, two kernels)",
                                             "fused": " (one call, quantiser fused into the "
                                                      "GEMM kernel)",
                                             "2call": " (two calls)"}.get(wl.get("path"), ""),
                        "nvfp4": "1x16 along K, E4M3, and fp32 per tensor (NVFP4)",
                        "grouped_nvfp4": "1x16 along K, E4M3, fp32 for A and per "
                                         "expert weight (NVFP4)",
                        "tensor": "per tensor"}[wl["kind"]]),
            "out": out,
            "l2": "GPU arm: each timed step reads one of several copies of the inputs "
                  "totalling > 2x L2 (count in l2_copies)",
            "parallelism": "replicas" if world > 1 else "1 GPU"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large8192", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    world, rank, local = _dist()
    wl = WORKLOADS[args.workload]

    if args.impl == "reference":
        return reference_arm(args, wl, world, rank)

    import fp8_block_scaled_06_gb300 as fp8g
    fp8g.build()
    fp8g.load()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    w, t = make_inputs(wl, device)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"quantiser status {st}"
    rows = (t["qa"] if "qa" in t else t["tmp_qa"]).shape[0]
    out_dt = torch.float32 if w.out == "f32" else torch.bfloat16
    C = torch.empty((rows, wl["N"]), dtype=out_dt, device=device)
    flops = w.flops
    abytes = algorithmic_bytes(wl, w)

    # rotate over input copies whose total exceeds 2x L2
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    in_bytes = sum(v.numel() * v.element_size() for k, v in t.items()
                   if k != "counts" and not k.startswith("tmp_"))
    copies = max(1, min(8, -(-2 * l2 // max(in_bytes, 1))))
    sets = [t] + [{k: v.clone() for k, v in t.items()} for _ in range(copies - 1)]
    stream = torch.cuda.current_stream(device)

    for i in range(args.warmup):
        run_once(fp8g, wl, w, sets[i % copies], C, stream)
    torch.cuda.synchronize(device)
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"GEMM status {st} detail {detail}"
    # a few more untimed calls give the per-call time that sizes the clock tail
    n_est = max(3, min(20, args.warmup))
    wu0 = torch.cuda.Event(enable_timing=True)
    wu1 = torch.cuda.Event(enable_timing=True)
    wu0.record(stream)
    for i in range(n_est):
        run_once(fp8g, wl, w, sets[i % copies], C, stream)
    wu1.record(stream)
    torch.cuda.synchronize(device)
    call_ms_est = max(wu0.elapsed_time(wu1) / n_est, 1e-3)

    # GPU timeline, back to back: the timed region (K calls); the kernel-timing
    # pass (below); a tail of the same calls, untimed, for TAIL_MS.  Clocks are
    # sampled over all three: a short region (a 20-step run lasts a few ms)
    # holds few samples on its own.  Samples taken while the GPU idled before
    # the region are left out.
    # The GEMM kernel alone (the roofline's "achieved"): the library records
    # CUDA events on the launching stream around each call's GEMM kernel
    # launch (after the scale packing, for block calls); a pass of its own,
    # because the recording keeps the GEMM's prologue from overlapping the
    # packing kernel (calls that launch only the GEMM: the timed region itself
    # is that kernel, and events around each launch would only add launch gaps)
    TAIL_MS = 250.0
    n_tail = int(min(20000, max(1, -(-TAIL_MS // call_ms_est))))
    kpass = launches_per_call(fp8g, wl) > 1
    # calls from tokens whose GEMM is a call of its own that launches only
    # the GEMM kernel (the two-call path's second call; the one-call path
    # runs the same kernel): the kernel pass runs that call back to back,
    # timed over the loop (events around each launch would add a launch gap
    # of a few us to every one)
    alone = (kpass and wl["kind"] == "grouped_quant" and wl["path"] in ("1call", "2call") and
             fp8g.fp8g_grouped_plan(wl["N"], wl["K"], wl["M"], 8)["BM"] == 128)
    nk = max(3, min(args.steps, 300))
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    ev0.record(stream)
    for i in range(args.steps):
        run_once(fp8g, wl, w, sets[i % copies], C, stream)
    ev1.record(stream)
    kms = []
    if alone:
        for i in range(min(copies, nk)):
            gemm_alone(fp8g, wl, sets[i], C, stream, prepare=True)
        ka0 = torch.cuda.Event(enable_timing=True)
        ka1 = torch.cuda.Event(enable_timing=True)
        ka0.record(stream)
        for i in range(nk):
            gemm_alone(fp8g, wl, sets[i % copies], C, stream)
        ka1.record(stream)
    elif kpass:
        fp8g.fp8g_kernel_timing_begin(nk)
        for i in range(nk):
            run_once(fp8g, wl, w, sets[i % copies], C, stream)
    ev1.synchronize()
    wall = time.perf_counter() - wall0
    if alone:
        ka1.synchronize()
        kms = [ka0.elapsed_time(ka1) / nk]
    elif kpass:
        kms = fp8g.fp8g_kernel_timing_end(nk)   # waits for the pass (every call records)
    for i in range(n_tail):
        run_once(fp8g, wl, w, sets[(args.steps + i) % copies], C, stream)
    torch.cuda.synchronize(device)
    wall_end = time.perf_counter()
    if dist is not None:
        dist.barrier()
    region_s = ev0.elapsed_time(ev1) * 1e-3
    clocks = sampler.stop(wall0, wall0 + region_s, wall_end, tail_ms=n_tail * call_ms_est)
    clocks["after_region"] = (f"{nk} kernel-timing calls, then {n_tail} calls"
                              if kpass else f"{n_tail} calls")
    st, detail = fp8g.fp8_gemm_status()
    assert st == 0, f"GEMM status {st} detail {detail}"
    ms = ev0.elapsed_time(ev1) / args.steps
    if dist is not None:
        tt = torch.tensor([ms], device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    kernel_ms = float(np.mean(kms)) if kms else ms

    # end to end through the C ABI with host buffers: every step copies its
    # inputs from pinned host memory, runs the GEMM and copies C back to pinned
    # host memory.  Copies and GEMMs of consecutive steps overlap (copy
    # streams per direction, a compute stream, two device buffers each),
    # ordered by events: step i's GEMM waits for its inputs and for step
    # i - 2's read-back of the same C buffer; step i's input copy waits for
    # step i - 2's GEMM.  Timed from the first copy in to the last copy out,
    # over the whole dependency chain.
    e2e_ms, e2e_steps = e2e_pipelined(fp8g, wl, w, t, C, device, args.steps)
    h2d = sum(v.numel() * v.element_size() for k, v in t.items() if not k.startswith("tmp_"))
    d2h = C.numel() * C.element_size()

    peaks = _peaks()
    # measured bf16 burst x the nominal dense ratio of the MMA kind that runs:
    # FP8 (and E2M1 on the FP8-rate MMA) 2, FP4 (kind::mxf4) 13.5 / 2.25 = 6,
    # TF32 (the literal-scale route) 1.1 / 2.25
    f4 = fp4_rate(fp8g, wl)
    tf32 = tf32_route(fp8g, wl)
    ratio = 6.0 if f4 else (1.1 / 2.25 if tf32 else 2.0)
    sustained, bf16_peak = bf16_peak_for(peaks, region_s)
    tc_peak = round(ratio * bf16_peak, 1)
    tflops = flops / (ms * 1e-3) / 1e12
    hbm_gbs = abytes / (ms * 1e-3) / 1e9
    k_tflops = flops / (kernel_ms * 1e-3) / 1e12
    k_hbm_gbs = abytes / (kernel_ms * 1e-3) / 1e9
    tensor_bound = (flops / (tc_peak * 1e12)) >= (abytes / (peaks["hbm"] * 1e9))
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": round(k_tflops, 1), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(k_tflops / tc_peak, 4),
                "call_achieved": round(tflops, 1), "call_frac": round(tflops / tc_peak, 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(k_hbm_gbs, 1), "peak": peaks["hbm"],
                "unit": "GB/s", "frac": round(k_hbm_gbs / peaks["hbm"], 4),
                "call_achieved": round(hbm_gbs, 1), "call_frac": round(hbm_gbs / peaks["hbm"], 4)}
    roof["traffic"] = TRAFFIC_BYTES.get(args.workload)
    if alone:
        roof["timed"] = (f"GEMM kernel alone: {nk} back-to-back fp8_grouped_gemm calls on the "
                         f"quantised rows (the GEMM kernel their only launch), CUDA events around "
                         f"the loop (a pass right after the timed region); call_* = the whole "
                         f"step (quantiser + GEMM) over the timed region")
    elif kms:
        roof["timed"] = (f"GEMM kernel alone: mean of {len(kms)} launches, CUDA events the "
                         f"library records on the launching stream around the launch (a pass "
                         f"right after the timed region); call_* = the whole call (quantising, "
                         f"packing or dequantising kernels + GEMM kernel) over the timed region")
    else:
        roof["timed"] = "the GEMM kernel (the call's only launch) over the timed region"
    roof["kernel_ms"] = round(kernel_ms, 5)
    kind_ratio = "fp4 = 6" if f4 else ("tf32 = 1.1/2.25" if tf32 else "fp8 = 2")
    roof["peak_source"] = (f"{peaks['src']}: {kind_ratio} x bf16 "
                           f"{'sustained' if sustained else 'burst'} {bf16_peak} TFLOP/s "
                           f"(timed region {region_s:.3f} s)" if tensor_bound else
                           f"{peaks['src']}: HBM copy {peaks['hbm']} GB/s")
    if tf32 and tensor_bound:
        roof["peak_source"] += (" (literal fp32 scales: operands dequantised to TF32, then the "
                                "kind::tf32 GEMM on CTA pairs)")
        fp8_peak = 2.0 * bf16_peak
        roof["call_frac_of_fp8_peak"] = round(tflops / fp8_peak, 4)
    if f4 and tensor_bound:
        roof["peak_source"] += (" (NVFP4: the FP4-rate MMA, kind::mxf4nvf4 scale_vec::4X)"
                                if wl["kind"] in ("nvfp4", "grouped_nvfp4") else
                                " (MXFP4 on CTA pairs: the FP4-rate MMA, kind::mxf4)")
    elif {2, 3, 4} & {wl.get("a_fmt", 0), wl.get("b_fmt", 0)} and tensor_bound:
        roof["peak_source"] += " (E2M1 / FP6 operands on the FP8-rate MMA, kind::f8f6f4)"
    roof["nominal_frac"] = round(max(flops / (13.5e15 if f4 else (1.1e15 if tf32 else 4.5e15)),
                                     abytes / 8e12) /
                                 (kernel_ms * 1e-3), 4)

    line = {
        "metric": METRIC,
        "value": round(tflops * world, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": (FMT_NAMES[wl.get("a_fmt", 0)] + " x " + FMT_NAMES[wl.get("b_fmt", 0)]
                  + " -> f32 accumulate"),
        "data": "synthetic (seeded CPU generators, quantised on the GPU)",
        "config": config_of(args.workload, wl, w.out, world),
        "l2_copies": copies,
        "roofline": roof,
        "achieved_hbm_gbs": round(hbm_gbs, 1),
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12 * world, 2), "unit": "TFLOPS",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "inputs": "the call's own inputs: quantised operand codes and their scales, "
                          "in pinned host memory",
                "overlap": "two buffers, a copy-in, a compute and a copy-out stream: step "
                           "i+1's copy in and step i-1's copy out run during step i's GEMM"},
        "gpu_launches": args.steps * launches_per_call(fp8g, wl),
        "clocks": clocks,
        "wall_s": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(oracle_inputs(wl, w))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def reference_arm(args, wl, world, rank):
    """The oracle, as it stands, on this host's cores: each step is a bounded
    row sample of the same workload, the whole run sized to about a minute."""
    if rank != 0:
        return
    import synth
    if wl["kind"] == "grouped_quant":
        w = synth.moe_tokens(seed=wl["seed"], tokens=wl["tokens"])[2]
    elif "batch" in wl:
        w = synth.skinny_batch(wl["batch"], seed=wl["seed"])
    elif wl["kind"] in ("grouped", "grouped_nvfp4"):
        w = synth.moe_grouped(seed=wl["seed"], experts=wl.get("experts", 8),
                              tokens=wl.get("tokens", 16384))
    elif wl["kind"] == "tensor":
        w = synth.square_tensor(wl["M"], seed=wl["seed"], out="f32" if wl["M"] == 1024 else "bf16")
    elif wl["M"] == 128:
        w = synth.skinny_block(seed=wl["seed"])
    else:
        w = synth.large_block(wl["M"], seed=wl["seed"])   # block, nvfp4
    oi = oracle_inputs(wl, w)
    budget = min(10.0, max(0.01, 60.0 / (args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(oi, budget_s=budget)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cb = cpu_baseline(oi, budget_s=budget)
        vals.append(cb["value"])
    wall = time.perf_counter() - t0
    v = float(np.median(vals))
    line = {"metric": METRIC, "impl": "reference", "value": round(v, 6), "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic (seeded CPU generators)",
            "config": config_of(args.workload, wl, w.out, world),
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOPS", "cores": cb["cores"],
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": round(v, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
