"""Host logic of bench.py that needs no GPU: the algorithmic bytes that are
the numerator of every HBM roofline figure, per workload, against the
per-array sums written out here (A and B at their stored element size, the
scales the call reads, C once), and the workload table's sizes."""
from types import SimpleNamespace

import pytest
import torch

import bench

MiB = 1 << 20


def _w(out="bf16", experts=None, counts=None):
    B = torch.empty((experts, 1, 1)) if experts else torch.empty((1, 1))
    return SimpleNamespace(out=out, B=B, counts=counts)


# name -> (A bytes, B bytes, scale bytes, C bytes), each written out
EXPECTED = {
    # E4M3 8192^3, fp32 1x32 scales of A and B, bf16 C
    "large8192": (64 * MiB, 64 * MiB, 2 * 4 * 8192 * 256, 128 * MiB),
    # per-tensor: two fp32 scales
    "tensor8192": (64 * MiB, 64 * MiB, 8, 128 * MiB),
    # E2M1: half a byte per element
    "mxfp4_8192": (32 * MiB, 32 * MiB, 2 * 4 * 8192 * 256, 128 * MiB),
    # FP6: three quarters of a byte per element
    "mxfp6_8192": (48 * MiB, 48 * MiB, 2 * 4 * 8192 * 256, 128 * MiB),
    # NVFP4: E4M3 scale bytes per 16 elements (4 MiB per operand) + gA, gB
    "nvfp4_8192": (32 * MiB, 32 * MiB, 2 * 4 * MiB + 8, 128 * MiB),
    # skinny 128 x 4096 x 4096
    "skinny": (128 * 4096, 16 * MiB, 4 * (128 + 4096) * 128, 128 * 4096 * 2),
}


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_algorithmic_bytes(name):
    wl = bench.WORKLOADS[name]
    assert bench.algorithmic_bytes(wl, _w()) == sum(EXPECTED[name])


def test_algorithmic_bytes_grouped():
    """MoE: 32768 routed rows, 8 experts of [14336, 4096]; the FP8 form reads
    fp32 1x32 scales and the counts, the NVFP4 form E4M3 scale bytes, gA, the
    8 gB and the counts."""
    rows, E, N, K = 32768, 8, 14336, 4096
    fp8 = rows * K + E * N * K + 4 * (rows + E * N) * K // 32 + rows * N * 2 + 4 * E
    assert bench.algorithmic_bytes(bench.WORKLOADS["moe"], _w(experts=E)) == fp8
    nv = rows * K // 2 + E * N * K // 2 + (rows + E * N) * K // 16 + 4 * (1 + E) + \
        rows * N * 2 + 4 * E
    assert bench.algorithmic_bytes(bench.WORKLOADS["moe_nvfp4"], _w(experts=E)) == nv


def test_workload_table():
    """Every workload is named by its sizes; formats are the library's codes."""
    for name, wl in bench.WORKLOADS.items():
        assert wl["kind"] in ("block", "tensor", "grouped", "nvfp4", "grouped_nvfp4",
                              "grouped_quant"), name
        assert wl.get("a_fmt", 0) in range(5) and wl.get("b_fmt", 0) in range(5), name
        assert wl["M"] > 0 and wl["N"] > 0 and wl["K"] % 32 == 0, name
    assert len(bench.FMT_NAMES) == len(bench.FMT_BYTES) == 5


def test_clock_record_keeps_the_load_window():
    """Samples before the timed region (GPU idle) are left out; the region's
    own samples are counted; throttle reasons come only from the window."""
    def row(mhz, w, slow="Not Active", cap="Not Active"):
        return f"0, {mhz}, 2070, {w}, 0x0, {slow}, Not Active, Not Active, {cap}"
    lines = [(0.00, row(2070, 150, slow="Active")),      # idle, before the region
             (0.10, row(1950, 1300)), (0.11, row(1950, 1350, cap="Active")),
             (0.20, row(1900, 1390)), (0.30, row(1890, 1395)),
             (0.50, row(2070, 160))]                     # after the tail
    c = bench.ClockSampler.summarize(lines, 0.05, 0.12, 0.35, tail_ms=200.0)
    assert c["samples"] == 4 and c["samples_in_timed_region"] == 2
    assert c["sm_mhz"] == 1925.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["power_w_max"] == 1395.0
    assert "200-ms run" in c["window"]


def test_both_arms_describe_the_same_workload():
    for name, wl in bench.WORKLOADS.items():
        a = bench.config_of(name, wl, "bf16", 1)
        assert a == bench.config_of(name, wl, "bf16", 1) and a["workload"] == name
        assert set(a) == {"workload", "M", "N", "K", "formats", "scales", "out", "l2",
                          "parallelism"}


def test_algorithmic_bytes_from_tokens():
    """MoE from bf16 tokens: each routed row's bf16 source read once, the int32
    routing index, the FP8 weights and their fp32 1x32 scales, C, the counts
    (the two-call path's extra write and read of the quantised rows is not
    part of the method's traffic)."""
    E, N, K = 8, 14336, 4096
    for name, rows in (("decode_bf16", 256), ("moe_bf16", 32768)):
        want = rows * K * 2 + 4 * rows + E * N * K + 4 * E * N * K // 32 + rows * N * 2 + 4 * E
        assert bench.algorithmic_bytes(bench.WORKLOADS[name], _w(experts=E)) == want
        two = bench.WORKLOADS[name + "_2call"]
        assert bench.algorithmic_bytes(two, _w(experts=E)) == want and two["path"] == "2call"


def test_algorithmic_bytes_skip_empty_experts():
    """Experts without routed rows: their weights and scales are never read."""
    E, N, K = 8, 14336, 4096
    counts = [208, 16158, 0, 0, 4, 14, 16384, 0]
    rows = sum(counts)
    used = 5
    want = rows * K + used * N * K + 4 * (rows + used * N) * K // 32 + rows * N * 2 + 4 * E
    assert bench.algorithmic_bytes(bench.WORKLOADS["moe"], _w(experts=E, counts=counts)) == want



def test_peak_burst_or_sustained_by_region_length():
    """Short timed regions are measured against the bf16 burst rate, regions
    of a second or more against the sustained rate."""
    peaks = {"bf16": 1901.5, "bf16_sus": 1728.6, "hbm": 6759.2, "src": "measured"}
    assert bench.bf16_peak_for(peaks, 0.007) == (False, 1901.5)
    assert bench.bf16_peak_for(peaks, 0.999) == (False, 1901.5)
    assert bench.bf16_peak_for(peaks, 1.0) == (True, 1728.6)
    assert bench.bf16_peak_for(peaks, 2.1) == (True, 1728.6)
