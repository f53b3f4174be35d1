"""Multi-rank partition logic on CPU (gloo, world_size 2).

The GEMM shards without any exchange: output tiles are independent, so ranks
can split N (rows of B / columns of C), or take disjoint experts of a grouped
GEMM, and the concatenation of their outputs is the unsharded result.  The
library runs one process per GPU as replicas; this checks the partition
arithmetic with the oracle on two gloo ranks: each rank computes its shard,
the shards are gathered, and the result must equal the unsharded oracle bit
for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def n_shard(N: int, world: int, rank: int, align: int = 8):
    """Contiguous split of N columns, each shard a multiple of `align` except the last."""
    per = -(-N // world)
    per = -(-per // align) * align
    lo = min(N, rank * per)
    hi = min(N, lo + per)
    return lo, hi


def expert_shard(counts, world: int, rank: int):
    """Greedy contiguous expert ranges balancing routed rows."""
    counts = np.asarray(counts)
    target = counts.sum() / world
    bounds = [0]
    acc = 0
    for e, c in enumerate(counts):
        acc += c
        if len(bounds) < world and acc >= target * len(bounds):
            bounds.append(e + 1)
    while len(bounds) < world:
        bounds.append(len(counts))
    bounds.append(len(counts))
    return bounds[rank], bounds[rank + 1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    rng = np.random.default_rng(0)                     # same data on every rank
    M, N, K = 24, 72, 64
    A = rng.integers(0, 0x7E, size=(M, K), dtype=np.uint8)
    B = rng.integers(0, 0x7E, size=(N, K), dtype=np.uint8)
    sfa = (2.0 ** rng.integers(-4, 4, size=(M, K // 32))).astype(np.float32)
    sfb = (2.0 ** rng.integers(-4, 4, size=(N, K // 32))).astype(np.float32)
    lo, hi = n_shard(N, world, rank)
    C_part, _, _ = oracle.gemm(A, B[lo:hi], sfa, sfb[lo:hi], True, oracle.OUT_BF16, threads=1)
    parts = [None] * world
    dist.all_gather_object(parts, (lo, hi, C_part))

    counts = np.array([5, 0, 9, 3, 7], np.int32)
    E = counts.size
    rows = int(counts.sum())
    Ag = rng.integers(0, 0x7E, size=(rows, K), dtype=np.uint8)
    Bg = rng.integers(0, 0x7E, size=(E, 16, K), dtype=np.uint8)
    sfa_g = np.ones((rows, K // 32), np.float32)
    sfb_g = (2.0 ** rng.integers(-2, 2, size=(E, 16, K // 32))).astype(np.float32)
    e0, e1 = expert_shard(counts, world, rank)
    off = oracle.grouped_offsets(counts)
    r0, r1 = int(off[e0]), int(off[e1])
    Cg, _, _ = oracle.grouped_gemm(Ag[r0:r1], Bg[e0:e1], sfa_g[r0:r1], sfb_g[e0:e1],
                                   counts[e0:e1], threads=1) if e1 > e0 else (
        np.zeros((0, 16), np.float32), None, None)
    gparts = [None] * world
    dist.all_gather_object(gparts, (r0, r1, Cg))
    if rank == 0:
        full, _, _ = oracle.gemm(A, B, sfa, sfb, True, oracle.OUT_BF16, threads=1)
        cat = np.concatenate([p[2] for p in sorted(parts, key=lambda p: p[0])], axis=1)
        fullg, _, _ = oracle.grouped_gemm(Ag, Bg, sfa_g, sfb_g, counts, threads=1)
        catg = np.concatenate([p[2] for p in sorted(gparts, key=lambda p: p[0])], axis=0)
        q.put((np.array_equal(cat, full), np.array_equal(catg, fullg),
               [p[:2] for p in parts], [p[:2] for p in gparts]))
    dist.barrier()
    dist.destroy_process_group()


def test_shard_helpers_cover_exactly():
    for N in (8, 72, 4096, 14336, 100):
        for world in (1, 2, 3, 8):
            cover = []
            for r in range(world):
                lo, hi = n_shard(N, world, r)
                cover.extend(range(lo, hi))
            assert cover == list(range(N))
    counts = [120, 1, 3570, 12806, 523, 15743, 4, 1]
    for world in (1, 2, 4, 8):
        ex = []
        for r in range(world):
            e0, e1 = expert_shard(counts, world, r)
            ex.extend(range(e0, e1))
        assert ex == list(range(len(counts)))


def test_two_gloo_ranks_shard_equals_unsharded(oracle_lib):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ok_n, ok_g, n_parts, g_parts = res
    assert ok_n, f"N-sharded GEMM differs ({n_parts})"
    assert ok_g, f"expert-sharded grouped GEMM differs ({g_parts})"
