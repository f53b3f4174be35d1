"""The seeded workload generators (no method arithmetic): determinism, the
MoE routing-count procedure and the shapes of the pages' workloads."""
import numpy as np
import torch

import synth


def test_moe_counts_pin_and_invariants():
    # seed 0 of the Zipf(1.2) procedure (normalise to 32768 slots, cap 16384,
    # largest remainder with ties to the lower expert)
    assert synth.moe_counts(0).tolist() == [120, 1, 3570, 12806, 523, 15743, 4, 1]
    for seed in range(10):
        c = synth.moe_counts(seed)
        assert c.sum() == 32768 and c.max() <= 16384 and c.min() >= 0 and c.size == 8


def test_generators_are_deterministic():
    a = synth.large_block(64, seed=3)
    b = synth.large_block(64, seed=3)
    assert torch.equal(a.A, b.A) and torch.equal(a.B, b.B)
    assert a.A.shape == (64, 64) and a.block and a.out == "bf16"
    s = synth.skinny_block(M=8, N=64, K=64)
    assert s.B.abs().amax(dim=1).min() > 0
    e = synth.exact_cases(16)
    assert torch.equal(e["identity"], torch.eye(16))
    P = e["permutation"]
    assert torch.equal(P.sum(0), torch.ones(16)) and torch.equal(P.sum(1), torch.ones(16))


def test_outlier_rate():
    g = torch.Generator().manual_seed(0)
    x = torch.ones(1000, 1000)
    y = synth.with_outliers(x, g)
    frac = float((y == 50).float().mean())
    assert 0.0007 < frac < 0.0013


def test_moe_workload_shape_small():
    w = synth.moe_grouped(counts=np.array([3, 0, 5], np.int32), experts=3, tokens=4, N=16, K=32)
    assert w.A.shape == (8, 32) and w.B.shape == (3, 16, 32)
    # token t fills slots t and t + tokens: the grouped matrix repeats token rows
    assert torch.equal(w.A[0], w.A[4])
    assert w.flops == 2.0 * 8 * 16 * 32
