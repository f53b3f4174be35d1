"""Seeded synthetic workloads shared by the CUDA path's tests/bench and the oracle.

This module holds none of the method's arithmetic: it draws the real-valued
(fp32) operands, routing counts and exact-case matrices only.  Quantisation,
scaling and the GEMM itself happen on each side separately (the CUDA library's
quantiser kernel and the CPU oracle's quantiser).

Recipe (all CPU, torch.Generator / numpy PCG64, so every run sees the same data):

- seed per workload; operand A draws from ``seed``, B from ``seed + 1000``,
  masks / permutations / row factors from ``seed + 2000``; the MoE routing
  counts draw from numpy PCG64(``seed``);
- square per-tensor case: A, B ~ N(0, 1);
- exact cases: B = identity, or B = a permutation matrix (1 at (n, pi(n)));
- skinny case: A, B ~ N(0, 1), row n of B multiplied by 10^U(-2, 2) (outlier rows);
- large case: N(0, 1) with each element independently multiplied by 50 with
  probability 0.001 (outliers), for both operands;
- MoE case: 8 experts, 16384 tokens routed top-2; expert token counts from a
  Zipf(1.2) draw normalised to 32768 slots, capped at 16384 per expert (a token
  cannot take one expert twice), excess handed out pro rata, then floor plus
  largest remainder (ties to the lower expert index).  Token t fills slots t and
  t + 16384, so the grouped activation matrix is the token matrix twice; expert
  weights B[e] ~ N(0, 0.02).

These mirror the workload descriptions of the FP8 GEMM pages (square FP8 GEMM,
skinny M=128, N=K=4096 memory-bound GEMM, large block-scaled GEMM with
outliers, MoE grouped GEMM with near-empty experts).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    """fp32 N(0, std^2) on the CPU."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def with_outliers(x: torch.Tensor, g: torch.Generator, p: float = 1e-3,
                  factor: float = 50.0) -> torch.Tensor:
    """Multiply each element by ``factor`` independently with probability p."""
    mask = torch.rand(x.shape, generator=g) < p
    return torch.where(mask, x * factor, x)


def permutation(n: int, seed: int) -> torch.Tensor:
    return torch.randperm(n, generator=_gen(seed))


def identity(n: int) -> torch.Tensor:
    return torch.eye(n, dtype=torch.float32)


def permutation_matrix(n: int, seed: int) -> torch.Tensor:
    """B[j, pi(j)] = 1."""
    pi = permutation(n, seed)
    B = torch.zeros(n, n, dtype=torch.float32)
    B[torch.arange(n), pi] = 1.0
    return B


def moe_counts(seed: int, experts: int = 8, tokens: int = 16384, topk: int = 2) -> np.ndarray:
    """Expert slot counts from a Zipf(1.2) draw, summing to tokens * topk."""
    z = np.random.Generator(np.random.PCG64(seed)).zipf(1.2, size=experts).astype(np.float64)
    total = tokens * topk
    cap = tokens
    capped = np.zeros(experts, dtype=bool)
    w = z / z.sum() * total
    while True:
        over = (w > cap) & ~capped
        if not over.any():
            break
        capped |= over
        free = ~capped
        w[capped] = cap
        rest = total - cap * int(capped.sum())
        w[free] = z[free] / z[free].sum() * rest
    fl = np.floor(w).astype(np.int64)
    left = total - int(fl.sum())
    frac = w - fl
    order = sorted(range(experts), key=lambda e: (-frac[e], e))
    for e in order[:left]:
        fl[e] += 1
    assert int(fl.sum()) == total and int(fl.max()) <= cap
    return fl.astype(np.int32)


@dataclass
class Workload:
    """Real-valued operands of one GEMM workload (CPU fp32)."""
    name: str
    M: int
    N: int
    K: int
    block: bool          # 1x32 block scales along K (else per-tensor)
    out: str             # "bf16" or "f32"
    A: torch.Tensor      # [M, K]  (grouped: [sum M_e, K])
    B: torch.Tensor      # [N, K]  (grouped: [E, N, K])
    counts: np.ndarray | None = None
    extra: dict = field(default_factory=dict)

    @property
    def flops(self) -> float:
        rows = int(self.counts.sum()) if self.counts is not None else self.M
        return 2.0 * rows * self.N * self.K


def square_tensor(n: int = 256, seed: int = 0, out: str = "bf16") -> Workload:
    """Per-tensor-scaled square GEMM, N(0,1) operands."""
    return Workload(f"square{n}_tensor", n, n, n, False, out,
                    normal((n, n), seed), normal((n, n), seed + 1000))


def exact_cases(n: int = 1024, seed: int = 1) -> dict:
    """Identity and permutation B for the n^3 per-tensor case (A ~ N(0,1))."""
    A = normal((n, n), seed)
    return {"identity": identity(n), "permutation": permutation_matrix(n, seed + 2000), "A": A}


def skinny_block(M: int = 128, N: int = 4096, K: int = 4096, seed: int = 2,
                 out: str = "bf16") -> Workload:
    """Memory-bound skinny GEMM: rows of B scaled by 10^U(-2,2)."""
    A = normal((M, K), seed)
    B = normal((N, K), seed + 1000)
    g = _gen(seed + 2000)
    u = torch.rand(N, generator=g) * 4.0 - 2.0
    B.mul_(torch.pow(10.0, u).unsqueeze(1))
    return Workload(f"skinny{M}x{N}x{K}_block", M, N, K, True, out, A, B)


def large_block(n: int = 8192, seed: int = 3, out: str = "bf16", M: int | None = None,
                N: int | None = None, K: int | None = None) -> Workload:
    """Large block-scaled GEMM: N(0,1) with 0.1% of elements x50, both operands."""
    M = M or n
    N = N or n
    K = K or n
    g = _gen(seed + 2000)
    A = with_outliers(normal((M, K), seed), g)
    B = with_outliers(normal((N, K), seed + 1000), g)
    return Workload(f"gemm{M}x{N}x{K}_block", M, N, K, True, out, A, B)


def moe_grouped(seed: int = 4, experts: int = 8, tokens: int = 16384, N: int = 14336,
                K: int = 4096, out: str = "bf16", counts: np.ndarray | None = None) -> Workload:
    """MoE grouped GEMM: top-2 routing with Zipf(1.2) counts, B[e] ~ N(0, 0.02)."""
    if counts is None:
        counts = moe_counts(seed, experts, tokens)
    counts = np.asarray(counts, dtype=np.int32)
    rows = int(counts.sum())
    A_tok = normal((tokens, K), seed)
    idx = torch.arange(rows) % tokens
    A = A_tok[idx].contiguous()
    B = normal((experts, N, K), seed + 1000, std=0.02)
    return Workload(f"moe{experts}x{N}x{K}_grouped", rows, N, K, True, out, A, B, counts)


def small_grouped(counts, N: int, K: int, seed: int = 7, out: str = "bf16") -> Workload:
    """Small grouped case with given counts (tests)."""
    counts = np.asarray(counts, dtype=np.int32)
    rows = int(counts.sum())
    A = normal((max(rows, 0), K), seed)
    B = normal((counts.size, N, K), seed + 1000, std=0.02)
    return Workload(f"grouped{counts.size}x{N}x{K}", rows, N, K, True, out, A, B, counts)


def moe_tokens(seed: int = 4, experts: int = 8, tokens: int = 16384, N: int = 14336,
               K: int = 4096, out: str = "bf16"):
    """The MoE workload before routing: token activations X [tokens, K] (the
    rows moe_grouped gathers), the routed-row -> token index (routed row r of
    the expert-ordered list takes token r % tokens: each token's two slots are
    rows t and t + tokens), and the grouped workload itself (counts, B)."""
    w = moe_grouped(seed, experts, tokens, N, K, out)
    X = normal((tokens, K), seed)
    idx = (torch.arange(w.M) % tokens).to(torch.int32)
    return X, idx, w


def skinny_batch(count: int = 8, seed: int = 2, M: int = 128, N: int = 4096, K: int = 4096,
                 out: str = "bf16") -> Workload:
    """`count` independent skinny products (the skinny_block recipe, problem i
    drawn with seed + i), laid out as a grouped workload: A rows of problem i
    at [i M, (i + 1) M), its B as B[i], counts M each."""
    parts = [skinny_block(M, N, K, seed + i, out) for i in range(count)]
    A = torch.cat([w.A for w in parts])
    B = torch.stack([w.B for w in parts])
    counts = np.full(count, M, dtype=np.int32)
    return Workload(f"skinny{count}x{M}x{N}x{K}_batch", count * M, N, K, True, out, A, B, counts)

