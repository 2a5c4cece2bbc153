"""Seeded synthetic inputs for the quantizers and GEMMs.

This module only draws random numbers and lays them out; it holds none of the
quantization or GEMM arithmetic. It serves both the CUDA path and the CPU
oracle, so both always see the same bf16 bytes.

Recipe (all on the CPU with ``torch.Generator().manual_seed(seed)``):
  * values are drawn in float32 as N(0, std^2), the outlier entries (a
    fraction of all entries, chosen uniformly without replacement) are
    multiplied by the outlier factor, and the result is rounded to bf16;
  * MoE routing: expert e (rank e+1) has popularity (e+1)^-zipf; every token
    draws ``topk`` distinct experts by Gumbel-top-k over log-popularity; the
    (token, expert) pairs are sorted by expert (then token) and ``m_offsets``
    holds the segment boundaries.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def bf16_normal(shape, std: float = 1.0, seed: int = 0, outlier_frac: float = 0.0,
                outlier_scale: float = 1.0) -> torch.Tensor:
    """bf16 CPU tensor ~ N(0, std^2) with ``round(outlier_frac * numel)`` entries
    multiplied by ``outlier_scale``."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32) * std
    n_out = int(round(outlier_frac * x.numel()))
    if n_out:
        idx = torch.randperm(x.numel(), generator=g)[:n_out]
        x.view(-1)[idx] *= outlier_scale
    return x.to(torch.bfloat16)


def moe_routing(tokens: int, experts: int, topk: int, zipf: float = 1.1, seed: int = 0):
    """Returns (token_of_row int64 [tokens*topk], m_offsets int32 [experts+1]).
    Row r of the expert-sorted activation matrix is token ``token_of_row[r]``."""
    g = torch.Generator().manual_seed(seed)
    logp = -zipf * torch.log(torch.arange(1, experts + 1, dtype=torch.float64))
    u = torch.rand((tokens, experts), generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u))
    chosen = torch.topk(logp[None, :] + gumbel, topk, dim=1).indices  # [tokens][topk]
    tok = torch.arange(tokens).repeat_interleave(topk)
    exp = chosen.reshape(-1)
    order = torch.argsort(exp * tokens + tok)  # by expert, then token
    counts = torch.bincount(exp, minlength=experts)
    offs = torch.zeros(experts + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(counts, 0)
    return tok[order], offs.to(torch.int32)


def dispatch_destinations(rows: torch.Tensor, tokens: int, topk: int) -> torch.Tensor:
    """The inverse of the routing permutation: dest[t][j] is the expert-ordered
    row of token t's j-th copy (rows lists the token of each expert-ordered row;
    every token appears exactly topk times)."""
    order = torch.argsort(rows, stable=True)
    return order.to(torch.int32).view(tokens, topk)


@dataclass
class GemmProblem:
    """Logical problem: D[M][N] = A[M][K] . W[K][N] (A row-major, W input-major)."""
    name: str
    M: int
    N: int
    K: int
    a_std: float
    w_std: float
    a_outlier_frac: float
    a_outlier_scale: float
    out: str  # "bf16" | "f32"
    seed: int = 0

    def make(self):
        a = bf16_normal((self.M, self.K), self.a_std, self.seed, self.a_outlier_frac,
                        self.a_outlier_scale)
        w = bf16_normal((self.K, self.N), self.w_std, self.seed + 1)
        return a, w

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


# The workloads the library is measured and checked on.
TINY = GemmProblem("tiny 256x256x512", 256, 256, 512, 1.0, 0.02, 0.001, 100.0, "f32")
DENSE_FWD = GemmProblem("dense forward 8192x7168x7168", 8192, 7168, 7168, 1.0, 0.02,
                        0.001, 50.0, "bf16")
SQUARE_8K = GemmProblem("square 8192x8192x8192", 8192, 8192, 8192, 1.0, 0.02, 0.001, 50.0,
                        "bf16")


@dataclass
class DgradProblem:
    """dX[T][Cin] = dY[T][Cout] . W[Cin][Cout]^T, the input gradient of the dense
    forward Linear: W is the forward's weight (same seed and shape), dY ~ N(0, 1e-3^2)."""
    T: int = 8192
    Cin: int = 7168
    Cout: int = 7168
    seed: int = 0

    @property
    def name(self):
        return f"dgrad T={self.T} Cin={self.Cin} Cout={self.Cout}"

    def make(self):
        dy = bf16_normal((self.T, self.Cout), 1e-3, self.seed + 2)
        w = bf16_normal((self.Cin, self.Cout), 0.02, self.seed + 1)
        return dy, w

    @property
    def flops(self) -> float:
        return 2.0 * self.T * self.Cin * self.Cout


def ksweep_problem(K: int) -> GemmProblem:
    return GemmProblem(f"k-sweep 4096x4096x{K}", 4096, 4096, K, 1.0, 1.0, 0.0, 1.0, "f32")


def ksweep_operand(rows: int, K: int, seed: int) -> torch.Tensor:
    """bf16 [rows][K] ~ N(0, 1) clipped to +-6, with the first entry of every
    128-element row tile set to 6. Every 1x128 tile then has max-abs exactly 6,
    so power-of-two tile scales are all 2^-6: one scale for the whole tensor,
    which is what the accumulation study needs (the promoted and the
    tensor-core-only GEMM then see identical codes and constant scales)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, K), generator=g, dtype=torch.float32).clamp_(-6.0, 6.0)
    x[:, ::128] = 6.0
    return x.to(torch.bfloat16)


@dataclass
class MoeProblem:
    """MoE up-projection: E experts with W_e [K][N]; tokens x topk routed rows."""
    tokens: int = 16384
    experts: int = 16
    topk: int = 9
    K: int = 7168
    N: int = 2048
    zipf: float = 1.1
    seed: int = 0

    @property
    def name(self):
        return (f"moe grouped up-projection {self.experts} experts, {self.tokens} tokens "
                f"top-{self.topk}, K={self.K} N={self.N}")

    def make(self):
        x = bf16_normal((self.tokens, self.K), 1.0, self.seed)
        w = torch.stack([bf16_normal((self.K, self.N), 0.02, self.seed + 1 + e)
                         for e in range(self.experts)])  # [E][K][N]
        rows, offs = moe_routing(self.tokens, self.experts, self.topk, self.zipf, self.seed)
        return x, w, rows, offs

    @property
    def rows(self):
        return self.tokens * self.topk

    @property
    def flops(self) -> float:
        return 2.0 * self.rows * self.N * self.K


# Small-M MoE decode: 256 tokens x top-9 over 16 experts (at most 256 rows per
# expert); reading the expert weights dominates.
MOE_DECODE = MoeProblem(tokens=256)


@dataclass
class MoeActGradProblem:
    """Gradient of the MoE down-projection input, [tokens x topk][N] bf16 ~ N(0, 1e-3^2),
    in expert order: quantized 1x128 along N with power-of-two scales before the
    down-projection's backward GEMMs."""
    rows: int = 16384 * 9
    N: int = 2048
    seed: int = 0

    @property
    def name(self):
        return f"moe activation gradient [{self.rows}][{self.N}]"

    def make(self):
        return bf16_normal((self.rows, self.N), 1e-3, self.seed + 5)


@dataclass
class WgradProblem:
    """dW[Cin][Cout] = X^T . dY over T tokens."""
    T: int = 16384
    C: int = 7168
    seed: int = 0

    @property
    def name(self):
        return f"wgrad T={self.T} C={self.C}"

    def make(self):
        x = bf16_normal((self.T, self.C), 1.0, self.seed)
        dy = bf16_normal((self.T, self.C), 1e-3, self.seed + 1)
        return x, dy

    @property
    def flops(self) -> float:
        return 2.0 * self.C * self.C * self.T
