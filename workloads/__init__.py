"""Seeded synthetic inputs for the orthonormalized optimizer step.

This module holds the workload shapes and the random-input recipe, and nothing
of the method's arithmetic.  Both the CUDA path's tests/benchmark and the
oracle's comparisons draw their inputs from here, so both sides see the same
stored values.

Shapes follow the workloads the talk page describes ("Dion: The distributed
orthonormal update revolution is here": a square-matrix microbenchmark at rank
fractions 1/4 and 1/16, and a Llama 3 405B dense configuration) together with a
GPT-small stack and a Llama-3-8B stack.  Inputs are Gaussian: weights
X ~ N(0, 0.02^2), gradients G ~ N(0, g_std^2), momentum M = 0 at the first
step, and the initial right factor Q0 ~ N(0, 1) with unit-norm columns.  X and
G are stored in the workload's dtype (fp32 or bf16); M and Q are fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch


@dataclass(frozen=True)
class Group:
    """A megabatch: `batch` same-shape m x n matrices."""
    batch: int
    m: int
    n: int
    head_dim: int = 0          # > 0: per-head Newton-Schulz on column blocks

    def rank(self, fraction: float) -> int:
        return max(1, int(fraction * min(self.m, self.n)))

    @property
    def elems(self) -> int:
        return self.batch * self.m * self.n


@dataclass(frozen=True)
class Workload:
    name: str
    groups: Tuple[Group, ...]
    dtype: torch.dtype
    fraction: float
    g_std: float
    x_std: float = 0.02
    mu: float = 0.95
    lr: float = 0.01
    wd: float = 0.01
    steps: int = 1
    ns_steps: int = 5
    extra_fractions: Tuple[float, ...] = field(default_factory=tuple)

    @property
    def params(self) -> int:
        return sum(g.elems for g in self.groups)


def gpt_small() -> Workload:
    L = 12
    return Workload("gpt-small-megabatch",
                    (Group(L, 768, 2304, head_dim=64), Group(L, 768, 768),
                     Group(L, 768, 3072), Group(L, 3072, 768)),
                    torch.bfloat16, 0.25, 1e-3)


def single_256() -> Workload:
    return Workload("single-256x256-fp32", (Group(1, 256, 256),), torch.float32, 0.25, 1.0,
                    steps=10)


def square(n: int) -> Workload:
    return Workload(f"square-{n}x{n}-batch8", (Group(8, n, n),), torch.bfloat16, 0.25, 1.0,
                    extra_fractions=(1.0 / 16,))


def llama3_8b() -> Workload:
    L = 32
    return Workload("llama3-8b-megabatch",
                    (Group(2 * L, 4096, 4096), Group(2 * L, 4096, 1024),
                     Group(2 * L, 4096, 14336), Group(L, 14336, 4096)),
                    torch.bfloat16, 1.0 / 16, 1e-3)


def llama3_405b_layer() -> Workload:
    return Workload("llama3-405b-layer",
                    (Group(2, 16384, 16384), Group(2, 16384, 1024),
                     Group(2, 16384, 53248), Group(1, 53248, 16384)),
                    torch.bfloat16, 1.0 / 16, 1.0)


WORKLOADS = {
    "single-256x256-fp32": single_256,
    "gpt-small-megabatch": gpt_small,
    "llama3-8b-megabatch": llama3_8b,
    "llama3-405b-layer": llama3_405b_layer,
    **{f"square-{n}x{n}-batch8": (lambda n=n: square(n)) for n in (1024, 2048, 4096, 8192, 16384)},
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, std: float, dtype, device, seed: int) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 from a seeded generator, then stored in dtype."""
    t = torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def init_q(batch: int, n: int, r: int, device, seed: int) -> torch.Tensor:
    """Initial right factor: N(0, 1) entries, each column scaled to unit norm."""
    q = torch.randn((batch, n, r), generator=_gen(device, seed), device=device,
                    dtype=torch.float32)
    q.div_(q.norm(dim=1, keepdim=True))
    return q


def make_state(group: Group, r: int, dtype, device, seed: int, x_std: float = 0.02):
    """Fresh optimizer state for one megabatch: X, M = 0 and Q0."""
    b, m, n = group.batch, group.m, group.n
    X = randn((b, m, n), x_std, dtype, device, seed * 7 + 1)
    M = torch.zeros((b, m, n), dtype=torch.float32, device=device)
    Q = init_q(b, n, r, device, seed * 7 + 2)
    return X, M, Q


def make_grad(group: Group, std: float, dtype, device, seed: int, step: int) -> torch.Tensor:
    """Gradient for one step, fresh per step from (seed, step)."""
    return randn((group.batch, group.m, group.n), std, dtype, device, seed * 1000 + step)


def make_momentum(group: Group, std: float, device, seed: int) -> torch.Tensor:
    """A non-zero momentum buffer (for teacher-forced steps past the first)."""
    return randn((group.batch, group.m, group.n), std, torch.float32, device, seed * 7 + 3)
