"""Seeded synthetic workloads for the OKLS step (inputs only).

This module holds the shapes, dtypes and gradient recipes of the benchmark
and test workloads and nothing of the optimizer's arithmetic.  Both the CUDA
path (tests, bench) and the float64 oracle (tests) draw their inputs here.

Workloads (the layer shapes come from the pages: the Llama-1.3B shape table of
the "Clean" paper (hidden 2048, intermediate 5461 rounded up to 5504) and the
4096 x 11008 layer of the optim-book's Shampoo chapter, Problem 15):

  single128x64   one 128 x 64 fp32 matrix, G iid N(0,1), seed 0, 20 steps
  batch16x512    16 square 512 x 512 fp32 matrices, Kronecker gradients
                 G = A^1/2 Z B^1/2, A and B SPD with log-uniform spectra on
                 [1, 100] (endpoints pinned), seed 1, 50 steps
  llama1.2b      24 layers x {q,k,v,o 2048x2048; gate,up 5504x2048;
                 down 2048x5504} = 168 matrices in 3 shape groups, Kronecker
                 gradients with condition number 1e3, bf16 W and G, seed 2,
                 10 steps
  rect8192       32 x (8192 x 1024) + 32 x (1024 x 8192), G_ij = r_i z_ij,
                 z iid N(0,1), r_i = exp(N(0,1)) fixed per row, seed 3, 10 steps
  llama7b_slice  8 layers x {q,k,v,o 4096x4096; gate,up 11008x4096;
                 down 4096x11008} = 56 matrices, Kronecker gradients with
                 condition number 1e4 and Student-t (nu = 3) entries of Z,
                 seed 5, 5 steps

W_0 is drawn by the README's spectral-muP Gaussian initialisation
(std = sigma* sqrt(n_out/n_in) / (sqrt(n_in) + sqrt(n_out)), sigma* = 0.07539)
with seed + 1000.

`scale` shrinks every dimension by an integer factor (rounded up to a
multiple of 8) for parity tests that must finish on the CPU oracle.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

INIT_OPERATOR_NORM = 0.07539


@dataclass
class Group:
    """One same-shape batch: `batch` matrices of m x n (W and G dtype)."""
    name: str
    batch: int
    m: int
    n: int
    dtype: torch.dtype


@dataclass
class Workload:
    name: str
    groups: list[Group]
    steps: int
    seed: int
    recipe: str                 # "iid" | "kron" | "rowscale"
    cond: float = 1.0
    student_t: float = 0.0      # nu of the Student-t entries (0 = Gaussian)
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def matrices(self) -> int:
        return sum(g.batch for g in self.groups)


def _r8(x: int) -> int:
    return max(8, ((x + 7) // 8) * 8)


def workload(name: str, scale: int = 1, layers: int | None = None) -> Workload:
    """The named workload; `scale` divides every dimension, `layers`
    overrides the layer count of the Llama-shaped sets."""
    s = lambda d: d if scale == 1 else _r8(d // scale)  # noqa: E731
    if name == "single128x64":
        return Workload(name, [Group("w", 1, s(128), s(64), torch.float32)],
                        steps=20, seed=0, recipe="iid")
    if name == "batch16x512":
        return Workload(name, [Group("w", 16, s(512), s(512), torch.float32)],
                        steps=50, seed=1, recipe="kron", cond=100.0)
    if name == "llama1.2b":
        L = 24 if layers is None else layers
        h, f = s(2048), s(5504)
        return Workload(name, [
            Group("qkvo", 4 * L, h, h, torch.bfloat16),
            Group("gate_up", 2 * L, f, h, torch.bfloat16),
            Group("down", L, h, f, torch.bfloat16)],
            steps=10, seed=2, recipe="kron", cond=1e3)
    if name == "rect8192":
        return Workload(name, [
            Group("tall", 32, s(8192), s(1024), torch.float32),
            Group("wide", 32, s(1024), s(8192), torch.float32)],
            steps=10, seed=3, recipe="rowscale")
    if name == "llama7b_slice":
        L = 8 if layers is None else layers
        h, f = s(4096), s(11008)
        return Workload(name, [
            Group("qkvo", 4 * L, h, h, torch.float32),
            Group("gate_up", 2 * L, f, h, torch.float32),
            Group("down", L, h, f, torch.float32)],
            steps=5, seed=5, recipe="kron", cond=1e4, student_t=3.0)
    raise KeyError(name)


WORKLOADS = ["single128x64", "batch16x512", "llama1.2b", "rect8192",
             "llama7b_slice"]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def spectral_mup_init(batch: int, m: int, n: int, seed: int, device="cpu",
                      dtype=torch.float32) -> torch.Tensor:
    """W ~ N(0, std^2), std = sigma* sqrt(m/n) / (sqrt(n) + sqrt(m)) with
    m = n_out (rows), n = n_in (cols)."""
    std = INIT_OPERATOR_NORM * math.sqrt(m / n) / (math.sqrt(n) + math.sqrt(m))
    w = torch.randn(batch, m, n, generator=_gen(device, seed), device=device,
                    dtype=torch.float32) * std
    return w.to(dtype)


def _spd_sqrt(batch: int, d: int, cond: float, gen, device) -> torch.Tensor:
    """Square roots of SPD matrices Q diag(w) Q^T, w log-uniform on
    [1, cond] with both endpoints present, Q from a QR of a Gaussian."""
    Q, _ = torch.linalg.qr(torch.randn(batch, d, d, generator=gen,
                                       device=device, dtype=torch.float32))
    u = torch.rand(batch, d, generator=gen, device=device, dtype=torch.float32)
    u[:, 0] = 0.0
    if d > 1:
        u[:, -1] = 1.0
    w = torch.exp(u * math.log(cond))
    return (Q * w.sqrt().unsqueeze(1)) @ Q.transpose(1, 2)


class GradientStream:
    """Per-group gradient generator; step t (1-based) is reproducible from
    (seed, group index, t) alone."""

    def __init__(self, wl: Workload, device="cpu"):
        self.wl = wl
        self.device = torch.device(device)
        self.fixed = []
        for gi, g in enumerate(wl.groups):
            gen = _gen(self.device, wl.seed * 7919 + gi)
            if wl.recipe == "kron":
                A = _spd_sqrt(g.batch, g.m, wl.cond, gen, self.device)
                B = _spd_sqrt(g.batch, g.n, wl.cond, gen, self.device)
                self.fixed.append((A, B))
            elif wl.recipe == "rowscale":
                r = torch.exp(torch.randn(g.batch, g.m, 1, generator=gen,
                                          device=self.device))
                self.fixed.append((r,))
            else:
                self.fixed.append(())

    def _z(self, g: Group, gen) -> torch.Tensor:
        z = torch.randn(g.batch, g.m, g.n, generator=gen, device=self.device)
        nu = self.wl.student_t
        if nu > 0:
            # Student-t: N(0,1) / sqrt(chi2_nu / nu), chi2 from nu normals
            k = int(round(nu))
            chi = torch.zeros(g.batch, g.m, g.n, device=self.device)
            for _ in range(k):
                e = torch.randn(g.batch, g.m, g.n, generator=gen,
                                device=self.device)
                chi += e * e
            z = z / torch.sqrt(chi / nu)
        return z

    def grad(self, gi: int, t: int) -> torch.Tensor:
        g = self.wl.groups[gi]
        gen = _gen(self.device, (self.wl.seed * 1_000_003 + gi * 10_007 + t)
                   % (2 ** 62))
        z = self._z(g, gen)
        if self.wl.recipe == "kron":
            A, B = self.fixed[gi]
            G = A @ z @ B
        elif self.wl.recipe == "rowscale":
            G = self.fixed[gi][0] * z
        else:
            G = z
        return G.to(g.dtype)

    def init_weights(self, gi: int) -> torch.Tensor:
        g = self.wl.groups[gi]
        return spectral_mup_init(g.batch, g.m, g.n, self.wl.seed + 1000 + gi,
                                 self.device, g.dtype)


def hand_example_gradient() -> torch.Tensor:
    """The optim-book's 2 x 3 gradient (output 2 x input 3)."""
    return torch.tensor([[3.0, 0.0, 1.0], [1.0, 2.0, 0.0]])
