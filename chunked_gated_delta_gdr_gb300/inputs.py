"""Seeded synthetic inputs for the chunked gated delta rule forward.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the fp64 oracle (in tests) and the CUDA path (in
tests and the bench) can consume the same tensors.

Distributions follow the accuracy report "FlashQLA GDN backend produces
different tokens from FLA Triton on correctness-test prompts" (maintainer's
reply: q and k L2-normalised per token and head, v Gaussian).  The gate is
``g = logsigmoid(N(3, 1))`` (natural-log decay, kept in fp32), the update
strength ``beta = sigmoid(N(0, 1))`` in bf16, the optional initial state
``h0 = 0.1 * N(0, 1)`` in fp32, and ``scale = d_k ** -0.5``.

Packing follows "Findings from integrating FlashQLA's Blackwell GDN kernels
into a JAX trainer", section 2: sequences are concatenated along the token
axis and described by an int32 ``cu_seqlens`` whose repeated offsets are
length-0 ("ghost") segments.

Layouts (row-major, contiguous):
  q, k  [T, Hk, dk]  bf16        v     [T, H, dv] bf16
  g     [T, H]       fp32        beta  [T, H]     bf16
  h0    [N, H, dk, dv] fp32 or None
  cu_seqlens [N + 1] int32

Draw order for a seeded workload: lengths, q, k, v, g, beta, h0.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import torch
import torch.nn.functional as F

CHUNK = 64


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: Optional[torch.Tensor]
    cu_seqlens: torch.Tensor
    scale: float
    want_ht: bool

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def Hk(self) -> int:
        return int(self.q.shape[1])

    @property
    def H(self) -> int:
        return int(self.v.shape[1])

    @property
    def dk(self) -> int:
        return int(self.q.shape[2])

    @property
    def dv(self) -> int:
        return int(self.v.shape[2])

    @property
    def n_seq(self) -> int:
        return int(self.cu_seqlens.numel()) - 1

    def lengths(self) -> List[int]:
        cu = self.cu_seqlens.tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]

    def n_chunks(self) -> int:
        return sum((n + CHUNK - 1) // CHUNK for n in self.lengths() if n > 0)

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(
            self, q=mv(self.q), k=mv(self.k), v=mv(self.v), g=mv(self.g),
            beta=mv(self.beta), h0=mv(self.h0), cu_seqlens=mv(self.cu_seqlens))


def cu_from_lengths(lengths: Sequence[int]) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def draw_tensors(gen: torch.Generator, T: int, Hk: int, H: int, dk: int, dv: int,
                 n_seq: int, with_h0: bool):
    """Draw q, k, v, g, beta, h0 (in that order) from ``gen``."""
    q = F.normalize(torch.randn(T, Hk, dk, generator=gen), dim=-1).to(torch.bfloat16)
    k = F.normalize(torch.randn(T, Hk, dk, generator=gen), dim=-1).to(torch.bfloat16)
    v = torch.randn(T, H, dv, generator=gen).to(torch.bfloat16)
    g = F.logsigmoid(torch.randn(T, H, generator=gen) + 3.0).to(torch.float32)
    beta = torch.sigmoid(torch.randn(T, H, generator=gen)).to(torch.bfloat16)
    h0 = None
    if with_h0:
        h0 = (0.1 * torch.randn(n_seq, H, dk, dv, generator=gen)).to(torch.float32)
    return q, k, v, g, beta, h0


def make_workload(name: str, seed: int, lengths: Sequence[int], Hk: int, H: int,
                  dk: int, dv: Optional[int] = None, with_h0: bool = False,
                  want_ht: bool = True, gen: Optional[torch.Generator] = None) -> Workload:
    """Build a workload from explicit segment lengths (zeros allowed)."""
    dv = dk if dv is None else dv
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    q, k, v, g, beta, h0 = draw_tensors(gen, T, Hk, H, dk, dv, len(lengths), with_h0)
    return Workload(name, q, k, v, g, beta, h0, cu, dk ** -0.5, want_ht)


# ---------------------------------------------------------------------------
# The five named workloads.  Seeds are 1234 + index, lengths drawn first.
# ---------------------------------------------------------------------------

def _lengths_packed_uniform(gen: torch.Generator, total: int, hi: int, n_ghost: int):
    lens = []
    acc = 0
    while acc < total:
        n = int(torch.randint(1, hi + 1, (1,), generator=gen))
        lens.append(n)
        acc += n
    lens[-1] -= acc - total
    return lens + [0] * n_ghost


def _lengths_mixed(gen: torch.Generator, total: int):
    lens = []
    acc = 0
    kind = 0
    while acc < total:
        if kind == 0:
            n = int(torch.randint(1, 64, (1,), generator=gen))
        elif kind == 1:
            n = 0
        elif kind == 2:
            n = 64 * int(torch.randint(1, 65, (1,), generator=gen))
        else:
            n = int(torch.randint(1, 16385, (1,), generator=gen))
        lens.append(n)
        acc += n
        kind = (kind + 1) % 4
    # clip the last non-zero segment so the total is exact
    i = len(lens) - 1
    while lens[i] == 0:
        i -= 1
    lens[i] -= acc - total
    return lens


WORKLOADS = ("tiny", "fixed_b4_t4096_h16", "packed_64k_h32", "long_t20468_h32",
             "gqa_packed_128k_h16x32")
# A smaller case of the bench workload's shapes, for profiler captures that must
# stay small (8 segments of 2048 tokens, H = Hk = 32, d = 128, no states).
PROFILE_WORKLOADS = ("packed_16k_h32",)


def make_named(name: str) -> Workload:
    """The five workloads: shapes, length mixes and state options as named."""
    if name == "tiny":
        gen = torch.Generator().manual_seed(1234 + 0)
        return make_workload(name, 0, [256], 2, 2, 64, with_h0=False, want_ht=True, gen=gen)
    if name == "fixed_b4_t4096_h16":
        gen = torch.Generator().manual_seed(1234 + 1)
        return make_workload(name, 0, [4096] * 4, 16, 16, 128, with_h0=False, want_ht=True, gen=gen)
    if name == "packed_64k_h32":
        gen = torch.Generator().manual_seed(1234 + 2)
        lens = _lengths_packed_uniform(gen, 65536, 8192, 16)
        return make_workload(name, 0, lens, 32, 32, 128, with_h0=False, want_ht=False, gen=gen)
    if name == "long_t20468_h32":
        gen = torch.Generator().manual_seed(1234 + 3)
        return make_workload(name, 0, [20468], 32, 32, 128, with_h0=True, want_ht=True, gen=gen)
    if name == "gqa_packed_128k_h16x32":
        gen = torch.Generator().manual_seed(1234 + 4)
        lens = _lengths_mixed(gen, 131072)
        return make_workload(name, 0, lens, 16, 32, 128, with_h0=True, want_ht=True, gen=gen)
    if name == "packed_16k_h32":
        gen = torch.Generator().manual_seed(1234 + 100)
        return make_workload(name, 0, [2048] * 8, 32, 32, 128, with_h0=False, want_ht=False,
                             gen=gen)
    raise KeyError(name)


def random_lengths(gen: torch.Generator, total_max: int, n: int, zero_frac: float = 0.0):
    """Random segment lengths in [1, total_max], some set to zero (for tests)."""
    lens = torch.randint(1, total_max + 1, (n,), generator=gen).tolist()
    if zero_frac > 0:
        mask = torch.rand(n, generator=gen) < zero_frac
        lens = [0 if m else x for x, m in zip(lens, mask.tolist())]
    return lens
