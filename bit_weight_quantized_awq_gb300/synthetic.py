"""Seeded synthetic inputs for the AWQ W4A16 linear forward.

This module holds none of the method's arithmetic: it only draws random
numbers. Both the GPU tests and the oracle-side checks take their inputs from
here, so neither side generates data for the other.

Distributions (the workload the library is measured on):

* x ~ N(0, 1), drawn in fp32 and rounded to fp16;
* every 4-bit weight code q and zero point z uniform on {0, ..., 15}. Eight
  independent uniform nibbles make one uniform 32-bit word, so qweight and
  qzeros are drawn directly as uniform random bytes viewed as int32: no
  packing code is involved;
* scales ~ U[1e-3, 1e-2], drawn in fp32 and rounded to fp16;
* bias ~ 0.1 * N(0, 1), drawn in fp32 and rounded to fp16 (only if asked).

Draw order is fixed: x, qweight, qzeros, scales, bias, all from one
``torch.Generator`` seeded with ``seed`` (0 unless a test says otherwise).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass
class Problem:
    x: torch.Tensor          # fp16, [M, K] or any [..., K]
    qweight: torch.Tensor    # int32 [K, N/8]
    qzeros: torch.Tensor     # int32 [G, N/8]
    scales: torch.Tensor     # fp16  [G, N]
    bias: torch.Tensor | None  # fp16 [N] or None
    group_size: int          # as passed to the library (may be -1)

    @property
    def K(self) -> int:
        return self.qweight.shape[0]

    @property
    def N(self) -> int:
        return self.qweight.shape[1] * 8

    @property
    def M(self) -> int:
        return self.x.numel() // self.x.shape[-1]

    def to(self, device) -> "Problem":
        mv = lambda t: None if t is None else t.to(device)
        return Problem(mv(self.x), mv(self.qweight), mv(self.qzeros), mv(self.scales),
                       mv(self.bias), self.group_size)


def random_words(gen: torch.Generator, rows: int, words: int) -> torch.Tensor:
    """[rows, words] int32 with every bit independent and uniform."""
    b = torch.randint(0, 256, (rows, words * 4), generator=gen, dtype=torch.uint8)
    return b.view(torch.int32)


def make_problem(M: int, K: int, N: int, group_size: int, bias: bool = False,
                 seed: int = 0, x_shape: tuple[int, ...] | None = None) -> Problem:
    """One seeded problem on the CPU. ``x_shape`` (e.g. (8, 256, 4096)) must
    hold M * K elements and end in K; it defaults to (M, K)."""
    g = K if group_size == -1 else group_size
    if g <= 0 or K % g != 0 or N % 8 != 0:
        raise ValueError("make_problem needs a valid shape")
    G = K // g
    gen = torch.Generator().manual_seed(seed)
    shape = (M, K) if x_shape is None else tuple(x_shape)
    x = torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.float16)
    qweight = random_words(gen, K, N // 8)
    qzeros = random_words(gen, G, N // 8)
    scales = torch.empty((G, N), dtype=torch.float32).uniform_(1e-3, 1e-2, generator=gen)
    scales = scales.to(torch.float16)
    b = None
    if bias:
        b = (0.1 * torch.randn((N,), generator=gen, dtype=torch.float32)).to(torch.float16)
    return Problem(x, qweight, qzeros, scales, b, group_size)


def make_activations(M: int, K: int, seed: int = 0) -> torch.Tensor:
    """A fresh x ~ N(0, 1) fp16 [M, K] from its own seeded generator."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randn((M, K), generator=gen, dtype=torch.float32).to(torch.float16)
