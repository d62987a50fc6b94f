"""Seeded synthetic workloads for the packed causal depthwise convolution.

This module only draws inputs: document lengths (numpy) and normal tensors
(torch), then casts them to the stated dtypes. It holds none of the operation's
arithmetic. Tests, the benchmark and the smoke check use it on both sides of a
comparison (the CUDA library and the FP64 oracle).

The five named recipes are the workloads the operation is specified on:

=========  =======  =====  =================================================  =========
name       S        C      documents                                          policy
=========  =======  =====  =================================================  =========
tiny       4096     256    lengths [1000, 0, 2048, 1048]                      bf16
mid        32768    2048   16 lognormal lengths, median 2048, sigma 1.0,      bf16
                           rescaled to sum to S
linattn    65536    6144   uniform lengths in [1, 8192] filling S (last one   bf16
                           truncated), plus 3 empty documents at seeded spots
boundary   131072   1032   uniform lengths in {0..5} filling S                fp32, bf16
large      262144   8192   geometric lengths (mean 4096) filling S            fp32
=========  =======  =====  =================================================  =========

x and dy are N(0, sigma^2) drawn in FP32 and rounded to BF16; weight and bias
are N(0, 0.5^2) and N(0, 0.1^2) in the recipe's dtypes. Every recipe can be
scaled down (``S=..., C=...``) with the same length distribution, which is how
the tests get sizes the oracle finishes in seconds.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

BF16, FP32 = torch.bfloat16, torch.float32


@dataclass(frozen=True)
class Recipe:
    name: str
    S: int
    C: int
    docs: tuple            # (kind, *params)
    x_sigma: float
    weight_dtype: torch.dtype
    bias_dtype: Optional[torch.dtype]
    policies: tuple
    seed: int
    note: str = ""


RECIPES = {
    "tiny": Recipe("tiny", 4096, 256, ("fixed", (1000, 0, 2048, 1048)), 1.0, FP32, FP32,
                   ("bf16",), 0),
    "mid": Recipe("mid", 32768, 2048, ("lognormal", 16, 2048.0, 1.0), 1.0, BF16, None,
                  ("bf16",), 1, "lognormal sigma is not stated; 1.0 is used"),
    "linattn": Recipe("linattn", 65536, 6144, ("uniform", 1, 8192, 3), 1.0, FP32, FP32,
                      ("bf16",), 2, "q|k|v short-conv shape, 3 x 2048 channels"),
    "boundary": Recipe("boundary", 131072, 1032, ("uniform", 0, 5, 0), 2.0, FP32, BF16,
                       ("fp32", "bf16"), 3),
    "large": Recipe("large", 262144, 8192, ("geometric", 4096.0), 1.0, BF16, BF16,
                    ("fp32",), 4),
}


@dataclass
class Workload:
    name: str
    S: int
    C: int
    x: torch.Tensor
    dy: torch.Tensor
    weight: torch.Tensor
    bias: Optional[torch.Tensor]
    cu_seqlens: torch.Tensor
    lengths: List[int] = field(default_factory=list)
    policies: tuple = ("bf16",)

    @property
    def num_docs(self):
        return len(self.lengths)

    def to(self, device):
        mv = lambda t: None if t is None else t.to(device)
        return Workload(self.name, self.S, self.C, mv(self.x), mv(self.dy), mv(self.weight),
                        mv(self.bias), mv(self.cu_seqlens), list(self.lengths), self.policies)


def _fill(draw, S):
    """Draw lengths until they reach S; the last one is cut to fit."""
    out, total = [], 0
    while total < S:
        n = int(draw())
        n = min(n, S - total)
        out.append(n)
        total += n
    return out


def doc_lengths(docs, S, rng):
    """Document lengths (non-negative ints summing to S) for a recipe."""
    kind = docs[0]
    if S == 0:
        return [0]
    if kind == "fixed":
        base = np.asarray(docs[1], dtype=np.float64)
        lens = np.floor(base * S / base.sum()).astype(np.int64)
        lens[-1] += S - lens.sum()
        return [int(v) for v in lens]
    if kind == "lognormal":
        n, median, sigma = docs[1], docs[2], docs[3]
        raw = rng.lognormal(mean=np.log(median), sigma=sigma, size=n)
        lens = np.floor(raw * S / raw.sum()).astype(np.int64)
        lens[-1] += S - lens.sum()
        return [int(v) for v in lens]
    if kind == "uniform":
        lo, hi, n_empty = docs[1], docs[2], docs[3]
        lens = _fill(lambda: rng.integers(lo, hi + 1), S)
        for _ in range(n_empty):
            lens.insert(int(rng.integers(0, len(lens) + 1)), 0)
        return lens
    if kind == "geometric":
        mean = docs[1]
        return _fill(lambda: rng.geometric(1.0 / mean), S)
    raise ValueError(f"unknown document recipe {kind!r}")


def cu_from_lengths(lengths, device="cpu"):
    cu = np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))])
    assert cu[-1] < 2**31
    return torch.from_numpy(cu.astype(np.int32)).to(device)


def make(name, device="cpu", S=None, C=None, seed=None, lengths=None):
    """Build the named recipe (optionally rescaled) on ``device``."""
    r = RECIPES[name]
    S = r.S if S is None else int(S)
    C = r.C if C is None else int(C)
    seed = r.seed if seed is None else int(seed)
    rng = np.random.default_rng(seed)
    if lengths is None:
        lengths = doc_lengths(r.docs, S, rng)
    assert sum(lengths) == S
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = (torch.randn(S, C, generator=g, device=device) * r.x_sigma).to(BF16)
    dy = (torch.randn(S, C, generator=g, device=device) * r.x_sigma).to(BF16)
    weight = (torch.randn(C, 4, generator=g, device=device) * 0.5).to(r.weight_dtype)
    bias = None
    if r.bias_dtype is not None:
        bias = (torch.randn(C, generator=g, device=device) * 0.1).to(r.bias_dtype)
    return Workload(name, S, C, x, dy, weight, bias, cu_from_lengths(lengths, device),
                    list(lengths), r.policies)


def custom(S, C, lengths, seed=0, device="cpu", x_sigma=1.0, weight_dtype=FP32,
           bias_dtype=FP32, w_sigma=0.5, b_sigma=0.1):
    """A workload with explicit document lengths and dtypes (edge cases)."""
    assert sum(lengths) == S
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = (torch.randn(S, C, generator=g, device=device) * x_sigma).to(BF16)
    dy = (torch.randn(S, C, generator=g, device=device) * x_sigma).to(BF16)
    weight = (torch.randn(C, 4, generator=g, device=device) * w_sigma).to(weight_dtype)
    bias = None
    if bias_dtype is not None:
        bias = (torch.randn(C, generator=g, device=device) * b_sigma).to(bias_dtype)
    return Workload("custom", S, C, x, dy, weight, bias, cu_from_lengths(lengths, device),
                    list(lengths), ("bf16", "fp32"))
