"""Seeded synthetic inputs for blockwise ring attention.

This module only draws random numbers and states the workload shapes.  It holds
none of the attention arithmetic, so the fp64 oracle and the CUDA path can both
take their inputs from here without sharing any of the method's code.

Recipe (one per workload):
  * q, k, v and dO are drawn, in that order, as float32 N(0, 1) from a seeded
    generator and rounded to bfloat16 (round-to-nearest-even, as torch does).
    The CPU recipe uses ``torch.Generator('cpu').manual_seed(seed)``; the CUDA
    recipe a seeded CUDA generator (different numbers, same distribution).
  * Tensors are in ORIGINAL token order with shape (b, h, s, d), d contiguous.
  * Varlen lengths: u_k ~ U(0, 1) from numpy's PCG64, x_k = lo * (hi/lo)**u_k
    (log-uniform on [lo, hi]), rescaled to sum to ``total``; floors are taken
    and the remaining +1s go to the largest fractional parts (ties to the lower
    index); every length is at least 1.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    b: int
    h: int
    s: int
    d: int
    layout: str          # "contiguous" | "zigzag" | "stripe"
    n_shards: int
    causal: bool
    backward: bool
    seed: int
    varlen_seqs: int = 0  # >0: packed sequences with one cu_seqlens (b must be 1)
    varlen_seed: int = 2000
    lengths: tuple = field(default=(), compare=False)
    length_multiple: int = 1  # every packed length a multiple of this (zigzag varlen needs 2N)

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5

    @property
    def shard_len(self) -> int:
        return self.s // self.n_shards

    def seq_lengths(self) -> list[int]:
        """Packed lengths: the log-uniform recipe of varlen_lengths; with a length
        multiple m, the same draw at a resolution of m tokens (lengths m * l_k
        with l_k = varlen_lengths(n, s / m, seed, 512 / m, 16384 / m))."""
        if not self.varlen_seqs:
            return []
        m = self.length_multiple
        if m == 1:
            return varlen_lengths(self.varlen_seqs, self.s, self.varlen_seed)
        units = varlen_lengths(self.varlen_seqs, self.s // m, self.varlen_seed, 512.0 / m, 16384.0 / m)
        return [m * u for u in units]

    def fwd_flops(self) -> float:
        """Causal-adjusted forward FLOP: 4*b*h*s_q*s_k*d, halved when causal.

        Varlen: the sum over sequences of 4*h*L_k^2*d, halved when causal."""
        if self.varlen_seqs:
            tot = sum(float(n) * float(n) for n in self.seq_lengths())
            f = 4.0 * self.h * tot * self.d
        else:
            f = 4.0 * self.b * self.h * float(self.s) * float(self.s) * self.d
        return f / 2.0 if self.causal else f


# The five benchmark workloads of the pages' long-context setting.  Seeds are
# 1000 + the workload number.
WORKLOADS = {
    1: Workload("tiny_noncausal_contiguous_fwd", 1, 2, 256, 64, "contiguous", 4, False, False, 1001),
    2: Workload("causal_contiguous_fwd_h32_s16k", 1, 32, 16384, 128, "contiguous", 8, True, False, 1002),
    3: Workload("causal_zigzag_fwdbwd_h32_s64k", 1, 32, 65536, 128, "zigzag", 8, True, True, 1003),
    4: Workload("causal_stripe_fwdbwd_h16_s128k", 1, 16, 131072, 128, "stripe", 8, True, True, 1004),
    5: Workload("varlen_causal_fwdbwd_64seq_128k", 1, 32, 131072, 128, "contiguous", 8, True, True, 1005,
                varlen_seqs=64),
    # zigzag varlen (the zigzag split of every packed sequence): workload 5's
    # recipe with lengths in multiples of 2N = 16 tokens
    6: Workload("varlen_zigzag_causal_fwdbwd_64seq_128k", 1, 32, 131072, 128, "zigzag", 8, True, True, 1006,
                varlen_seqs=64, length_multiple=16),
}


def varlen_lengths(n_seqs: int, total: int, seed: int = 2000, lo: float = 512.0,
                   hi: float = 16384.0) -> list[int]:
    """Log-uniform lengths on [lo, hi], rescaled to ``total`` (largest-remainder rounding)."""
    if n_seqs <= 0:
        return []
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.random(n_seqs)
    x = lo * (hi / lo) ** u
    y = x * (float(total) / float(x.sum()))
    lens = np.floor(y).astype(np.int64)
    rem = int(total - int(lens.sum()))
    frac = y - lens
    order = sorted(range(n_seqs), key=lambda k: (-frac[k], k))
    for k in order[:rem]:
        lens[k] += 1
    lens = np.maximum(lens, 1)
    # clamping can only add tokens; take them back from the longest sequences
    extra = int(lens.sum()) - total
    while extra > 0:
        k = int(np.argmax(lens))
        lens[k] -= 1
        extra -= 1
    return [int(v) for v in lens]


def cu_seqlens(lengths) -> np.ndarray:
    """int32 prefix sums [0, L0, L0+L1, ...]."""
    out = np.zeros(len(lengths) + 1, dtype=np.int32)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64)).astype(np.int32)
    return out


def make_qkv(b: int, h: int, s: int, d: int, seed: int, with_do: bool = True, device: str = "cpu"):
    """q, k, v (and dO) as bf16 tensors of shape (b, h, s, d), original token order."""
    import torch

    if device == "cpu":
        g = torch.Generator("cpu")
    else:
        g = torch.Generator(device)
    g.manual_seed(seed)
    names = ["q", "k", "v"] + (["do"] if with_do else [])
    out = {}
    for n in names:
        x = torch.randn((b, h, s, d), dtype=torch.float32, generator=g, device=device)
        out[n] = x.to(torch.bfloat16)
        del x
    return out


def make_workload_inputs(w: Workload, device: str = "cpu"):
    return make_qkv(w.b, w.h, w.s, w.d, w.seed, with_do=w.backward, device=device)
