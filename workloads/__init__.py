"""Seeded synthetic workloads for context-parallel causal attention.

This module only draws inputs: it holds no attention arithmetic, no shard
permutation and no merge.  Both the float64 oracle (``oracle/``) and the CUDA
path consume what it returns, so the two sides always see the same numbers.

Every tensor is returned in GLOBAL token order (the order of the packed
sequence before any context-parallel sharding); putting rows into the
per-rank sharded order is the job of the code under test.

Workload shapes follow the long-context training setups the source pages
discuss ("Ulysses与Ring-Attention详解", §4 Ring-Attention; "LLM context
parallel production guide", sections on ring attention and varlen metadata):
B = 1 packed streams, GQA head groups, head dim 128, an MLA-shaped variant
with a 192-wide query/key head (128 no-rope + 64 rope) and a 128-wide value
head, and varlen packs of sub-sequences described by int32 ``cu_seqlens``.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "get",
    "varlen_lengths",
    "make_inputs",
    "make_cu_seqlens",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem.

    total_tokens : packed length T (sum of sequence lengths)
    seqlens      : per-sequence lengths (None = one sequence of length T)
    hq, hkv      : query / key-value head counts (hq % hkv == 0)
    d_qk, d_v    : head dims of q/k and of v/o
    cp_size      : number of context-parallel shards C
    layout       : "contiguous", "zigzag" or "striped"
    dtype        : "f32" or "bf16"
    sigma        : standard deviation of the N(0, sigma^2) inputs
    seed         : generator seed
    causal       : causal mask inside each sequence
    backward     : whether the workload includes the backward pass
    """

    name: str
    total_tokens: int
    hq: int
    hkv: int
    d_qk: int
    d_v: int
    cp_size: int
    layout: str
    dtype: str
    sigma: float = 1.0
    seed: int = 0
    causal: bool = True
    backward: bool = True
    seqlens: Optional[tuple] = None
    varlen_range: Optional[tuple] = None  # (lo, hi) uniform lengths, drawn by seed

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_qk)

    def lengths(self) -> List[int]:
        if self.seqlens is not None:
            return list(self.seqlens)
        if self.varlen_range is not None:
            lo, hi = self.varlen_range
            return varlen_lengths(self.total_tokens, lo, hi, self.seed)
        return [self.total_tokens]

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the mask leaves visible, per head."""
        tot = 0
        for L in self.lengths():
            tot += L * (L + 1) // 2 if self.causal else L * L
        return tot

    def flops_fwd(self) -> float:
        return float(self.visible_pairs()) * self.hq * (2 * self.d_qk + 2 * self.d_v)

    def flops_bwd(self) -> float:
        return float(self.visible_pairs()) * self.hq * (6 * self.d_qk + 4 * self.d_v)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def varlen_lengths(total: int, lo: int, hi: int, seed: int) -> List[int]:
    """Sub-sequence lengths drawn uniformly from [lo, hi] (inclusive) until
    they cover ``total`` tokens; the last one is truncated to fill exactly."""
    rng = np.random.RandomState(seed)
    out: List[int] = []
    acc = 0
    while acc < total:
        L = int(rng.randint(lo, hi + 1))
        L = min(L, total - acc)
        out.append(L)
        acc += L
    return out


def make_cu_seqlens(lengths: List[int]) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


# The five standard problems, smallest first.  The first is small enough for
# the float64 oracle to finish in milliseconds; the second is the 16K GQA
# problem; the third (S=64K, C=8 zigzag) is the throughput workload.
WORKLOADS = {
    "f32_mha_s256_d64_c2_contiguous": Workload(
        name="f32_mha_s256_d64_c2_contiguous", total_tokens=256, hq=2, hkv=2,
        d_qk=64, d_v=64, cp_size=2, layout="contiguous", dtype="f32", seed=0,
        backward=False),
    "bf16_gqa_s16k_h32kv8_d128_c2_zigzag": Workload(
        name="bf16_gqa_s16k_h32kv8_d128_c2_zigzag", total_tokens=16384, hq=32,
        hkv=8, d_qk=128, d_v=128, cp_size=2, layout="zigzag", dtype="bf16", seed=1),
    "bf16_gqa_s64k_h32kv8_d128_c8_zigzag": Workload(
        name="bf16_gqa_s64k_h32kv8_d128_c8_zigzag", total_tokens=65536, hq=32,
        hkv=8, d_qk=128, d_v=128, cp_size=8, layout="zigzag", dtype="bf16", seed=2),
    "bf16_varlen_t128k_h16kv4_d128_c16_zigzag": Workload(
        name="bf16_varlen_t128k_h16kv4_d128_c16_zigzag", total_tokens=131072,
        hq=16, hkv=4, d_qk=128, d_v=128, cp_size=16, layout="zigzag",
        dtype="bf16", seed=3, varlen_range=(64, 16384)),
    "bf16_mla_s256k_h64_dqk192_dv128_c32_zigzag": Workload(
        name="bf16_mla_s256k_h64_dqk192_dv128_c32_zigzag", total_tokens=262144,
        hq=64, hkv=64, d_qk=192, d_v=128, cp_size=32, layout="zigzag",
        dtype="bf16", sigma=0.5, seed=4),
}

ORDER = list(WORKLOADS)


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _randn(shape, sigma: float, dtype: str, gen: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    if sigma != 1.0:
        x.mul_(sigma)
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    return x


def make_inputs(w: Workload, device="cpu", with_dout: Optional[bool] = None) -> dict:
    """Seeded q, k, v (and dout) in global order plus int32 cu_seqlens (CPU).

    q [T, hq, d_qk], k [T, hkv, d_qk], v [T, hkv, d_v], dout [T, hq, d_v];
    iid N(0, sigma^2), rounded to bf16 for bf16 workloads.
    """
    if with_dout is None:
        with_dout = w.backward
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    T = w.total_tokens
    out = {
        "q": _randn((T, w.hq, w.d_qk), w.sigma, w.dtype, gen, dev),
        "k": _randn((T, w.hkv, w.d_qk), w.sigma, w.dtype, gen, dev),
        "v": _randn((T, w.hkv, w.d_v), w.sigma, w.dtype, gen, dev),
        "cu_seqlens": make_cu_seqlens(w.lengths()),
    }
    if with_dout:
        out["dout"] = _randn((T, w.hq, w.d_v), w.sigma, w.dtype, gen, dev)
    return out


def sample_rows(n_total: int, n_sample: int, seed: int) -> np.ndarray:
    """Sorted distinct row indices drawn by seed (used to pick checked rows)."""
    rng = np.random.RandomState(seed + 7919)
    n_sample = min(n_sample, n_total)
    return np.sort(rng.choice(n_total, size=n_sample, replace=False))
