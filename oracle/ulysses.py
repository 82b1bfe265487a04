"""Ulysses (all-to-all) context parallelism on one device (oracle; test
infrastructure only).

"Ulysses Context Parallelism 的工程取舍全记录" §1.2 and the figure there: each
device first holds 1/C of the sequence with every head; an all-to-all turns
that into the whole sequence for H/C heads (device r takes heads
r*H/C .. (r+1)*H/C - 1), each device runs ordinary full-sequence attention on
its heads, and a second all-to-all turns the output back into sequence
shards.  "超长上下文训练速度翻倍秘籍", All2All CP 实现, describes the same
transposition (sequence split -> head split, reuse the unsharded kernels,
then back).  §2 of the first page: with GQA every device needs at least one
whole KV head, so C must divide both head counts.

Readings taken: the head range of device r is contiguous (as in the page's
CP=2 figure); the sequence order after the first all-to-all is the global
token order (the unsharded layout of the cu_seqlens metadata).

Arrays: token-major tensors are [T, H, ...] in sharded order (perm from
``sharding.shard_order``); the head-sharded form is [C, T, H/C, ...] in
global token order; lse-like tensors are [H, T] (sharded) and [C, H/C, T]
(global order).
"""

from __future__ import annotations

import numpy as np

from .sharding import to_global


def ulysses_scatter(x_sharded, perm: np.ndarray, C: int):
    """Sequence shards of all heads -> full sequence of each device's heads."""
    xg = to_global(x_sharded, perm)
    T, H = xg.shape[0], xg.shape[1]
    if H % C:
        raise ValueError("head count not divisible by C")
    hc = H // C
    return np.stack([xg[:, r * hc:(r + 1) * hc] for r in range(C)], axis=0)


def ulysses_gather(y, perm: np.ndarray):
    """Inverse of ulysses_scatter: [C, T, H/C, ...] -> [T, H, ...] sharded."""
    C, T, hc = y.shape[0], y.shape[1], y.shape[2]
    xg = np.concatenate([y[r] for r in range(C)], axis=1)
    return xg[perm]


def ulysses_scatter_lse(l_sharded, perm: np.ndarray, C: int):
    """[H, T] in sharded token order -> [C, H/C, T] in global token order."""
    H, T = l_sharded.shape
    lg = np.empty_like(l_sharded)
    lg[:, perm] = l_sharded
    hc = H // C
    return np.stack([lg[r * hc:(r + 1) * hc] for r in range(C)], axis=0)


def ulysses_gather_lse(l_u, perm: np.ndarray):
    """Inverse of ulysses_scatter_lse."""
    C, hc, T = l_u.shape
    lg = np.concatenate([l_u[r] for r in range(C)], axis=0)
    return lg[:, perm]
