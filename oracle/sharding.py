"""Global <-> sharded token order (oracle; test infrastructure only).

Placement rules, from the pages:

* Contiguous: shard r of C holds the r-th of C consecutive pieces of the
  sequence ("LLM context parallel production guide", "核心原理": each rank keeps
  about S/C tokens; "因果 Attention 会制造 Rank 负载不均": plain consecutive
  token ranges).
* Zigzag: the sequence is cut into 2C chunks and rank r holds chunk r followed
  by chunk 2C-1-r ("Ulysses与Ring-Attention详解" §4.2, the device/block table
  for 4 devices and 8 blocks: device 0 holds blocks 0 and 7, ..., device 3
  holds blocks 3 and 4).
* Striped: token t of a sequence goes to rank t mod C, so every rank holds
  early and late tokens ("LLM context parallel production guide",
  "因果 Attention 会制造 Rank 负载不均": interleaved or striped token
  placement as a cure for the causal imbalance).  Reading taken: the stripe
  is one token wide and a rank keeps its tokens in increasing order.
* Packed variable-length input: every sub-sequence is cut into its own CP
  pieces ("超长上下文训练速度翻倍秘籍" §3, varlen CP implementation), and the
  cu_seqlens metadata follows the same mapping ("LLM context parallel
  production guide", "位置编码必须跟序列分片一起走").

Reading taken where the pages are silent: a sub-sequence of length L cut into
n pieces is cut at floor(j*L/n), j = 0..n, so pieces differ by at most one
token and may be empty when L < n; no padding is inserted.  Rank r's shard is,
for each sequence in order, its pieces in the order listed above.
"""

from __future__ import annotations

from typing import List, Sequence

import numpy as np


def chunk_bounds(L: int, n: int) -> List[int]:
    """Cut points of a length-L sequence into n pieces: floor(j*L/n)."""
    return [(j * L) // n for j in range(n + 1)]


def striped_rows(L: int, C: int, r: int) -> List[int]:
    """Token indices t in [0, L) with t mod C == r, in increasing order."""
    return list(range(r, L, C))


def rank_chunks(r: int, C: int, layout: str) -> List[int]:
    """Chunk indices held by rank r, in storage order, and chunks per sequence."""
    if layout == "contiguous":
        return [r]
    if layout == "zigzag":
        return [r, 2 * C - 1 - r]
    raise ValueError(layout)


def chunks_per_sequence(C: int, layout: str) -> int:
    return C if layout == "contiguous" else 2 * C


def shard_order(cu_seqlens: Sequence[int], C: int, layout: str) -> np.ndarray:
    """perm with perm[sharded_row] = global_row, over all T tokens.

    Sharded order is the concatenation of the C ranks' local buffers.
    """
    cu = [int(x) for x in cu_seqlens]
    perm: List[int] = []
    if layout == "striped":
        for r in range(C):
            for s in range(len(cu) - 1):
                perm.extend(cu[s] + t for t in striped_rows(cu[s + 1] - cu[s], C, r))
        return np.asarray(perm, dtype=np.int64)
    n = chunks_per_sequence(C, layout)
    for r in range(C):
        for s in range(len(cu) - 1):
            a, L = cu[s], cu[s + 1] - cu[s]
            b = chunk_bounds(L, n)
            for c in rank_chunks(r, C, layout):
                perm.extend(range(a + b[c], a + b[c + 1]))
    return np.asarray(perm, dtype=np.int64)


def rank_offsets(cu_seqlens: Sequence[int], C: int, layout: str) -> np.ndarray:
    """Start row of each rank's shard in sharded order (length C+1)."""
    cu = [int(x) for x in cu_seqlens]
    off = [0]
    for r in range(C):
        cnt = 0
        for s in range(len(cu) - 1):
            L = cu[s + 1] - cu[s]
            if layout == "striped":
                cnt += len(striped_rows(L, C, r))
                continue
            b = chunk_bounds(L, chunks_per_sequence(C, layout))
            for c in rank_chunks(r, C, layout):
                cnt += b[c + 1] - b[c]
        off.append(off[-1] + cnt)
    return np.asarray(off, dtype=np.int64)


def rank_visible_pairs(cu_seqlens: Sequence[int], C: int, layout: str, causal: bool = True) -> np.ndarray:
    """Per-rank count of visible (query, key) pairs: the attention work each
    rank's queries carry ("LLM context parallel production guide",
    "因果 Attention 会制造 Rank 负载不均": watch the effective QK work per
    rank, not the token count).  A query at position t of a length-L
    sequence sees t + 1 keys when causal, L otherwise."""
    cu = [int(x) for x in cu_seqlens]
    perm = shard_order(cu, C, layout)
    off = rank_offsets(cu, C, layout)
    seq_of = np.searchsorted(np.asarray(cu[1:]), perm, side="right")
    start = np.asarray(cu)[seq_of]
    length = np.asarray(cu)[seq_of + 1] - start
    work = (perm - start + 1) if causal else length
    return np.asarray([int(work[off[r]:off[r + 1]].sum()) for r in range(C)], dtype=np.int64)


def to_sharded(x, perm: np.ndarray):
    """Rows of x (global order, first axis) into sharded order."""
    return x[perm]


def to_global(xs, perm: np.ndarray):
    """Rows of xs (sharded order, first axis) back into global order."""
    out = xs.copy() if hasattr(xs, "copy") else xs.clone()
    out[perm] = xs
    return out
