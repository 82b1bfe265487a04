"""Float64 CPU oracle for context-parallel causal attention — TEST INFRASTRUCTURE.

This package is the independent statement of what the GPU path must compute.
It is test infrastructure only: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the product path never does,
and it shares no code with the CUDA library (no kernels, headers, tables or
pre/post-processing).  Inputs come from ``workloads`` (seeded draws only).

Contents and the passage each follows:

* ``attention``  — exact softmax attention and its analytic gradients, per
  sequence, per head, with a full-row softmax for every query row (no online
  merge).  "Ulysses与Ring-Attention详解" §4.1 (block attention returns
  (out, lse)), §4.3 (backward recomputes from the forward statistics);
  "超长上下文训练速度翻倍秘籍" §2 pitfall 1 (the diagonal block is causal,
  earlier blocks are fully visible); "LLM context parallel production guide"
  sections "核心原理" (the result is exact attention) and "变长序列" (packed
  sequences never attend across their boundaries).
* ``sharding``   — the global <-> sharded token order for contiguous, zigzag and
  striped placement, and the per-rank visible-pair counts.  "Ulysses与Ring-Attention详解" §4.2 (zigzag pairs block i with
  block 2C-1-i); "超长上下文训练速度翻倍秘籍" §3 varlen CP (every sub-sequence
  is itself cut into CP pieces).
* ``ulysses``    — the all-to-all re-layout of Ulysses CP on one device
  (sequence shards <-> head shards).  "Ulysses Context Parallelism
  的工程取舍全记录" §1.2, §2 (GQA: C divides the KV head count);
  "超长上下文训练速度翻倍秘籍", All2All CP 实现.
* ``linear_attention`` — decayed linear attention (definition and
  recurrence) and its AllGather CP state recovery.  "超长上下文训练速度翻倍秘籍",
  the linear-attention recurrence and the AllGather CP / varlen sections.
* ``merge``      — the exact log-sum-exp merge of two partial results.
  "Ulysses与Ring-Attention详解" §4.2 (lse_new = log(exp(lse_prev) +
  exp(lse_cur))); "LLM context parallel production guide" "核心原理" (partials
  are merged through the softmax statistics, not averaged).

Parity pins for every function live in ``tests/test_oracle_*.py``.
"""

from .attention import (  # noqa: F401
    kv_head,
    attn_forward,
    attn_backward,
    attn_forward_rows,
    attn_backward_dq_rows,
    attn_backward_dkdv_rows,
    attn_forward_keyset,
)
from .sharding import (  # noqa: F401
    chunk_bounds,
    rank_chunks,
    shard_order,
    rank_offsets,
    rank_visible_pairs,
    striped_rows,
    to_sharded,
    to_global,
)
from .merge import lse_merge  # noqa: F401
from .ulysses import (  # noqa: F401
    ulysses_scatter,
    ulysses_gather,
    ulysses_scatter_lse,
    ulysses_gather_lse,
)
from .linear_attention import (  # noqa: F401
    linear_attn_forward,
    linear_attn_recurrent,
    linear_attn_cp,
    local_state,
)
