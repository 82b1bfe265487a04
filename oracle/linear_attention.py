"""Decayed linear attention and its AllGather context parallelism (oracle;
test infrastructure only).

"超长上下文训练速度翻倍秘籍" (Ling): linear attention computes, per head,
h_t = alpha * h_{t-1} + K_t^T V_t and O_t = Q_t h_t (kernel feature map
omitted), a recurrence over the sequence; the AllGather CP section has every
rank compute the local hidden state and local output of its sequence piece,
gathers the local states ([B, H, D, D]), recovers each rank's initial state
by a prefix over the preceding ranks (kv_state = kv_state * decay + cur_kv_state,
decay = exp(g_gamma * seg_len)) and corrects the local output by
(q * decay) @ init_state, with q scaled by 1/sqrt(head_dim); varlen input has
every sub-sequence cut into cp_size pieces.

Readings taken (the printed pseudo-code is garbled):
* alpha = exp(g) per head (g = g_gamma, a per-head scalar); h_{-1} = 0 at the
  start of every sequence; O_t = scale * Q_t h_t.
* Rank r's initial state is the recovered state after ranks 0 .. r-1 of the
  same sequence (the printed "if i > 1" guard is read as "for the ranks
  before this one").
* The per-token decay of the correction is alpha^(j+1) for the j-th token of
  the piece (0-based), i.e. the decay from the piece start to the token.
* Pieces are contiguous, cut at floor(r*L/C) like the contiguous softmax
  layout.
"""

from __future__ import annotations

from typing import Sequence

import numpy as np

from .sharding import chunk_bounds


def linear_attn_forward(q, k, v, cu_seqlens: Sequence[int], g, scale: float):
    """The definition: o_t = scale * sum_{s<=t} exp(g (t-s)) (q_t . k_s) v_s
    inside each sequence.  q, k: [T, H, Dk]; v: [T, H, Dv]; g: [H]."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    g = np.asarray(g, dtype=np.float64)
    T, H, _ = q.shape
    o = np.zeros((T, H, v.shape[2]))
    cu = [int(x) for x in cu_seqlens]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        n = b - a
        if n == 0:
            continue
        t = np.arange(n)
        diff = t[:, None] - t[None, :]
        for h in range(H):
            w = np.where(diff >= 0, np.exp(g[h] * np.maximum(diff, 0)), 0.0)
            scores = (q[a:b, h] @ k[a:b, h].T) * w
            o[a:b, h] = scale * scores @ v[a:b, h]
    return o


def linear_attn_recurrent(q, k, v, cu_seqlens: Sequence[int], g, scale: float):
    """The recurrence h_t = exp(g) h_{t-1} + k_t^T v_t, o_t = scale q_t h_t."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    g = np.asarray(g, dtype=np.float64)
    T, H, Dk = q.shape
    Dv = v.shape[2]
    o = np.zeros((T, H, Dv))
    cu = [int(x) for x in cu_seqlens]
    for s in range(len(cu) - 1):
        h = np.zeros((H, Dk, Dv))
        for t in range(cu[s], cu[s + 1]):
            h = np.exp(g)[:, None, None] * h + k[t][:, :, None] * v[t][:, None, :]
            o[t] = scale * np.einsum("hd,hde->he", q[t], h)
    return o


def local_state(k, v, g) -> np.ndarray:
    """h at the end of one piece started from zero: sum_s exp(g (n-1-s)) k_s^T v_s."""
    n = k.shape[0]
    w = np.exp(np.asarray(g, dtype=np.float64)[None, :] * (n - 1 - np.arange(n))[:, None])  # [n, H]
    return np.einsum("sh,shd,she->hde", w, k, v)


def linear_attn_cp(q, k, v, cu_seqlens: Sequence[int], g, scale: float, C: int):
    """AllGather CP in the page's steps: local states and local outputs per
    rank piece, gathered states, prefix recovery of each rank's initial
    state, output correction (q * decay) @ init_state."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    g = np.asarray(g, dtype=np.float64)
    T, H, Dk = q.shape
    Dv = v.shape[2]
    o = np.zeros((T, H, Dv))
    cu = [int(x) for x in cu_seqlens]
    for s in range(len(cu) - 1):
        L = cu[s + 1] - cu[s]
        b = [cu[s] + x for x in chunk_bounds(L, C)]
        # intra-GPU: every rank's local state and local output from a zero state
        states = [local_state(k[b[r]:b[r + 1]], v[b[r]:b[r + 1]], g) for r in range(C)]
        local = [linear_attn_forward(q[b[r]:b[r + 1]], k[b[r]:b[r + 1]], v[b[r]:b[r + 1]],
                                     [0, b[r + 1] - b[r]], g, scale) for r in range(C)]
        # inter-GPU: gathered states, prefix over the preceding ranks
        kv_state = np.zeros((H, Dk, Dv))
        for r in range(C):
            init_state = kv_state
            n = b[r + 1] - b[r]
            if n:
                decay_tok = np.exp(g[None, :] * (np.arange(n) + 1)[:, None])  # [n, H]
                corr = scale * np.einsum("th,thd,hde->the", decay_tok, q[b[r]:b[r + 1]], init_state)
                o[b[r]:b[r + 1]] = local[r] + corr
            kv_state = np.exp(g * n)[:, None, None] * kv_state + states[r]
    return o
