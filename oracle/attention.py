"""Exact softmax attention and its gradients in float64 (oracle; test infrastructure).

What is computed (global token order, one packed stream of sequences):

* visibility: key j is visible to query i iff both lie in the same sequence
  (cu_seqlens) and, when causal, pos(j) <= pos(i).  "超长上下文训练速度翻倍秘籍"
  §2 pitfall 1: a rank's own diagonal block needs the causal mask, keys from
  earlier shards are fully visible; "LLM context parallel production guide",
  "因果 Attention 会制造 Rank 负载不均": blocks above the diagonal are never
  visible; "变长序列" + "位置编码必须跟序列分片一起走": packed sequences do not
  see each other.
* forward, per query head h with key/value head kv(h):
      s_ij = scale * q_i . k_j
      lse_i = log sum_{j visible} exp(s_ij)          (natural log, scaled scores)
      o_i   = sum_j exp(s_ij - lse_i) v_j
  "Ulysses与Ring-Attention详解" §4.1: the block step returns (out, lse).
* backward, recomputing P from the forward statistics
  ("Ulysses与Ring-Attention详解" §4.3):
      D_i  = dO_i . o_i
      dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i)
      dq_i = scale sum_j dS_ij k_j
      dk_j = scale sum_{h in group(kv)} sum_i dS_ij q_i
      dv_j = sum_{h in group(kv)} sum_i P_ij dO_i

Every query row's softmax is taken over its whole visible key set at once.
The online (blockwise) merge the method uses is deliberately NOT used here;
rows are only processed in blocks to bound memory.

GQA mapping (the pages only say "GQA"): blocked by default, kv(h) = h // G
with G = hq // hkv; "interleaved" gives kv(h) = h % hkv.
"""

from __future__ import annotations

from typing import Iterable, Optional, Sequence

import numpy as np


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor -> exact float64 copy
        import torch

        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def kv_head(h: int, hq: int, hkv: int, gqa: str = "blocked") -> int:
    G = hq // hkv
    if gqa == "blocked":
        return h // G
    if gqa == "interleaved":
        return h % hkv
    raise ValueError(gqa)


def _heads_of(kv: int, hq: int, hkv: int, gqa: str):
    return [h for h in range(hq) if kv_head(h, hq, hkv, gqa) == kv]


def _cu(cu_seqlens) -> list:
    return [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]


def _softmax_rows(S: np.ndarray, vis: np.ndarray):
    """Row softmax over visible entries: returns (P, lse).  Rows with no
    visible entry give P = 0 and lse = -inf."""
    Sm = np.where(vis, S, -np.inf)
    m = Sm.max(axis=1)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.where(vis, np.exp(Sm - m_safe[:, None]), 0.0)
    l = E.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(l))
        P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, l)[:, None])
    return P, lse


def _vis_block(r0: int, r1: int, L: int, causal: bool) -> np.ndarray:
    """Visibility of keys 0..L-1 for query positions r0..r1-1 of one sequence."""
    i = np.arange(r0, r1)[:, None]
    j = np.arange(L)[None, :]
    if causal:
        return j <= i
    return np.ones((r1 - r0, L), dtype=bool)


def attn_forward(q, k, v, cu_seqlens, scale: float, causal: bool = True,
                 gqa: str = "blocked", row_block: int = 1024):
    """Full forward.  q [T,hq,dk], k [T,hkv,dk], v [T,hkv,dv] (global order).

    Returns o [T,hq,dv] float64 and lse [hq,T] float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, hq, _ = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    cu = _cu(cu_seqlens)
    o = np.zeros((T, hq, dv))
    lse = np.full((hq, T), -np.inf)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        L = b - a
        for h in range(hq):
            kvh = kv_head(h, hq, hkv, gqa)
            K, V = k[a:b, kvh], v[a:b, kvh]
            for r0 in range(0, L, row_block):
                r1 = min(L, r0 + row_block)
                S = scale * (q[a + r0:a + r1, h] @ K.T)
                P, l = _softmax_rows(S, _vis_block(r0, r1, L, causal))
                o[a + r0:a + r1, h] = P @ V
                lse[h, a + r0:a + r1] = l
    return o, lse


def attn_backward(q, k, v, dout, cu_seqlens, scale: float, causal: bool = True,
                  gqa: str = "blocked", row_block: int = 1024):
    """Full backward.  Returns dict(dq, dk, dv, o, lse, D), all float64."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, hq, dk_ = q.shape
    hkv, dv_ = k.shape[1], v.shape[2]
    cu = _cu(cu_seqlens)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.zeros((T, hq, dv_))
    lse = np.full((hq, T), -np.inf)
    D = np.zeros((hq, T))
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        L = b - a
        for h in range(hq):
            kvh = kv_head(h, hq, hkv, gqa)
            K, V = k[a:b, kvh], v[a:b, kvh]
            for r0 in range(0, L, row_block):
                r1 = min(L, r0 + row_block)
                Qb = q[a + r0:a + r1, h]
                dOb = dout[a + r0:a + r1, h]
                S = scale * (Qb @ K.T)
                P, l = _softmax_rows(S, _vis_block(r0, r1, L, causal))
                Ob = P @ V
                Db = (dOb * Ob).sum(axis=1)
                dP = dOb @ V.T
                dS = P * (dP - Db[:, None])
                dq[a + r0:a + r1, h] = scale * (dS @ K)
                dk[a:b, kvh] += scale * (dS.T @ Qb)
                dv[a:b, kvh] += P.T @ dOb
                o[a + r0:a + r1, h] = Ob
                lse[h, a + r0:a + r1] = l
                D[h, a + r0:a + r1] = Db
    return {"dq": dq, "dk": dk, "dv": dv, "o": o, "lse": lse, "D": D}


def _seq_of_rows(cu: list, rows: np.ndarray) -> np.ndarray:
    return np.searchsorted(np.asarray(cu), rows, side="right") - 1


def _rows_by_seq(cu: list, rows: np.ndarray):
    """Groups sampled global rows by sequence: yields (a, b, positions in rows)."""
    seq = _seq_of_rows(cu, rows)
    for s in np.unique(seq):
        yield cu[s], cu[s + 1], np.nonzero(seq == s)[0]


def attn_forward_rows(q, k, v, cu_seqlens, scale: float, rows: Sequence[int],
                      heads: Iterable[int], causal: bool = True, gqa: str = "blocked",
                      chunk: int = 64):
    """Forward for selected global query rows and query heads only.

    Every selected row gets the full-row softmax over its visible keys; rows
    of one sequence are handled together as a small matrix product.
    Returns o [n_rows, n_heads, dv] and lse [n_heads, n_rows].
    """
    rows = np.asarray(rows, dtype=np.int64)
    heads = list(heads)
    hq, hkv = q.shape[1], k.shape[1]
    cu = _cu(cu_seqlens)
    dv = v.shape[2]
    o = np.zeros((len(rows), len(heads), dv))
    lse = np.full((len(heads), len(rows)), -np.inf)
    for hi, h in enumerate(heads):
        kvh = kv_head(h, hq, hkv, gqa)
        for a, b, idx in _rows_by_seq(cu, rows):
            K = _f64(k[a:b, kvh])
            V = _f64(v[a:b, kvh])
            for c0 in range(0, len(idx), chunk):
                sel = idx[c0:c0 + chunk]
                pos = rows[sel] - a
                Qs = _f64(q[rows[sel], h])
                S = scale * (Qs @ K.T)
                vis = (np.arange(b - a)[None, :] <= pos[:, None]) if causal else np.ones_like(S, dtype=bool)
                P, l = _softmax_rows(S, vis)
                o[sel, hi] = P @ V
                lse[hi, sel] = l
    return o, lse


def attn_backward_dq_rows(q, k, v, dout, cu_seqlens, scale: float, rows: Sequence[int],
                          heads: Iterable[int], causal: bool = True, gqa: str = "blocked",
                          chunk: int = 64):
    """dq for selected global query rows / query heads: [n_rows, n_heads, dk]."""
    rows = np.asarray(rows, dtype=np.int64)
    heads = list(heads)
    hq, hkv = q.shape[1], k.shape[1]
    cu = _cu(cu_seqlens)
    out = np.zeros((len(rows), len(heads), q.shape[2]))
    for hi, h in enumerate(heads):
        kvh = kv_head(h, hq, hkv, gqa)
        for a, b, idx in _rows_by_seq(cu, rows):
            K = _f64(k[a:b, kvh])
            V = _f64(v[a:b, kvh])
            for c0 in range(0, len(idx), chunk):
                sel = idx[c0:c0 + chunk]
                pos = rows[sel] - a
                Qs, dOs = _f64(q[rows[sel], h]), _f64(dout[rows[sel], h])
                S = scale * (Qs @ K.T)
                vis = (np.arange(b - a)[None, :] <= pos[:, None]) if causal else np.ones_like(S, dtype=bool)
                P, _ = _softmax_rows(S, vis)
                O = P @ V
                Di = (dOs * O).sum(axis=1)
                dP = dOs @ V.T
                dS = P * (dP - Di[:, None])
                out[sel, hi] = scale * (dS @ K)
    return out


def attn_backward_dkdv_rows(q, k, v, dout, cu_seqlens, scale: float, keys: Sequence[int],
                            kv_heads: Iterable[int], causal: bool = True, gqa: str = "blocked"):
    """dk, dv for selected global key rows and key/value heads.

    Needs every query row that sees a selected key (its lse and D), so the
    cost grows with the distance of the key from the end of its sequence.
    Returns dk [n_keys, n_kv, dk], dv [n_keys, n_kv, dv].
    """
    keys = np.asarray(keys, dtype=np.int64)
    kv_heads = list(kv_heads)
    hq, hkv = q.shape[1], k.shape[1]
    cu = _cu(cu_seqlens)
    seq = _seq_of_rows(cu, keys)
    dk = np.zeros((len(keys), len(kv_heads), q.shape[2]))
    dv = np.zeros((len(keys), len(kv_heads), v.shape[2]))
    for s in np.unique(seq):
        a, b = cu[s], cu[s + 1]
        sel = np.nonzero(seq == s)[0]
        jmin = int(keys[sel].min()) if causal else a
        for ki, kvh in enumerate(kv_heads):
            K = _f64(k[a:b, kvh])
            V = _f64(v[a:b, kvh])
            for h in _heads_of(kvh, hq, hkv, gqa):
                # every query row that can see any selected key of this sequence
                rlo = jmin - a
                Qb = _f64(q[a + rlo:b, h])
                dOb = _f64(dout[a + rlo:b, h])
                L = b - a
                S = scale * (Qb @ K.T)
                P, _ = _softmax_rows(S, _vis_block(rlo, L, L, causal))
                Ob = P @ V
                Db = (dOb * Ob).sum(axis=1)
                for idx in sel:
                    j = int(keys[idx]) - a
                    dPj = dOb @ V[j]
                    dSj = P[:, j] * (dPj - Db)
                    dk[idx, ki] += scale * (dSj @ Qb)
                    dv[idx, ki] += P[:, j] @ dOb
    return dk, dv


def attn_forward_keyset(q, k, v, cu_seqlens, scale: float, key_mask, causal: bool = True,
                        gqa: str = "blocked"):
    """Partial forward restricted to the keys where key_mask (global order,
    length T) is True: out normalised over that subset, lse over that subset
    (-inf and out = 0 for rows that see none of them)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    key_mask = np.asarray(key_mask, dtype=bool)
    T, hq, _ = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    cu = _cu(cu_seqlens)
    o = np.zeros((T, hq, dv))
    lse = np.full((hq, T), -np.inf)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        L = b - a
        vis = _vis_block(0, L, L, causal) & key_mask[a:b][None, :]
        for h in range(hq):
            kvh = kv_head(h, hq, hkv, gqa)
            S = scale * (q[a:b, h] @ k[a:b, kvh].T)
            P, l = _softmax_rows(S, vis)
            o[a:b, h] = P @ v[a:b, kvh]
            lse[h, a:b] = l
    return o, lse
