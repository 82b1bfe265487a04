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


# ---------------------------------------------------------------------------
# Samplers for long sequences.  They compute the same definitions as
# attn_forward / attn_backward for selected rows only, in plain PyTorch
# float64 CPU ops (matrix products and elementwise exp/max/sum spread over the
# host cores), so that problems of 64K-256K tokens stay within seconds to a
# minute.  Every selected row still gets its full-row softmax over all of its
# visible keys in one piece.

def _t64(x):
    """Exact float64 CPU torch copy of a numpy array or a torch tensor."""
    import torch

    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))


def _gather_rows(x, idx, h):
    """x[idx, h] (global rows idx of head h) as float64 torch."""
    import torch

    if isinstance(x, torch.Tensor):
        return _t64(x[torch.as_tensor(np.asarray(idx, dtype=np.int64)), h])
    return _t64(np.asarray(x)[np.asarray(idx, dtype=np.int64), h])


class _Scores:
    """scale * Q K^T into one reused float64 buffer (allocating a fresh
    multi-hundred-MB matrix per block costs more than the product itself)."""

    def __init__(self):
        self.buf = None

    def __call__(self, Qs, K, scale: float):
        import torch

        n, m = Qs.shape[0], K.shape[0]
        if self.buf is None or self.buf.numel() < n * m:
            self.buf = torch.empty(max(n * m, 1), dtype=torch.float64)
        S = self.buf[:n * m].view(n, m)
        torch.mm(Qs, K.T, out=S)
        return S.mul_(scale)


def _softmax_rows_t(S, qpos, causal: bool):
    """Row softmax of the scaled scores S [n, m] of queries at sequence
    positions qpos [n] against the keys at positions 0..m-1 (key j is masked
    for query i when causal and j > pos(i)).  S is overwritten.  Returns
    (P, lse); rows that see no key give P = 0 and lse = -inf."""
    import torch

    n, m = S.shape
    if m == 0:
        return S, torch.full((n,), float("-inf"), dtype=torch.float64)
    if causal:
        c0 = int(qpos.min())  # keys before the earliest query are visible to every row
        if c0 < m:
            j = torch.arange(c0, m)
            S[:, c0:].masked_fill_(j[None, :] > qpos[:, None], float("-inf"))
    mx = S.amax(dim=1)
    empty = torch.isneginf(mx)
    mx = torch.where(empty, torch.zeros_like(mx), mx)
    S.sub_(mx[:, None]).exp_()  # masked entries: exp(-inf) = 0
    l = S.sum(dim=1)
    lse = torch.where(empty, torch.full_like(mx, float("-inf")), mx + torch.log(l))
    P = S.div_(torch.where(empty, torch.ones_like(l), l)[:, None])
    return P, lse


def _sampled_rows_forward(q, k, v, cu, scale, rows, h, kvh, causal, chunk, dout=None):
    """Yields (positions in rows, P, O, Q, K, V, dO) per chunk of the selected
    rows of one sequence at a time, for query head h / kv head kvh."""
    import torch

    scores = _Scores()
    for a, b, idx in _rows_by_seq(cu, rows):
        pos_all = rows[idx] - a
        m_seq = int(pos_all.max()) + 1 if causal else b - a
        K = _t64(k[a:a + m_seq, kvh])
        V = _t64(v[a:a + m_seq, kvh])
        for c0 in range(0, len(idx), chunk):
            sel = idx[c0:c0 + chunk]
            pos = torch.as_tensor(rows[sel] - a)
            m = int(pos.max()) + 1 if causal else b - a
            Qs = _gather_rows(q, rows[sel], h)
            P, lse = _softmax_rows_t(scores(Qs, K[:m], scale), pos, causal)
            dOs = _gather_rows(dout, rows[sel], h) if dout is not None else None
            yield sel, P, lse, Qs, K[:m], V[:m], dOs


def attn_forward_rows(q, k, v, cu_seqlens, scale: float, rows: Sequence[int],
                      heads: Iterable[int], causal: bool = True, gqa: str = "blocked",
                      chunk: int = 128):
    """Forward for selected global query rows and query heads only.

    Every selected row gets the full-row softmax over its visible keys; rows
    of one sequence are handled together as a matrix product.
    Returns o [n_rows, n_heads, dv] and lse [n_heads, n_rows] (numpy float64).
    """
    rows = np.asarray(rows, dtype=np.int64)
    heads = list(heads)
    hq, hkv = q.shape[1], k.shape[1]
    cu = _cu(cu_seqlens)
    o = np.zeros((len(rows), len(heads), v.shape[2]))
    lse = np.full((len(heads), len(rows)), -np.inf)
    for hi, h in enumerate(heads):
        kvh = kv_head(h, hq, hkv, gqa)
        for sel, P, l, _, _, V, _ in _sampled_rows_forward(q, k, v, cu, scale, rows, h, kvh, causal, chunk):
            o[sel, hi] = (P @ V).numpy()
            lse[hi, sel] = l.numpy()
    return o, lse


def attn_backward_dq_rows(q, k, v, dout, cu_seqlens, scale: float, rows: Sequence[int],
                          heads: Iterable[int], causal: bool = True, gqa: str = "blocked",
                          chunk: int = 128):
    """dq for selected global query rows / query heads: [n_rows, n_heads, dk]."""
    rows = np.asarray(rows, dtype=np.int64)
    heads = list(heads)
    hq, hkv = q.shape[1], k.shape[1]
    cu = _cu(cu_seqlens)
    out = np.zeros((len(rows), len(heads), q.shape[2]))
    for hi, h in enumerate(heads):
        kvh = kv_head(h, hq, hkv, gqa)
        for sel, P, _, _, K, V, dOs in _sampled_rows_forward(q, k, v, cu, scale, rows, h, kvh, causal, chunk,
                                                               dout=dout):
            O = P @ V
            Di = (dOs * O).sum(dim=1)
            dS = P * (dOs @ V.T - Di[:, None])
            out[sel, hi] = (scale * (dS @ K)).numpy()
    return out


def attn_backward_dkdv_rows(q, k, v, dout, cu_seqlens, scale: float, keys: Sequence[int],
                            kv_heads: Iterable[int], causal: bool = True, gqa: str = "blocked",
                            row_block: int = 1024):
    """dk, dv for selected global key rows and key/value heads.

    dk_j and dv_j sum over every query row i that sees key j, and each such
    row needs its own lse_i and D_i = dO_i . o_i, i.e. its whole forward row.
    The query rows of a sequence, from its earliest selected key on, are
    therefore visited in blocks of row_block consecutive rows; each block
    takes its full visible key range (keys past the block's last row are
    masked for all of it), computes P, o and D, and adds the selected keys'
    terms.  Memory stays bounded at any sequence length; the cost is that of
    the forward over those rows.
    Returns dk [n_keys, n_kv, dk], dv [n_keys, n_kv, dv] (numpy float64).
    """
    import torch

    keys = np.asarray(keys, dtype=np.int64)
    kv_heads = list(kv_heads)
    hq, hkv = q.shape[1], k.shape[1]
    cu = _cu(cu_seqlens)
    seq = _seq_of_rows(cu, keys)
    dk = torch.zeros(len(keys), len(kv_heads), q.shape[2], dtype=torch.float64)
    dv = torch.zeros(len(keys), len(kv_heads), v.shape[2], dtype=torch.float64)
    scores = _Scores()
    for s in np.unique(seq):
        a, b = cu[s], cu[s + 1]
        L = b - a
        sel = np.nonzero(seq == s)[0]
        kpos = torch.as_tensor(keys[sel] - a)
        r_start = int(kpos.min()) if causal else 0  # earlier rows see none of the selected keys
        for ki, kvh in enumerate(kv_heads):
            K = _t64(k[a:b, kvh])
            V = _t64(v[a:b, kvh])
            Vsel = V[kpos]
            for h in _heads_of(kvh, hq, hkv, gqa):
                Q = _t64(q[a + r_start:b, h])
                dO = _t64(dout[a + r_start:b, h])
                for r0 in range(r_start, L, row_block):
                    r1 = min(L, r0 + row_block)
                    m = r1 if causal else L
                    Qb, dOb = Q[r0 - r_start:r1 - r_start], dO[r0 - r_start:r1 - r_start]
                    P, _ = _softmax_rows_t(scores(Qb, K[:m], scale), torch.arange(r0, r1), causal)
                    Db = (dOb * (P @ V[:m])).sum(dim=1)
                    seen = kpos < m  # selected keys some row of this block can see
                    if not bool(seen.any()):
                        continue
                    Pj = P[:, kpos[seen]]
                    dSj = Pj * (dOb @ Vsel[seen].T - Db[:, None])
                    tgt = torch.as_tensor(sel)[seen]
                    dk[tgt, ki] += scale * (dSj.T @ Qb)
                    dv[tgt, ki] += Pj.T @ dOb
    return dk.numpy(), dv.numpy()


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
