"""Exact merge of two partial attention results (oracle; test infrastructure).

"Ulysses与Ring-Attention详解" §4.2 gives the statistic update
lse_new = log(exp(lse_prev) + exp(lse_cur)); §4.1 names the step
update(out_i, lse_i, out_ij, lse_ij).  "LLM context parallel production
guide" ("核心原理") states that the partials must be combined through the
softmax statistics, never averaged.

Each partial output is already normalised over its own key subset
(out_x = sum_j exp(s_j - lse_x) v_j), so the merged output is the
lse-weighted sum: out = exp(lse_a - lse) out_a + exp(lse_b - lse) out_b.

Reading for empty partials (the pages say nothing): a partial whose key set is
empty has lse = -inf and out = 0 and is the identity of the merge.
"""

from __future__ import annotations

import numpy as np


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Merge two partials.

    o_x   : [rows, H, dv] float64 (each row normalised over its own keys)
    lse_x : [H, rows]      float64 natural-log sum of exp(scaled scores)
    returns (o, lse) with the same shapes.
    """
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    la = np.asarray(lse_a, dtype=np.float64).T  # [rows, H]
    lb = np.asarray(lse_b, dtype=np.float64).T
    m = np.maximum(la, lb)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    with np.errstate(divide="ignore", invalid="ignore"):
        # log(exp(a) + exp(b)), written with the larger term factored out
        ea = np.exp(la - m_safe)
        eb = np.exp(lb - m_safe)
        lse = np.where(empty, -np.inf, m_safe + np.log(ea + eb))
        wa = np.where(empty, 0.0, np.exp(la - np.where(empty, 0.0, lse)))
        wb = np.where(empty, 0.0, np.exp(lb - np.where(empty, 0.0, lse)))
    o = wa[..., None] * o_a + wb[..., None] * o_b
    return o, lse.T.copy()
