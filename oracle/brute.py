"""O(n^2) rank-rule selection, independent of any sort (pins ``topk_row``).

The rank of position t in a window s is the number of positions that beat it:
``rank(t) = #{u : s[u] > s[t] or (s[u] == s[t] and u < t)}``. Ranks are a
permutation of 0..n-1; t is selected iff ``rank(t) < k`` and sits at output
position ``rank(t)``. This is the ordering rule (higher score first, equal
scores to the lower index) stated directly, with IEEE comparisons (so -0 == +0).
"""

from __future__ import annotations

import numpy as np


def rank_select_bruteforce(window: np.ndarray, k: int) -> np.ndarray:
    s = np.asarray(window, dtype=np.float32).astype(np.float64)
    n = s.size
    out = np.full(min(n, k), -1, dtype=np.int64)
    if n == 0:
        return out
    u = np.arange(n)
    beats = (s[None, :] > s[:, None]) | ((s[None, :] == s[:, None]) & (u[None, :] < u[:, None]))
    rank = beats.sum(axis=1)
    for t in range(n):
        if rank[t] < k:
            out[rank[t]] = t
    return out
