"""Per-row window top-k and the page-table transform (the plain definition).

What is computed follows sglang PR #37889 "[AMD] Enable GLM DSA prefill top-k
to the v2 kernel", Modifications (the addressing table of
``topk_transform_512_v2``):

* the score window of row i is ``scores[i, :seq_lens[i]]``, or
  ``scores[i, row_starts[i] : row_starts[i] + seq_lens[i]]`` when
  ``row_starts`` is supplied; the selected index stays row-local;
* the page-table row is ``page_tables[i]``, or ``page_tables[row_to_batch[i]]``
  when ``row_to_batch`` is supplied;
* the selected row-local positions are mapped through that page-table row to
  physical KV slots, which is also what "merge build sparse block into topk"
  (ROCm/ATOM PR #1282, title and Motivation) folds into the top-k kernel.

Readings where the pages are silent (each one listed in the design notes):

* the k outputs are ordered by score descending, equal scores by row-local
  index ascending; this is exactly the prefix of a stable sort by descending
  score of the index-ordered window;
* -0.0 and +0.0 are equal scores; +-inf are ordinary values; NaN is not an
  admissible input;
* positions ``[min(n, k), k)`` of both outputs are -1;
* with page size ``ps`` the slot of row-local index ``t`` is
  ``page_row[t // ps] * ps + t % ps`` (``ps = 1`` is the "wide" page_size=1
  table of the same page), computed in int64 and stored as int32.
"""

from __future__ import annotations

from typing import Optional

import numpy as np


def topk_row(window: np.ndarray, k: int) -> np.ndarray:
    """Row-local indices of the top-k of one window, in output order.

    A full stable sort of the index-ordered window by descending score; the
    first ``min(n, k)`` positions are the answer. Negating an fp32 value is
    exact, and numpy's stable sort keeps equal keys (including -0 == +0) in
    index order.
    """
    w = np.asarray(window, dtype=np.float32)
    if w.size and np.isnan(w).any():
        raise ValueError("NaN scores are not an admissible input")
    order = np.argsort(-w.astype(np.float64), kind="stable")
    return order[: min(w.size, k)].astype(np.int64)


def page_transform(idx: np.ndarray, page_row: np.ndarray, page_size: int) -> np.ndarray:
    """Physical slot of each row-local index through one page-table row."""
    idx = np.asarray(idx, dtype=np.int64)
    pages = np.asarray(page_row, dtype=np.int64)[idx // page_size]
    return pages * page_size + idx % page_size


def topk_transform(scores: np.ndarray, seq_lens: np.ndarray, page_tables: np.ndarray,
                   page_size: int, k: int, row_starts: Optional[np.ndarray] = None,
                   row_to_batch: Optional[np.ndarray] = None, rows=None):
    """Top-k + page transform of every row (or of the rows listed in ``rows``).

    Returns ``(slots, indices)``, both int32 ``[len(rows), k]``, -1 padded.
    """
    all_rows = list(range(int(len(seq_lens))) if rows is None else rows)
    slots = np.full((len(all_rows), k), -1, dtype=np.int32)
    idxs = np.full((len(all_rows), k), -1, dtype=np.int32)
    for j, i in enumerate(all_rows):
        n = int(seq_lens[i])
        start = 0 if row_starts is None else int(row_starts[i])
        b = i if row_to_batch is None else int(row_to_batch[i])
        sel = topk_row(scores[i, start : start + n], k)
        idxs[j, : sel.size] = sel
        slots[j, : sel.size] = page_transform(sel, page_tables[b], page_size)
    return slots, idxs
