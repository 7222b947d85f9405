"""FP8 index score and the fused index-score + top-k (plain definition).

The fused decode kernel of ROCm/ATOM PR #1473 "enable minimax m3 fp8 index
cache and fuse index_score_kernel with partial_topk kernel" computes index
scores from the FP8 index-key cache and runs partial top-k in the same kernel
(pull request overview, "Changes"; the launch of
``_decode_index_score_topk_partial_kernel`` over ``(total_q, num_idx_heads,
num_topk_chunks)``). Its key loop walks the request's block table: block
``blk`` holds positions ``blk*BLOCK + o`` of the page ``block_table[b][blk]``
and a position is live while ``pos < causal_len`` (review diff of
``index_topk.py``). The pages print no score formula; the one adopted is

    score(i, t) = kscale[p, o] * sum_h w[i, h] * relu( sum_d q[i, h, d] * k[p, o, d] )

with ``p = block_table[b][t // BLOCK]``, ``o = t % BLOCK``, ``b`` the row's
block-table row, no extra 1/sqrt(d) factor (a caller folds constants into w),
and the scale applied outside the relu.

Precision: e4m3 values are integer multiples of 2^-9, so each q*k product is
an integer number of 2^-18 units and a 128-term dot product of them stays far
below 2^53 units. The dot products are therefore formed EXACTLY as float64
integer matrix products (any summation order is exact); relu, the w-weighted
head sum and the scale are applied in float64, and the result is rounded once
to fp32.
"""

from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .fp8 import e4m3fn_units
from .topk import page_transform, topk_row

_PROD_UNIT = 2.0 ** -18  # one unit of an e4m3 x e4m3 product
_MAX_UNITS = 229376  # 448 / 2^-9


def _key_units(kcache: np.ndarray, bt_row: np.ndarray, n: int, block_size: int):
    t = np.arange(n, dtype=np.int64)
    pages = np.asarray(bt_row, dtype=np.int64)[t // block_size]
    return e4m3fn_units(kcache[pages, t % block_size, :]).astype(np.float64), pages, t % block_size


def _scores_from_units(qu: np.ndarray, w: np.ndarray, ku: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """qu [H, D] and ku [n, D] integer-valued float64; returns fp32 [n]."""
    assert qu.shape[1] * _MAX_UNITS * _MAX_UNITS < 2.0 ** 53
    s_units = qu @ ku.T  # [H, n], exact integers
    relu = np.maximum(s_units * _PROD_UNIT, 0.0)  # power-of-two scaling is exact
    acc = np.asarray(w, dtype=np.float64) @ relu  # [n]
    return (acc * np.asarray(scale, dtype=np.float64)).astype(np.float32)


def index_scores_row(q_row: np.ndarray, w_row: np.ndarray, kcache: np.ndarray, kscale: np.ndarray,
                     bt_row: np.ndarray, n: int) -> np.ndarray:
    """Scores of one query row against its first ``n`` keys (fp32 [n])."""
    block_size = kcache.shape[1]
    if n <= 0:
        return np.zeros(0, np.float32)
    ku, pages, offs = _key_units(kcache, bt_row, n, block_size)
    qu = e4m3fn_units(q_row).astype(np.float64)
    return _scores_from_units(qu, w_row, ku, kscale[pages, offs])


def index_scores(inp, rows: Optional[Sequence[int]] = None) -> list:
    """Scores of the listed rows (all by default), one fp32 array per row.

    Rows that share a block-table row reuse the gathered keys.
    """
    rows = list(range(inp.rows)) if rows is None else list(rows)
    out = [None] * len(rows)
    by_batch = {}
    for j, i in enumerate(rows):
        b = i if inp.row_to_batch is None else int(inp.row_to_batch[i])
        by_batch.setdefault(b, []).append(j)
    for b, js in by_batch.items():
        nmax = max(int(inp.seq_lens[rows[j]]) for j in js)
        if nmax <= 0:
            for j in js:
                out[j] = np.zeros(0, np.float32)
            continue
        ku, pages, offs = _key_units(inp.kcache, inp.block_table[b], nmax, inp.block_size)
        scale = inp.kscale[pages, offs]
        for j in js:
            i = rows[j]
            n = int(inp.seq_lens[i])
            qu = e4m3fn_units(inp.q[i]).astype(np.float64)
            out[j] = _scores_from_units(qu, inp.w[i], ku[:n], scale[:n]) if n > 0 else np.zeros(0, np.float32)
    return out


def index_score_topk(inp, rows: Optional[Sequence[int]] = None):
    """Fused score + top-k + slot transform of the listed rows.

    Returns ``(slots, indices, top_scores, scores)``: int32 ``[R, k]`` slots and
    row-local indices (-1 padded), fp32 ``[R, k]`` selected scores (NaN
    padded), and the per-row score arrays the selection was made on.
    """
    rows = list(range(inp.rows)) if rows is None else list(rows)
    k = inp.k
    scores = index_scores(inp, rows)
    slots = np.full((len(rows), k), -1, np.int32)
    idxs = np.full((len(rows), k), -1, np.int32)
    tops = np.full((len(rows), k), np.nan, np.float32)
    for j, i in enumerate(rows):
        b = i if inp.row_to_batch is None else int(inp.row_to_batch[i])
        sel = topk_row(scores[j], k)
        idxs[j, : sel.size] = sel
        tops[j, : sel.size] = scores[j][sel]
        slots[j, : sel.size] = page_transform(sel, inp.block_table[b], inp.block_size)
    return slots, idxs, tops, scores
