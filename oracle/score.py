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

bfloat16 index cache (the "auto" cache type, which is the model dtype): q and
the keys are bfloat16 bit patterns (``inp.dtype == "bf16"``). Each product of
two bfloat16 values has at most 16 significant bits and is exact in float64;
the 128-term sums are float64 (rounding error below 2^-46 of the sum of the
products' magnitudes), then the same relu, head sum and scale follow. A bf16
cache carries no per-key scale in the pages; ``kscale=None`` means scale 1.
"""

from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .bf16 import bf16_finite
from .fp8 import e4m3fn_units
from .topk import page_transform, topk_row

_PROD_UNIT = 2.0 ** -18  # one unit of an e4m3 x e4m3 product
_MAX_UNITS = 229376  # 448 / 2^-9


def _units(codes: np.ndarray, dtype: str) -> np.ndarray:
    """float64 operand values: e4m3 in integer units of 2^-9, bf16 as values."""
    if dtype == "e4m3":
        return e4m3fn_units(codes).astype(np.float64)
    if dtype == "bf16":
        return bf16_finite(codes)
    raise ValueError(f"unknown index cache dtype {dtype!r}")


def _key_units(kcache: np.ndarray, bt_row: np.ndarray, n: int, block_size: int, dtype: str = "e4m3"):
    t = np.arange(n, dtype=np.int64)
    pages = np.asarray(bt_row, dtype=np.int64)[t // block_size]
    return _units(kcache[pages, t % block_size, :], dtype), pages, t % block_size


def _scale_of(kscale, pages, offs) -> np.ndarray:
    if kscale is None:
        return np.ones(pages.shape, np.float64)
    return kscale[pages, offs]


def _scores_from_units(qu: np.ndarray, w: np.ndarray, ku: np.ndarray, scale: np.ndarray,
                       dtype: str = "e4m3") -> np.ndarray:
    """qu [H, D] and ku [n, D] float64 operands; returns fp32 [n]."""
    if dtype == "e4m3":
        assert qu.shape[1] * _MAX_UNITS * _MAX_UNITS < 2.0 ** 53
        relu = np.maximum((qu @ ku.T) * _PROD_UNIT, 0.0)  # exact integers; power-of-two scaling
    else:
        relu = np.maximum(qu @ ku.T, 0.0)
    acc = np.asarray(w, dtype=np.float64) @ relu  # [n]
    return (acc * np.asarray(scale, dtype=np.float64)).astype(np.float32)


def index_scores_row(q_row: np.ndarray, w_row: np.ndarray, kcache: np.ndarray, kscale: Optional[np.ndarray],
                     bt_row: np.ndarray, n: int, dtype: str = "e4m3") -> np.ndarray:
    """Scores of one query row against its first ``n`` keys (fp32 [n])."""
    block_size = kcache.shape[1]
    if n <= 0:
        return np.zeros(0, np.float32)
    ku, pages, offs = _key_units(kcache, bt_row, n, block_size, dtype)
    return _scores_from_units(_units(q_row, dtype), w_row, ku, _scale_of(kscale, pages, offs), dtype)


def index_scores(inp, rows: Optional[Sequence[int]] = None) -> list:
    """Scores of the listed rows (all by default), one fp32 array per row.

    Rows that share a block-table row reuse the gathered keys.
    """
    rows = list(range(inp.rows)) if rows is None else list(rows)
    dtype = getattr(inp, "dtype", "e4m3")
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
        ku, pages, offs = _key_units(inp.kcache, inp.block_table[b], nmax, inp.block_size, dtype)
        scale = _scale_of(inp.kscale, pages, offs)
        for j in js:
            i = rows[j]
            n = int(inp.seq_lens[i])
            qu = _units(inp.q[i], dtype)
            out[j] = _scores_from_units(qu, inp.w[i], ku[:n], scale[:n], dtype) if n > 0 else np.zeros(0, np.float32)
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


def index_scores_per_head(inp, rows: Optional[Sequence[int]] = None) -> list:
    """Per-index-head scores: one float32 array [H, n] per listed row with
    ``score_h(t) = kscale[p, o] * w[i, h] * relu(q[i, h] . k[p, o])``.

    The fused decode kernel of ROCm/ATOM PR #1473 is launched over
    ``(total_q, num_idx_heads, num_topk_chunks)`` (review diff of
    ``index_topk.py``), one program per index head, which admits a selection
    per head; a head's score is then its summand of the head-summed score.
    The dot products are exact (integer e4m3 units) or float64 (bf16), the
    product ``kscale * w * relu`` is formed in float64 and rounded once.
    """
    rows = list(range(inp.rows)) if rows is None else list(rows)
    dtype = getattr(inp, "dtype", "e4m3")
    out = []
    for i in rows:
        b = i if inp.row_to_batch is None else int(inp.row_to_batch[i])
        n = int(inp.seq_lens[i])
        heads = inp.q.shape[1]
        if n <= 0:
            out.append(np.zeros((heads, 0), np.float32))
            continue
        ku, pages, offs = _key_units(inp.kcache, inp.block_table[b], n, inp.block_size, dtype)
        scale = _scale_of(inp.kscale, pages, offs).astype(np.float64)
        dots = _units(inp.q[i], dtype) @ ku.T  # [H, n]
        if dtype == "e4m3":
            dots = dots * _PROD_UNIT
        relu = np.maximum(dots, 0.0)
        w = np.asarray(inp.w[i], dtype=np.float64)[:, None]
        out.append((relu * w * scale[None, :]).astype(np.float32))
    return out


def index_score_topk_per_head(inp, rows: Optional[Sequence[int]] = None):
    """Top-k per (row, index head): ``(slots, indices, scores)`` with slots and
    indices int32 ``[R, H, k]`` (-1 padded) selected by (score desc, index
    asc) from each head's scores, and the per-row [H, n] score arrays."""
    rows = list(range(inp.rows)) if rows is None else list(rows)
    k = inp.k
    heads = inp.q.shape[1]
    scores = index_scores_per_head(inp, rows)
    slots = np.full((len(rows), heads, k), -1, np.int32)
    idxs = np.full((len(rows), heads, k), -1, np.int32)
    for j, i in enumerate(rows):
        b = i if inp.row_to_batch is None else int(inp.row_to_batch[i])
        for h in range(heads):
            sel = topk_row(scores[j][h], k)
            idxs[j, h, : sel.size] = sel
            slots[j, h, : sel.size] = page_transform(sel, inp.block_table[b], inp.block_size)
    return slots, idxs, scores

