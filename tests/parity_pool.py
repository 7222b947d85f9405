"""Full-size parity checks spread over the host cores.

The oracle is a plain single-threaded program; checking every row of the
full-size workloads against it (16384 packed-extend rows of ~66000 scores,
4096 fused prefill rows of ~30000 keys) takes a few core-minutes, so the
rows are split into chunks and checked in a pool of worker processes, one
per host core. The pool uses the "spawn" start method: a process forked
after the parent has used CUDA can hang. Workers get the GPU's outputs for
their rows and return the rows that fail, with the reason; the inputs are
regenerated from their seeds (top-k windows) or memory-mapped from .npy
files the parent writes (fused inputs).
"""

from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

TOL = 1e-3  # fused scores: relative, floored at the row's k-th oracle score


def workers() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _pool():
    # one BLAS thread per worker; the children read these at their numpy import
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    return mp.get_context("spawn").Pool(workers())


def _chunks(rows, n_chunks):
    rows = np.asarray(rows, dtype=np.int64)
    return [c for c in np.array_split(rows, n_chunks) if c.size]


# ------------------------------------------------------------------ top-k
def _topk_task(args):
    import workloads as W
    from oracle.blocks import sparse_blocks as oracle_blocks
    from oracle.topk import topk_transform

    seed, rows, seq_lens, r2b, pt, page_size, k, gs, gi, gb, gc, block_size = args
    bad = []
    for j, i in enumerate(rows):
        n = int(seq_lens[j])
        w = W.packed_extend_window(seed, int(i), n)
        rs, ri = topk_transform(w[None, :], np.array([n]), pt[[int(r2b[j])]], page_size, k)
        if not np.array_equal(gi[j], ri[0]):
            bad.append(f"row {int(i)}: indices differ at {np.flatnonzero(gi[j] != ri[0])[:5].tolist()}")
        elif not np.array_equal(gs[j], rs[0]):
            bad.append(f"row {int(i)}: slots differ at {np.flatnonzero(gs[j] != rs[0])[:5].tolist()}")
        elif gb is not None:
            rb, rc = oracle_blocks(rs, block_size)
            if not (np.array_equal(gb[j], rb[0]) and int(gc[j]) == int(rc[0])):
                bad.append(f"row {int(i)}: block list differs")
    return bad


def check_packed_extend_rows(seed, seq_lens, row_to_batch, page_tables, page_size, k, slots, idx, rows=None,
                             blocks=None, counts=None, block_size=128):
    """Every listed row (all by default) of a packed-extend output against the
    oracle, element by element (and the block lists, when given, against the
    oracle's block lists of the oracle's slots); returns the failing rows'
    messages."""
    rows = np.arange(seq_lens.size) if rows is None else np.asarray(rows)
    tasks = [(seed, c, seq_lens[c], row_to_batch[c], page_tables, page_size, k, slots[c], idx[c],
              None if blocks is None else blocks[c], None if counts is None else counts[c], block_size)
             for c in _chunks(rows, 8 * workers())]
    with _pool() as pool:
        return [m for part in pool.imap_unordered(_topk_task, tasks) for m in part]


# ------------------------------------------------------------------ fused
def kth(s, k):
    return float(np.sort(s)[::-1][min(s.size, k) - 1]) if s.size else 0.0


def check_fused_rows(inp, rows, ref_scores, slots, idx, scores, k=512, blocks=None, counts=None, block_size=128):
    """The fused top-k of the listed rows against the oracle's scores
    (``ref_scores[j]`` for ``rows[j]``; ``slots``/``idx``/``scores`` indexed by
    row). Selection rule: count min(n, k), distinct in-range indices, every
    pick's oracle score >= the oracle k-th score minus the tolerance; the
    GPU's scores within the tolerance of the oracle's, descending, equal GPU
    scores in ascending index order; slots = the transform of the GPU's own
    indices. Block lists (when given): where the GPU picked the oracle's
    set, equal to the oracle's block lists of the oracle's slots; on every
    row, the ascending distinct blocks of the GPU's own slots. Returns the
    failing rows' messages."""
    from oracle.blocks import sparse_blocks as oracle_blocks
    from oracle.topk import page_transform, topk_row

    bad = []
    for j, i in enumerate(rows):
        i = int(i)
        n = int(inp.seq_lens[i])
        kk = min(n, k)
        gi = idx[i]
        if not ((gi[kk:] == -1).all() and (slots[i][kk:] == -1).all()):
            bad.append(f"row {i}: padding")
            continue
        sel = gi[:kk].astype(np.int64)
        if not ((sel >= 0).all() and (sel < n).all()):
            bad.append(f"row {i}: index range")
            continue
        if np.unique(sel).size != kk:
            bad.append(f"row {i}: duplicates")
            continue
        s_ora = np.asarray(ref_scores[j], dtype=np.float64)
        s_k = kth(ref_scores[j], k)
        tol = TOL * max(abs(s_k), 1e-30)
        if not (s_ora[sel] >= s_k - tol).all():
            bad.append(f"row {i}: a pick below the k-th score")
            continue
        gs = scores[i][:kk].astype(np.float64)
        if not (np.abs(gs - s_ora[sel]) <= TOL * np.maximum(np.abs(s_ora[sel]), abs(s_k)) + 1e-30).all():
            bad.append(f"row {i}: selected score mismatch")
            continue
        if not (gs[:-1] >= gs[1:]).all():
            bad.append(f"row {i}: not score-descending")
            continue
        ties = gs[:-1] == gs[1:]
        if not (sel[:-1][ties] < sel[1:][ties]).all():
            bad.append(f"row {i}: equal scores not in ascending index order")
            continue
        b = i if inp.row_to_batch is None else int(inp.row_to_batch[i])
        pages = inp.block_table[b][sel // 128].astype(np.int64)
        if not np.array_equal(slots[i][:kk], pages * 128 + sel % 128):
            bad.append(f"row {i}: slots")
            continue
        if blocks is not None:
            own = np.unique(slots[i][:kk].astype(np.int64) // block_size)
            gb, gc = np.asarray(blocks[i]), int(counts[i])
            if gc != own.size or not np.array_equal(gb[:gc], own) or not (gb[gc:] == -1).all():
                bad.append(f"row {i}: block list is not the distinct blocks of the row's slots")
                continue
            ora = topk_row(s_ora.astype(np.float32), k)
            if np.array_equal(np.sort(ora), np.sort(sel)):
                ora_slots = np.full((1, gb.size), -1, np.int32)
                ora_slots[0, :ora.size] = page_transform(ora, inp.block_table[b], 128)
                ob, oc = oracle_blocks(ora_slots, block_size)
                if oc[0] != gc or not np.array_equal(ob[0], gb):
                    bad.append(f"row {i}: block list differs from the oracle's")
    return bad


_FIELDS = ("q", "w", "kcache", "kscale", "block_table", "seq_lens", "row_to_batch")


def _fused_task(args):
    import workloads as W
    from oracle.score import index_scores

    folder, dtype, rows, slots, idx, scores, blocks, counts, block_size = args
    arr = {}
    for f in _FIELDS:
        path = os.path.join(folder, f + ".npy")
        arr[f] = np.load(path, mmap_mode="r") if os.path.exists(path) else None
    inp = W.FusedInputs(arr["q"], arr["w"], arr["kcache"], arr["kscale"], arr["block_table"],
                        np.asarray(arr["seq_lens"]), None if arr["row_to_batch"] is None else np.asarray(
                            arr["row_to_batch"]), dtype=dtype)
    ref = index_scores(inp, list(rows))
    # the GPU outputs of this chunk are indexed by position in `rows`
    local = {int(r): j for j, r in enumerate(rows)}
    sl = {int(r): slots[j] for r, j in local.items()}
    ix = {int(r): idx[j] for r, j in local.items()}
    sc = {int(r): scores[j] for r, j in local.items()}
    bl = None if blocks is None else {int(r): blocks[j] for r, j in local.items()}
    cn = None if counts is None else {int(r): counts[j] for r, j in local.items()}
    return check_fused_rows(inp, rows, ref, sl, ix, sc, inp.k, bl, cn, block_size)


def check_fused_all_rows(inp, slots, idx, scores, rows=None, blocks=None, counts=None, block_size=128):
    """check_fused_rows over every listed row (all by default), in the pool."""
    rows = np.arange(inp.rows) if rows is None else np.asarray(rows)
    with tempfile.TemporaryDirectory() as folder:
        for f in _FIELDS:
            a = getattr(inp, f)
            if a is not None:
                np.save(os.path.join(folder, f + ".npy"), np.ascontiguousarray(a))
        tasks = [(folder, inp.dtype, c, slots[c], idx[c], scores[c], None if blocks is None else blocks[c],
                  None if counts is None else counts[c], block_size) for c in _chunks(rows, 8 * workers())]
        with _pool() as pool:
            return [m for part in pool.imap_unordered(_fused_task, tasks) for m in part]
