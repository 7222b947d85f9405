"""Per-row sparse KV block lists from top-k slots (the plain definition).

What is computed follows ROCm/ATOM PR #1282 "merge build sparse block into
topk" (title and Motivation): after the top-k has produced physical KV slots,
the sparse attention that consumes them works on KV blocks, so each row's
selected slots are turned into the list of distinct blocks they fall in.

Readings where the page is silent (each one listed in the design notes):

* the block of a slot s is ``s // block_size`` (block_size 128, the KV block
  of the fused path; any block_size >= 1 is accepted);
* slots < 0 are padding and contribute no block;
* each row's distinct blocks are listed in ascending order in the first
  ``count`` positions of a k-wide row, the rest is -1, and ``count`` is
  returned per row.
"""

from __future__ import annotations

import numpy as np


def sparse_blocks(slots: np.ndarray, block_size: int = 128) -> tuple[np.ndarray, np.ndarray]:
    """Distinct blocks of each row's valid slots, ascending, -1 padded.

    ``slots`` is int32 [rows, k]. Returns (blocks int32 [rows, k], counts
    int32 [rows]). A library routine (``np.unique``, which sorts) does the
    deduplication; the tests pin it against a brute-force set construction.
    """
    slots = np.asarray(slots)
    rows, k = slots.shape
    blocks = np.full((rows, k), -1, dtype=np.int32)
    counts = np.zeros(rows, dtype=np.int32)
    for i in range(rows):
        row = slots[i].astype(np.int64)
        u = np.unique(row[row >= 0] // int(block_size))
        blocks[i, : u.size] = u
        counts[i] = u.size
    return blocks, counts
