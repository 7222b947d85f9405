"""Pins of the sparse-block oracle (no GPU).

A hand-worked example, a brute-force set construction on random rows with
heavy duplication, and the invariants (ascending, distinct, exactly the
blocks of the valid slots, -1 after the count).
"""

import numpy as np

from oracle.blocks import sparse_blocks


def test_hand_worked_row():
    # slots 5, 130, 127, 300, -1, 256, 129 with 128-slot blocks: blocks
    # 0, 1, 0, 2, (padding), 2, 1 -> distinct ascending 0, 1, 2
    slots = np.array([[5, 130, 127, 300, -1, 256, 129, -1]], np.int32)
    blocks, counts = sparse_blocks(slots, 128)
    assert counts.tolist() == [3]
    assert blocks.tolist() == [[0, 1, 2, -1, -1, -1, -1, -1]]


def test_empty_and_single_block_rows():
    slots = np.array([[-1, -1, -1, -1], [7, 7, 0, 127]], np.int32)
    blocks, counts = sparse_blocks(slots, 128)
    assert counts.tolist() == [0, 1]
    assert blocks[0].tolist() == [-1, -1, -1, -1]
    assert blocks[1].tolist() == [0, -1, -1, -1]


def test_block_size_one_keeps_every_distinct_slot():
    slots = np.array([[9, 3, 9, 1, -1, 3]], np.int32)
    blocks, counts = sparse_blocks(slots, 1)
    assert counts.tolist() == [3]
    assert blocks[0, :3].tolist() == [1, 3, 9]


def test_against_brute_force_sets():
    rng = np.random.default_rng(7)
    for bs in (1, 16, 128):
        slots = rng.integers(-1, 3000, size=(40, 64)).astype(np.int32)
        slots[::5, 30:] = -1
        blocks, counts = sparse_blocks(slots, bs)
        for i in range(slots.shape[0]):
            want = sorted({int(s) // bs for s in slots[i] if s >= 0})
            assert counts[i] == len(want)
            assert blocks[i, : counts[i]].tolist() == want
            assert (blocks[i, counts[i]:] == -1).all()
            got = blocks[i, : counts[i]]
            assert (np.diff(got) > 0).all()
