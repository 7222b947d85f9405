"""GPU parity of the per-row sparse block lists against the CPU oracle.

Integer work: the block lists and counts must match the oracle bit for bit.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle.blocks import sparse_blocks as oracle_blocks
from oracle.topk import topk_transform as oracle_topk

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _run(slots, block_size):
    import sparse_attention_indexer_top_gb300 as sai

    s = torch.from_numpy(np.ascontiguousarray(slots)).to(DEV)
    blocks, counts = sai.sparse_blocks(s, block_size)
    torch.cuda.synchronize()
    return blocks.cpu().numpy(), counts.cpu().numpy()


def _check(slots, block_size):
    gb, gc = _run(slots, block_size)
    ob, oc = oracle_blocks(slots, block_size)
    assert np.array_equal(gc, oc), f"counts differ at rows {np.flatnonzero(gc != oc)[:5]}"
    assert np.array_equal(gb, ob), f"blocks differ at rows {np.flatnonzero((gb != ob).any(axis=1))[:5]}"


@pytest.mark.parametrize("k", [512, 100, 1])
@pytest.mark.parametrize("block_size", [128, 16, 1])
def test_random_slots_with_duplicates_and_padding(k, block_size):
    rng = np.random.default_rng(100 + k + block_size)
    rows = 37  # not a multiple of the four rows per CTA
    slots = rng.integers(0, 9000, size=(rows, k)).astype(np.int32)
    slots[::3, k // 2:] = -1            # padded tails
    slots[1::4] = slots[1::4] % 300     # heavy duplication
    slots[5] = -1                       # an empty row
    slots[6] = 777                      # one block, repeated
    _check(slots, block_size)


@pytest.mark.parametrize("span", [4095, 4097, 8193, 12289, 16384])
def test_bitmap_spans_across_word_fields(span):
    """Rows whose blocks span just across 128, 256 and 384 bitmap words (the
    second to fourth word each thread owns) and the bitmap's full 16384 ids:
    the packed per-thread word counts must keep the blocks in order."""
    rng = np.random.default_rng(300 + span)
    rows, k = 9, 512
    lo = rng.integers(0, 1 << 20, size=(rows, 1))
    slots = (lo + rng.integers(0, span, size=(rows, k))).astype(np.int32)
    slots[:, 0] = lo[:, 0]                   # both ends of the span present
    slots[:, 1] = lo[:, 0] + span - 1
    slots[2, 300:] = -1                      # padding
    slots[4] = np.sort(slots[4])[::-1]       # order of the input slots is irrelevant
    _check(slots, 1)


def test_blocks_of_a_topk_output():
    import sparse_attention_indexer_top_gb300 as sai

    inp = W.decode_topk()
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    slots, _ = sai.topk_transform(t(inp.scores), t(inp.seq_lens), t(inp.page_tables), page_size=inp.page_size,
                                  row_starts=t(inp.row_starts), row_to_batch=t(inp.row_to_batch), want_indices=True)
    torch.cuda.synchronize()
    s = slots.cpu().numpy()
    ref_slots, _ = oracle_topk(inp.scores, inp.seq_lens, inp.page_tables, inp.page_size, 512,
                               row_starts=inp.row_starts, row_to_batch=inp.row_to_batch)
    assert np.array_equal(s, ref_slots)
    _check(s, 128)


@pytest.mark.parametrize("block_size", [1, 128])
def test_wide_block_ranges_take_the_sorting_path(block_size):
    # blocks spread over more than 16384 ids: the bitmap does not apply
    rng = np.random.default_rng(200 + block_size)
    rows, k = 21, 512
    slots = rng.integers(0, 1 << 30, size=(rows, k)).astype(np.int32)
    slots[2] = slots[2] % 5000 + (1 << 29)  # narrow again: one row on the bitmap path
    slots[3, 100:] = slots[3, :412]        # duplicates on the sorting path
    slots[4, ::2] = -1
    _check(slots, block_size)
