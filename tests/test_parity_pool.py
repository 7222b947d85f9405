"""The pooled full-size checkers accept the oracle's own outputs and reject
altered ones (CPU only: the "GPU outputs" here come from the oracle, and each
alteration is planted in a copy of them)."""

import numpy as np

import workloads as W
from oracle.score import index_score_topk
from oracle.topk import topk_transform
from parity_pool import check_fused_all_rows, check_packed_extend_rows


def test_packed_extend_checker():
    row_starts, seq_lens, r2b, width = W.packed_extend_meta(reqs=2, new_tokens=24, kv_len=3000)
    pt = W.page_table_perm(3, (2, 3000))
    rows = seq_lens.size
    slots = np.empty((rows, 512), np.int32)
    idx = np.empty((rows, 512), np.int32)
    for i in range(rows):
        n = int(seq_lens[i])
        s, x = topk_transform(W.packed_extend_window(3, i, n)[None, :], np.array([n]), pt[[r2b[i]]], 1, 512)
        slots[i], idx[i] = s[0], x[0]
    assert check_packed_extend_rows(3, seq_lens, r2b, pt, 1, 512, slots, idx) == []
    bad_idx = idx.copy()
    bad_idx[5, [10, 11]] = bad_idx[5, [11, 10]]  # two outputs swapped
    bad_slots = slots.copy()
    bad_slots[30, 0] += 1
    msgs = check_packed_extend_rows(3, seq_lens, r2b, pt, 1, 512, bad_slots, bad_idx)
    assert sorted(m.split(":")[0] for m in msgs) == ["row 30", "row 5"]


def test_fused_checker():
    rows, kv = 12, 1500
    lens = (kv - rows + 1 + np.arange(rows)).astype(np.int32)
    blocks = -(-kv // 128)
    inp = W.make_fused_inputs(61, rows, 64, 128, blocks, lens, (1, blocks), row_to_batch=np.zeros(rows, np.int32))
    slots, idx, tops, scores = index_score_topk(inp)
    assert check_fused_all_rows(inp, slots, idx, tops) == []
    bad_idx = idx.copy()
    bad_idx[3, 0] = int(np.argmin(scores[3]))  # the best key replaced by the worst
    bad_tops = tops.copy()
    bad_tops[7, 5] *= 1.01  # a score off by 1%
    msgs = check_fused_all_rows(inp, slots, bad_idx, bad_tops)
    assert sorted(m.split(":")[0] for m in msgs) == ["row 3", "row 7"]


def test_fused_checker_block_lists():
    from oracle.blocks import sparse_blocks
    from parity_pool import check_fused_rows

    inp = W.make_fused_inputs(61, 6, 64, 128, 24, np.array([1, 130, 300, 330, 200, 380], np.int32), (6, 4))
    slots, idx, tops, scores = index_score_topk(inp)
    for bs in (128, 1):
        blocks, counts = sparse_blocks(slots, bs)
        assert check_fused_rows(inp, list(range(6)), scores, slots, idx, tops, 512, blocks, counts, bs) == []
    blocks, counts = sparse_blocks(slots, 128)
    blocks[2, 0] += 1  # a wrong block
    msgs = check_fused_rows(inp, list(range(6)), scores, slots, idx, tops, 512, blocks, counts, 128)
    assert [m.split(":")[0] for m in msgs] == ["row 2"]
