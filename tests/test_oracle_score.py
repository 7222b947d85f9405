"""Pins of the oracle's FP8 index score and fused top-k (CPU only).

The exact value of each score is recomputed with Python ``Fraction``s from
torch's e4m3 decoding (a library routine, not the oracle's decoder), with the
block-table gather written out by hand; shapes are non-square (heads != dim,
block size != dim) so a transposed operand or a swapped page/offset fails.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W
from oracle.brute import rank_select_bruteforce
from oracle.score import index_score_topk, index_scores, index_scores_row


def _dec(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _exact_scores(inp, i):
    q = _dec(inp.q[i])
    b = i if inp.row_to_batch is None else int(inp.row_to_batch[i])
    out = []
    bs = inp.kcache.shape[1]
    for t in range(int(inp.seq_lens[i])):
        page = int(inp.block_table[b][t // bs])
        kk = _dec(inp.kcache[page, t % bs])
        acc = Fraction(0)
        for h in range(q.shape[0]):
            dot = sum((Fraction(float(q[h, d])) * Fraction(float(kk[d])) for d in range(q.shape[1])), Fraction(0))
            if dot > 0:
                acc += Fraction(float(inp.w[i, h])) * dot
        out.append(acc * Fraction(float(inp.kscale[page, t % bs])))
    return out


def _tiny(kind="normal", seed=7, rows=3, heads=3, dim=5, bs=4, blocks=24, lens=(13, 1, 30), per_row=None):
    per_row = per_row or -(-max(lens) // bs)
    inp = W.make_fused_inputs(seed, rows, heads, dim, blocks, lens, (rows, per_row), block_size=bs,
                              q_std=1.0, k_std=1.0, kind=kind, k=8)
    return inp


def test_exact_against_fractions():
    inp = _tiny(blocks=24, per_row=8, lens=(13, 1, 30))
    scores = index_scores(inp)
    for i in range(inp.rows):
        ex = _exact_scores(inp, i)
        assert len(ex) == scores[i].size
        for t, e in enumerate(ex):
            ref = np.float32(float(e))
            # one rounding to fp32 after a float64 head sum: within 1 fp32 ulp
            assert abs(float(scores[i][t]) - float(ref)) <= float(np.spacing(np.float32(abs(ref)))) + 1e-30, (i, t)


def test_integer_inputs_are_bit_exact():
    inp = _tiny(kind="int", blocks=24, per_row=8, lens=(32, 17, 5))
    scores = index_scores(inp)
    for i in range(inp.rows):
        ex = _exact_scores(inp, i)
        assert all(e.denominator == 1 for e in ex)
        assert scores[i].tolist() == [float(e) for e in ex]


def test_single_product():
    q = np.zeros((2, 5), np.uint8)
    q[1, 3] = 0x38  # 1.0
    kc = np.zeros((2, 4, 5), np.uint8)
    kc[1, 2, 3] = 0x40  # 2.0 at block 1, offset 2
    kc[0, 0, 3] = 0xC0  # -2.0 at block 0 offset 0: relu removes it
    w = np.array([0.75, 0.5], np.float32)
    ks = np.full((2, 4), 3.0, np.float32)
    bt = np.array([1, 0])  # logical block 0 -> physical 1
    s = index_scores_row(q, w, kc, ks, bt, 8)
    exp = np.zeros(8, np.float32)
    exp[2] = 3.0 * 0.5 * 2.0
    assert s.tolist() == exp.tolist()


def test_zero_q_selects_lowest_indices():
    inp = W.make_fused_inputs(3, 2, 4, 16, 50, (700, 300), (2, 22), block_size=32, kind="zero_q")
    slots, idx, tops, _ = index_score_topk(inp)
    assert idx[0].tolist() == list(range(512))
    assert idx[1].tolist() == list(range(300)) + [-1] * 212
    assert (tops[0] == 0).all()


def test_scale_doubling_is_exact():
    inp = _tiny()
    a = index_scores(inp)
    inp.kscale = inp.kscale * np.float32(2.0)
    b = index_scores(inp)
    for x, y in zip(a, b):
        assert np.array_equal(2 * x, y)


def test_fused_topk_rank_rule_tiny():
    inp = W.make_fused_inputs(9, 2, 2, 4, 80, (300, 257), (2, 40), block_size=8, kind="int", k=50)
    slots, idx, tops, scores = index_score_topk(inp)
    for i in range(2):
        ex = np.array([float(e) for e in _exact_scores(inp, i)], np.float32)
        ref = rank_select_bruteforce(ex, 50)
        assert idx[i, : ref.size].tolist() == ref.tolist()
        pages = inp.block_table[i][ref // 8]
        assert slots[i, : ref.size].tolist() == (pages * 8 + ref % 8).tolist()
