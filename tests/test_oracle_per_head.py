"""Pins of the oracle's per-index-head scores and top-k (CPU only).

Exact values come from Python ``Fraction`` sums over torch's e4m3 decoding
(a library routine) with the block-table gather written out by hand; the
head sum of the per-head scores must equal the (separately pinned)
head-summed score on integer inputs; a one-head input must select exactly
what the head-summed path selects; each head's selection must equal the
brute-force rank rule; a head with zero weight selects its first k keys.
"""

from fractions import Fraction

import numpy as np
import torch

import workloads as W
from oracle.brute import rank_select_bruteforce
from oracle.score import index_score_topk, index_score_topk_per_head, index_scores, index_scores_per_head


def _dec(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def test_exact_against_fractions():
    inp = W.make_fused_inputs(21, 2, 3, 5, 12, (9, 14), (2, 4), block_size=4, q_std=1.0, k_std=1.0, k=8)
    ph = index_scores_per_head(inp)
    for i in range(inp.rows):
        q = _dec(inp.q[i])
        for t in range(int(inp.seq_lens[i])):
            page = int(inp.block_table[i][t // 4])
            kk = _dec(inp.kcache[page, t % 4])
            for h in range(3):
                dot = sum((Fraction(float(q[h, d])) * Fraction(float(kk[d])) for d in range(5)), Fraction(0))
                ex = max(dot, Fraction(0)) * Fraction(float(inp.w[i, h])) * Fraction(float(inp.kscale[page, t % 4]))
                ref = np.float32(float(ex))
                got = float(ph[i][h, t])
                assert abs(got - float(ref)) <= float(np.spacing(np.float32(abs(ref)))) + 1e-30, (i, h, t)


def test_head_sum_equals_summed_score_on_integers():
    inp = W.make_fused_inputs(22, 3, 6, 16, 30, (40, 1, 97), (3, 10), block_size=16, kind="int", k=20)
    for ph, hs in zip(index_scores_per_head(inp), index_scores(inp)):
        assert ph.shape[0] == 6
        assert np.array_equal(ph.astype(np.float64).sum(axis=0), hs.astype(np.float64))


def test_one_head_selects_like_the_summed_path():
    inp = W.make_fused_inputs(23, 2, 1, 8, 40, (300, 77), (2, 20), block_size=16, k=64)
    s1, i1, _ = index_score_topk_per_head(inp)
    s2, i2, _, _ = index_score_topk(inp)
    assert np.array_equal(i1[:, 0, :], i2) and np.array_equal(s1[:, 0, :], s2)


def test_each_head_follows_the_rank_rule():
    inp = W.make_fused_inputs(24, 2, 4, 8, 70, (250, 130), (2, 32), block_size=8, kind="int", k=50)
    slots, idx, scores = index_score_topk_per_head(inp)
    for i in range(2):
        for h in range(4):
            ref = rank_select_bruteforce(scores[i][h], 50)
            assert idx[i, h, : ref.size].tolist() == ref.tolist()
            assert (idx[i, h, ref.size:] == -1).all()
            pages = inp.block_table[i][ref // 8]
            assert slots[i, h, : ref.size].tolist() == (pages * 8 + ref % 8).tolist()


def test_zero_weight_head_takes_the_first_keys():
    inp = W.make_fused_inputs(25, 1, 3, 8, 40, (200,), (1, 25), block_size=8, k=32)
    inp.w[0, 1] = 0.0
    _, idx, scores = index_score_topk_per_head(inp)
    assert (scores[0][1] == 0).all()
    assert idx[0, 1].tolist() == list(range(32))
