"""Pins of the oracle's bfloat16 decoding and bf16-cache index score (CPU only).

Decoding is checked on all 65536 patterns against torch's bfloat16 -> float32
conversion (a library routine, not the oracle's decoder). Scores are checked
against Python ``Fraction`` sums built from torch's decoding with the
block-table gather written out by hand, against the e4m3 path on integer
inputs that both formats hold exactly, and on hand-built single products at
extreme exponents (normal and subnormal keys).
"""

from fractions import Fraction

import numpy as np
import torch

import workloads as W
from oracle.bf16 import bf16_decode
from oracle.score import index_score_topk, index_scores, index_scores_row


def _dec(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns
        return t.to(torch.float32).numpy().astype(np.float64)


def test_decode_all_patterns():
    bits = np.arange(65536, dtype=np.int64).astype(np.uint16)
    got = bf16_decode(bits)
    ref = _dec(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_golden_values():
    """tests/golden/bf16_format_values.txt: patterns whose values follow from
    the format definition (min normal 2^-126, min subnormal 2^-133, largest
    finite (2 - 2^-7) 2^127, infinities, NaNs)."""
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "bf16_format_values.txt")
    bits, vals = [], []
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        b, v = line.split()
        bits.append(int(b, 16))
        vals.append(float(v))
    got = bf16_decode(np.array(bits, np.uint16))
    for b, g, v in zip(bits, got, vals):
        if np.isnan(v):
            assert np.isnan(g), hex(b)
        else:
            assert g == v and np.signbit(g) == np.signbit(v), (hex(b), g, v)


def test_decode_fields():
    assert bf16_decode(np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000], np.uint16)).tolist() == \
        [1.0, -2.0, 2.0**-133, (2 - 2**-7) * 2.0**127, -0.0]


def _exact_scores(inp, i):
    q = _dec(inp.q[i])
    b = i if inp.row_to_batch is None else int(inp.row_to_batch[i])
    bs = inp.kcache.shape[1]
    out = []
    for t in range(int(inp.seq_lens[i])):
        page = int(inp.block_table[b][t // bs])
        kk = _dec(inp.kcache[page, t % bs])
        acc = Fraction(0)
        for h in range(q.shape[0]):
            dot = sum((Fraction(float(q[h, d])) * Fraction(float(kk[d])) for d in range(q.shape[1])), Fraction(0))
            if dot > 0:
                acc += Fraction(float(inp.w[i, h])) * dot
        sc = 1 if inp.kscale is None else Fraction(float(inp.kscale[page, t % bs]))
        out.append(acc * sc)
    return out


def _tiny(kind="normal", seed=11, lens=(13, 1, 30), no_scale=False):
    bs = 4
    per_row = -(-max(lens) // bs)
    inp = W.make_fused_inputs(seed, len(lens), 3, 5, 3 * per_row + 2, lens, (len(lens), per_row), block_size=bs,
                              q_std=1.0, k_std=1.0, kind=kind, k=8, dtype="bf16")
    if no_scale:
        inp.kscale = None
    return inp


def test_exact_against_fractions():
    for no_scale in (False, True):
        inp = _tiny(no_scale=no_scale)
        scores = index_scores(inp)
        for i in range(inp.rows):
            ex = _exact_scores(inp, i)
            assert len(ex) == scores[i].size
            for t, e in enumerate(ex):
                ref = np.float32(float(e))
                assert abs(float(scores[i][t]) - float(ref)) <= float(np.spacing(np.float32(abs(ref)))) + 1e-30, (i, t)


def test_integer_inputs_match_the_e4m3_path():
    # integers in [-3, 3] are exact in both formats: the two paths must agree bit for bit
    a = W.make_fused_inputs(5, 3, 4, 16, 40, (90, 33, 150), (3, 12), block_size=16, kind="int", k=20, dtype="bf16")
    b = W.make_fused_inputs(5, 3, 4, 16, 40, (90, 33, 150), (3, 12), block_size=16, kind="int", k=20)
    assert np.array_equal(bf16_decode(a.q), _dec(a.q))
    for x, y in zip(index_scores(a), index_scores(b)):
        assert np.array_equal(x, y)
    sa, ia, _, _ = index_score_topk(a)
    sb, ib, _, _ = index_score_topk(b)
    assert np.array_equal(sa, sb) and np.array_equal(ia, ib)


def test_single_products_at_extreme_exponents():
    q = np.zeros((2, 3), np.uint16)
    q[0, 2] = 0x5F80  # 2^64
    q[1, 0] = 0x3F80  # 1.0
    kc = np.zeros((2, 4, 3), np.uint16)
    kc[0, 1, 2] = 0x2080  # 2^-62: q0 . k = 4
    kc[1, 3, 0] = 0x0001  # 2^-133 (smallest subnormal): q1 . k = 2^-133
    kc[1, 2, 0] = 0xBF80  # -1: relu removes it
    w = np.array([0.5, 2.0], np.float32)
    bt = np.array([1, 0])  # logical block 0 -> physical 1
    s = index_scores_row(q, w, kc, None, bt, 8, dtype="bf16")
    exp = np.zeros(8, np.float64)
    exp[3] = 2.0 * 2.0**-133
    exp[5] = 0.5 * 4.0
    assert s.tolist() == exp.astype(np.float32).tolist()
