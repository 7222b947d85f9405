"""GPU parity of the per-index-head scores and top-k against the CPU oracle.

Scores: each head's summand of the index score. A single 128-term dot
product accumulated in FP32 is off by at most ~128 * 2^-24 of the sum of its
terms' magnitudes, and a head's score (unlike the head sum) can sit near
zero through cancellation, so the bound is |gpu - oracle| <= 1e-3 |oracle| +
1e-5 A, with A the same score over |q| and |k| (the oracle on sign-cleared
codes). Integer-valued inputs make every score an exact integer on both
sides (bit-exact, pins the per-head store layout). Selection per (row,
head): count, range and distinctness exact, every pick's oracle score at
least the oracle k-th score minus the tolerance, picks in non-increasing
oracle order within it, slots equal to the transform of the GPU's own
indices.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle.score import index_scores_per_head

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
TOL = 1e-3


def _t(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _dev(inp):
    if inp.dtype == "bf16":
        def elem(a):
            return _t(a.view(np.int16)).view(torch.bfloat16)
    else:
        elem = _t
    return dict(q=elem(inp.q), w=_t(inp.w), kcache=elem(inp.kcache), kscale=_t(inp.kscale),
                block_table=_t(inp.block_table), seq_lens=_t(inp.seq_lens), row_to_batch=_t(inp.row_to_batch))


def _abs_inputs(inp):
    """The same inputs with every q and key element replaced by its magnitude."""
    import copy

    a = copy.copy(inp)
    mask = 0x7FFF if inp.dtype == "bf16" else 0x7F
    a.q = inp.q & inp.q.dtype.type(mask)
    a.kcache = inp.kcache & inp.kcache.dtype.type(mask)
    return a


def _kth(s, k):
    return float(np.sort(s)[::-1][min(s.size, k) - 1]) if s.size else 0.0


def _small(kind="normal", dtype="e4m3", seed=61, lens=(1, 127, 128, 300, 1000, 2500)):
    lens = np.asarray(lens, np.int32)
    rows = lens.size
    per_row = int(-(-lens.max() // 128))
    return W.make_fused_inputs(seed, rows, 64, 128, rows * per_row + 3, lens, (rows, per_row), kind=kind,
                               dtype=dtype)


def _dense(inp):
    import sparse_attention_indexer_top_gb300 as sai

    d = _dev(inp)
    out = sai.index_score_per_head(d["q"], d["w"], d["kcache"], d["kscale"], d["block_table"], d["seq_lens"],
                                   max_seq_len=int(inp.seq_lens.max()), row_to_batch=d["row_to_batch"])
    torch.cuda.synchronize()
    assert sai.device_status() == 0
    return out.cpu().numpy()


def _topk(inp):
    import sparse_attention_indexer_top_gb300 as sai

    d = _dev(inp)
    slots, idx = sai.index_score_topk_per_head(d["q"], d["w"], d["kcache"], d["kscale"], d["block_table"],
                                               d["seq_lens"], max_seq_len=int(inp.seq_lens.max()),
                                               row_to_batch=d["row_to_batch"])
    torch.cuda.synchronize()
    assert sai.device_status() == 0
    return slots.cpu().numpy(), idx.cpu().numpy()


def _check_dense(got, inp, exact=False):
    ref = index_scores_per_head(inp)
    mag = index_scores_per_head(_abs_inputs(inp))
    for i in range(inp.rows):
        n = int(inp.seq_lens[i])
        g = got[i, :, :n].astype(np.float64)
        r = ref[i].astype(np.float64)
        if exact:
            assert np.array_equal(g, r), f"row {i}: first diff at {np.argwhere(g != r)[:3]}"
        else:
            bound = TOL * np.abs(r) + 1e-5 * mag[i].astype(np.float64)
            bad = np.argwhere(np.abs(g - r) > bound)
            assert bad.size == 0, f"row {i}: {len(bad)} scores off, first (head, key) {bad[:3].tolist()}"


def _check_topk(got, inp, rows=None, heads=range(64), k=512):
    slots, idx = got
    rows = list(range(inp.rows)) if rows is None else rows
    ref = index_scores_per_head(inp, rows)
    mag = index_scores_per_head(_abs_inputs(inp), rows)
    for j, i in enumerate(rows):
        n = int(inp.seq_lens[i])
        kk = min(n, k)
        b = i if inp.row_to_batch is None else int(inp.row_to_batch[i])
        for h in heads:
            gi = idx[i, h]
            assert (gi[kk:] == -1).all() and (slots[i, h, kk:] == -1).all(), f"row {i} head {h}: padding"
            sel = gi[:kk].astype(np.int64)
            assert (sel >= 0).all() and (sel < n).all(), f"row {i} head {h}: index range"
            assert np.unique(sel).size == kk, f"row {i} head {h}: duplicates"
            s = ref[j][h].astype(np.float64)
            s_k = _kth(ref[j][h], k)
            tol = TOL * abs(s_k) + 1e-5 * float(mag[j][h].max(initial=0.0)) + 1e-30
            assert (s[sel] >= s_k - tol).all(), f"row {i} head {h}: a pick below the k-th score"
            assert (np.diff(s[sel]) <= TOL * np.abs(s[sel][:-1]) + tol).all(), f"row {i} head {h}: not score-descending"
            pages = inp.block_table[b][sel // 128].astype(np.int64)
            assert np.array_equal(slots[i, h, :kk], pages * 128 + sel % 128), f"row {i} head {h}: slots"


@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
def test_dense_integer_inputs_exact(dtype):
    inp = _small("int", dtype=dtype)
    _check_dense(_dense(inp), inp, exact=True)


@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
def test_dense_normal_inputs(dtype):
    inp = _small("normal", dtype=dtype, seed=62)
    _check_dense(_dense(inp), inp)


@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
def test_topk_small(dtype):
    inp = _small("normal", dtype=dtype, seed=63)
    if dtype == "bf16":
        inp.kscale = None
    _check_topk(_topk(inp), inp)


def test_topk_zero_q_takes_lowest_indices():
    inp = _small("zero_q")
    slots, idx = _topk(inp)
    for i in range(inp.rows):
        kk = min(int(inp.seq_lens[i]), 512)
        assert (idx[i, :, :kk] == np.arange(kk)[None, :]).all()


def test_topk_packed_requests():
    lens, r2b = [], []
    for b, (p, nr) in enumerate(zip([2900, 700], [5, 3])):
        lens += [p + i + 1 for i in range(nr)]
        r2b += [b] * nr
    per_row = -(-max(lens) // 128)
    inp = W.make_fused_inputs(64, len(lens), 64, 128, 2 * per_row + 5, lens, (2, per_row), row_to_batch=r2b)
    _check_topk(_topk(inp), inp)


def test_topk_decode_full_size_sampled():
    """The fused decode workload (64 rows, U[4096, 32768] keys): every head of
    a sample of rows against the oracle."""
    inp = W.fused_decode()
    got = _topk(inp)
    _check_topk(got, inp, rows=[0, 7, 31, 63])
