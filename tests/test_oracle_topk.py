"""Pins of the oracle's window top-k and page transform (CPU only).

The selection is pinned by an O(n^2) rank rule that uses no sort, by closed
forms, by invariants, and by the packed-extend vs decode layout equivalence
that sglang PR #37889 ("Accuracy Tests": the packed-rows cases checked
against a row-local reference) uses to test ``row_starts`` / ``row_to_batch``.
"""

import numpy as np
import pytest

import workloads as W
from oracle.brute import rank_select_bruteforce
from oracle.topk import page_transform, topk_row, topk_transform

KINDS = ["normal", "bf16", "int", "const", "signed_zero", "inf", "ascending", "descending"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [0, 1, 7, 511, 512, 513, 1500])
def test_stable_sort_equals_rank_rule(kind, n):
    w = W.packed_extend_window(11, n, n, kind)
    for k in (1, 5, 512):
        got = topk_row(w, k)
        ref = rank_select_bruteforce(w, k)
        assert np.array_equal(got, ref), (kind, n, k)


def test_hand_example():
    # scores by index: 0:0.5 1:2 2:-1 3:2 4:-0 5:+0 6:3 7:-inf 8:+inf
    w = np.array([0.5, 2.0, -1.0, 2.0, -0.0, 0.0, 3.0, -np.inf, np.inf], np.float32)
    assert topk_row(w, 4).tolist() == [8, 6, 1, 3]
    assert topk_row(w, 7).tolist() == [8, 6, 1, 3, 0, 4, 5]
    assert topk_row(w, 20).tolist() == [8, 6, 1, 3, 0, 4, 5, 2, 7]


def test_constant_row_takes_lowest_indices():
    w = np.full(5000, -1.25, np.float32)
    assert topk_row(w, 512).tolist() == list(range(512))


def test_permutation_closed_form():
    rng = np.random.default_rng(5)
    n = 3000
    pi = rng.permutation(n)
    w = pi.astype(np.float32)
    inv = np.argsort(pi)
    assert topk_row(w, 512).tolist() == [int(inv[n - 1 - j]) for j in range(512)]


def test_short_row_returns_all_in_order():
    w = np.array([3.0, 1.0, 2.0], np.float32)
    s, i = topk_transform(w[None, :], np.array([3]), np.array([[10, 20, 30]]), 1, 8)
    assert i[0].tolist() == [0, 2, 1] + [-1] * 5
    assert s[0].tolist() == [10, 30, 20] + [-1] * 5


def test_empty_row_all_padding():
    s, i = topk_transform(np.zeros((1, 16), np.float32), np.array([0]), np.zeros((1, 16), np.int32), 1, 4)
    assert (s == -1).all() and (i == -1).all()


def test_invariants_large_row():
    w = W.packed_extend_window(3, 0, 66000, "bf16")
    k = 512
    sel = topk_row(w, k)
    assert sel.size == k and np.unique(sel).size == k
    assert sel.min() >= 0 and sel.max() < w.size
    mask = np.zeros(w.size, bool)
    mask[sel] = True
    lo = w[mask].min()
    hi = w[~mask].max()
    assert lo >= hi
    if lo == hi:  # ties at the cut: selected indices precede unselected ones
        assert np.flatnonzero(mask & (w == lo)).max() < np.flatnonzero(~mask & (w == lo)).min()
    # output order: score descending, ties by index ascending
    ws = w[sel]
    assert np.all((ws[:-1] > ws[1:]) | ((ws[:-1] == ws[1:]) & (sel[:-1] < sel[1:])))


def test_page_transform_closed_form():
    row = np.array([7, 3, 9], np.int32)
    assert page_transform(np.array([0, 5, 11, 4]), row, 4).tolist() == [28, 13, 39, 12]
    ident = np.arange(100, dtype=np.int32)
    idx = np.array([99, 0, 42])
    assert page_transform(idx, ident, 1).tolist() == idx.tolist()


def test_packed_equals_decode_layout():
    inp = W.packed_extend(seed=21, reqs=3, new_tokens=40, kv_len=900, fill=np.inf)
    s_packed, i_packed = topk_transform(inp.scores, inp.seq_lens, inp.page_tables, 1, 512,
                                        inp.row_starts, inp.row_to_batch)
    rows = inp.rows
    dec = np.zeros((rows, 900), np.float32)
    pt = np.zeros((rows, 900), np.int32)
    for i in range(rows):
        s0, n = int(inp.row_starts[i]), int(inp.seq_lens[i])
        dec[i, :n] = inp.scores[i, s0:s0 + n]
        pt[i] = inp.page_tables[inp.row_to_batch[i]]
    s_dec, i_dec = topk_transform(dec, inp.seq_lens, pt, 1, 512)
    assert np.array_equal(i_packed, i_dec) and np.array_equal(s_packed, s_dec)


def test_row_shuffle_permutes_outputs():
    inp = W.decode_topk(seed=8, rows=12, max_len=3000, min_len=100)
    s, i = topk_transform(inp.scores, inp.seq_lens, inp.page_tables, inp.page_size, 512)
    perm = np.random.default_rng(1).permutation(12)
    s2, i2 = topk_transform(inp.scores[perm], inp.seq_lens[perm], inp.page_tables[perm], inp.page_size, 512)
    assert np.array_equal(s[perm], s2) and np.array_equal(i[perm], i2)


def test_poison_outside_window_changes_nothing():
    a = W.packed_extend(seed=4, reqs=2, new_tokens=16, kv_len=1200, fill=0.0)
    b = W.packed_extend(seed=4, reqs=2, new_tokens=16, kv_len=1200, fill=np.inf)
    ra = topk_transform(a.scores, a.seq_lens, a.page_tables, 1, 512, a.row_starts, a.row_to_batch)
    rb = topk_transform(b.scores, b.seq_lens, b.page_tables, 1, 512, b.row_starts, b.row_to_batch)
    assert np.array_equal(ra[0], rb[0]) and np.array_equal(ra[1], rb[1])
