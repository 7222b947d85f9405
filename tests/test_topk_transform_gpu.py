"""GPU parity of sai_topk_transform against the CPU oracle (bit-exact).

Indices and slots are integer outputs selected from given fp32 scores, so
they must equal the oracle's exactly, element by element.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle.blocks import sparse_blocks as oracle_blocks
from oracle.topk import topk_transform as oracle_topk
from parity_pool import check_packed_extend_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _t(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _run(inp, force_single=False, scores_t=None, block_size=None):
    """GPU (slots, indices), plus (blocks, counts) built by the same call when
    block_size is given."""
    import sparse_attention_indexer_top_gb300 as sai

    ws = torch.empty(16, dtype=torch.uint8, device=DEV) if force_single else None
    s = _t(inp.scores) if scores_t is None else scores_t
    out = sai.topk_transform(s, _t(inp.seq_lens), _t(inp.page_tables), page_size=inp.page_size,
                             row_starts=_t(inp.row_starts), row_to_batch=_t(inp.row_to_batch), want_indices=True,
                             want_blocks=block_size is not None, block_size=block_size or 128, workspace=ws)
    torch.cuda.synchronize()
    assert sai.device_status() == 0
    return tuple(t.cpu().numpy() for t in out)


def _oracle(inp, rows=None, block_size=None):
    slots, idx = oracle_topk(inp.scores, inp.seq_lens, inp.page_tables, inp.page_size, 512, inp.row_starts,
                             inp.row_to_batch, rows=rows)
    if block_size is None:
        return slots, idx
    return (slots, idx) + oracle_blocks(slots, block_size)


def _assert_equal(got, ref, what=""):
    assert len(got) == len(ref)
    bad = np.zeros(got[0].shape[0], bool)
    for g, r in zip(got, ref):
        bad |= (g != r).reshape(g.shape[0], -1).any(axis=1)
    bad = np.flatnonzero(bad)
    assert bad.size == 0, f"{what}: {bad.size} rows differ, first {bad[:5]}"


def test_tiny_decode():
    inp = W.tiny_decode()
    _assert_equal(_run(inp), _oracle(inp), "tiny decode")
    _assert_equal(_run(inp, block_size=128), _oracle(inp, block_size=128), "tiny decode, block lists")


def test_decode_long_rows_split_ties():
    """Few rows longer than two split pieces (rows of 33K-60K bf16-rounded
    scores, so ties are certain): split over CTAs and merged, with the block
    lists built by the merge."""
    inp = W.decode_topk(seed=24, rows=40, min_len=33000, max_len=60000)
    _assert_equal(_run(inp, block_size=128), _oracle(inp, block_size=128), "long decode rows")


@pytest.mark.parametrize("single", [False, True])
def test_decode_bf16_ties(single):
    # the decode workload's page size is 128: the block lists are the
    # distinct pages of the selected slots (split rows: built by the merge)
    inp = W.decode_topk()
    _assert_equal(_run(inp, force_single=single, block_size=128), _oracle(inp, block_size=128),
                  f"decode single={single}")


@pytest.mark.parametrize("kind", ["normal", "bf16", "int", "const", "signed_zero", "inf", "ascending", "descending"])
@pytest.mark.parametrize("single", [False, True])
def test_value_kinds(kind, single):
    # around k, one and two 1024/2048/3072-score stages, and long rows
    lens = [0, 1, 3, 7, 9, 100, 511, 512, 513, 2047, 2048, 2049, 3071, 3072, 3073, 6000, 6143, 6145, 9001, 20000,
            33333]
    inp = W.make_topk_inputs(31, lens, 33340, 128, (len(lens), 261), kind=kind, fill=np.inf)
    _assert_equal(_run(inp, force_single=single, block_size=64), _oracle(inp, block_size=64), kind)


@pytest.mark.parametrize("stride_pad", [0, 1, 2, 3])
def test_packed_extend_ragged(stride_pad):
    # stride not a multiple of 4 and odd row starts: scalar heads/tails
    inp = W.packed_extend(seed=12, reqs=3, new_tokens=97, kv_len=12345, fill=np.inf, stride_pad=stride_pad)
    _assert_equal(_run(inp), _oracle(inp), f"packed pad={stride_pad}")
    _assert_equal(_run(inp, force_single=True), _oracle(inp), f"packed single pad={stride_pad}")


@pytest.mark.parametrize("block_size", [1, 7, 9, 16, 128, 1 << 20])
def test_block_lists_block_sizes(block_size):
    """Block lists built by the top-k call for page size 1 slots of a
    140000-slot pool: one slot per block (block_size 1, blocks spanning far
    more than the 16384 ids of the bitmap; 7 likewise), spans of ~15600 and
    ~8750 blocks (9, 16: bitmap words beyond the first 128 and 256, i.e.
    every thread's second to fourth word), ~1100 blocks (128), and one block
    for everything."""
    inp = W.packed_extend(seed=17, reqs=2, new_tokens=40, kv_len=70000, fill=np.inf)
    _assert_equal(_run(inp, block_size=block_size), _oracle(inp, block_size=block_size), f"bs={block_size}")
    _assert_equal(_run(inp, force_single=True, block_size=block_size), _oracle(inp, block_size=block_size),
                  f"single bs={block_size}")


@pytest.mark.parametrize("single", [False, True])
def test_row_to_row_scale_changes(single):
    # Rows whose scale jumps by 1e3 between neighbours: a threshold carried
    # over from one row to the next is often far too high or too low.
    lens = np.random.default_rng(3).integers(0, 3000, size=2500).astype(np.int32)
    lens[::7] = 512
    inp = W.make_topk_inputs(33, lens, 3001, 1, (2500, 3001), kind="scaled", fill=np.inf)
    _assert_equal(_run(inp, force_single=single), _oracle(inp), "scaled rows")


def test_unaligned_base_pointer():
    inp = W.packed_extend(seed=13, reqs=2, new_tokens=50, kv_len=7001, fill=np.inf)
    big = np.full((inp.rows, inp.scores.shape[1] + 1), np.inf, np.float32)
    big[:, 1:] = inp.scores
    view = _t(big)[:, 1:]  # base pointer 4 bytes past a 16-byte boundary
    _assert_equal(_run(inp, scores_t=view), _oracle(inp), "unaligned base")


def test_many_rows_single_unit_path():
    inp = W.packed_extend(seed=14, reqs=2, new_tokens=400, kv_len=3000, fill=np.inf)
    _assert_equal(_run(inp), _oracle(inp), "many rows")


def test_packed_equals_decode_layout():
    inp = W.packed_extend(seed=15, reqs=2, new_tokens=64, kv_len=9000, fill=np.inf)
    got_packed = _run(inp)
    dec = np.zeros((inp.rows, 9000), np.float32)
    pt = np.zeros((inp.rows, 9000), np.int32)
    for i in range(inp.rows):
        s0, n = int(inp.row_starts[i]), int(inp.seq_lens[i])
        dec[i, :n] = inp.scores[i, s0:s0 + n]
        pt[i] = inp.page_tables[inp.row_to_batch[i]]
    dinp = W.TopkInputs(dec, inp.seq_lens, pt, 1)
    got_dec = _run(dinp)
    _assert_equal(got_packed, got_dec, "packed vs decode layout")


def test_indices_only_without_page_table():
    import sparse_attention_indexer_top_gb300 as sai

    inp = W.tiny_decode(seed=9)
    idx = sai.topk_transform(_t(inp.scores), _t(inp.seq_lens))
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), _oracle(inp)[1])


def test_bad_row_metadata_is_flagged_and_emptied():
    import sparse_attention_indexer_top_gb300 as sai

    inp = W.make_topk_inputs(5, [100, 600, 700], 1000, 1, (3, 1000), row_starts=[0, 0, 0])
    bad_starts = np.array([0, 500, 0], np.int32)  # row 1: 500 + 600 > stride 1000
    slots, idx = sai.topk_transform(_t(inp.scores), _t(inp.seq_lens), _t(inp.page_tables),
                                    row_starts=_t(bad_starts), want_indices=True)
    bits = sai.device_status(clear=True)
    assert bits & 1
    ref = _oracle(inp, rows=[0, 2])
    assert np.array_equal(idx.cpu().numpy()[[0, 2]], ref[1])
    assert (idx.cpu().numpy()[1] == -1).all() and (slots.cpu().numpy()[1] == -1).all()
    assert sai.device_status() == 0


def test_packed_extend_full_size():
    """The packed-extend prefill workload at full size ([16384, 140000]
    scores, two requests on a 70000-token KV, +inf outside the windows), in
    the launch configuration the benchmark times, with the block lists of
    128-token blocks built by the same call; every row against the oracle,
    element by element (the oracle runs in a pool of processes over the host
    cores, each regenerating its rows' windows from the seed)."""
    import sparse_attention_indexer_top_gb300 as sai

    row_starts, seq_lens, r2b, width = W.packed_extend_meta()
    rows = seq_lens.size
    scores = torch.empty((rows, width), dtype=torch.float32, device=DEV)
    chunk = 1024
    host = torch.empty((chunk, width), dtype=torch.float32).pin_memory()
    hn = host.numpy()
    for r0 in range(0, rows, chunk):
        W.fill_rows(hn, r0, 3, row_starts, seq_lens, fill=np.inf)
        scores[r0:r0 + chunk].copy_(host)
    pt = W.page_table_perm(3, (2, 70000))
    slots, idx, blocks, counts = sai.topk_transform(scores, _t(seq_lens), _t(pt), row_starts=_t(row_starts),
                                                    row_to_batch=_t(r2b), want_indices=True, want_blocks=True,
                                                    block_size=128)
    torch.cuda.synchronize()
    assert sai.device_status() == 0
    bad = check_packed_extend_rows(3, seq_lens, r2b, pt, 1, 512, slots.cpu().numpy(), idx.cpu().numpy(),
                                   blocks=blocks.cpu().numpy(), counts=counts.cpu().numpy(), block_size=128)
    assert not bad, f"{len(bad)} rows differ: {bad[:5]}"


def test_chunked_prefix_calls_match_one_call():
    """Chunked-prefix-cache extend: the packed plan (row_starts, seq_lens,
    row_to_batch) covers the whole forward, but each call holds one chunk of
    the score rows and that chunk's slice of the plan. Each chunk's outputs
    equal the rows of one call over everything, and the oracle."""
    import sparse_attention_indexer_top_gb300 as sai

    inp = W.packed_extend(seed=16, reqs=2, new_tokens=150, kv_len=6000, fill=np.inf)
    whole = _run(inp)
    _assert_equal(whole, _oracle(inp), "one call vs oracle")
    pt = _t(inp.page_tables)
    for lo, hi in ((0, 70), (70, 151), (151, 300)):
        slots, idx = sai.topk_transform(_t(inp.scores[lo:hi]), _t(inp.seq_lens[lo:hi]), pt, page_size=inp.page_size,
                                        row_starts=_t(inp.row_starts[lo:hi]), row_to_batch=_t(inp.row_to_batch[lo:hi]),
                                        want_indices=True)
        torch.cuda.synchronize()
        assert sai.device_status() == 0
        _assert_equal((slots.cpu().numpy(), idx.cpu().numpy()), (whole[0][lo:hi], whole[1][lo:hi]), f"chunk {lo}:{hi}")


@pytest.mark.parametrize("single", [True, False])
def test_sampled_start_threshold_too_high_is_redone(single):
    """A unit with no threshold carried from its CTA's previous unit starts
    from one estimated on 1024 evenly spaced samples of its window. Here the
    largest scores sit exactly at those positions, so the estimate lies above
    the 512th score and fewer than 512 scores pass: the unit must be redone
    exactly. (White-box: the positions are the kernel's sample positions,
    (2j + 1) * n / 2048, for a window of n scores.)"""
    rows, n = 6, 65536
    rng = np.random.default_rng(71)
    scores = rng.standard_normal((rows, n)).astype(np.float32)
    pos = ((2 * np.arange(1024, dtype=np.int64) + 1) * n) // 2048
    scores[:, pos] = (100.0 + rng.permutation(1024)).astype(np.float32)
    pt = rng.permutation(rows * n).astype(np.int32).reshape(rows, n)
    inp = W.TopkInputs(scores, np.full(rows, n, np.int32), pt, 1)
    _assert_equal(_run(inp, force_single=single), _oracle(inp), "sampled threshold redo")


def test_sampled_start_threshold_short_and_mixed_rows():
    """First units of many CTAs with windows of 1535..70000 scores, including
    heavy ties (bf16-rounded values) and a constant row."""
    rng = np.random.default_rng(72)
    lens = np.array([4096, 4097, 9000, 30000, 70000, 65536, 5000, 12000, 1535, 1536, 2048, 3000], np.int32)
    width = int(lens.max())
    scores = rng.standard_normal((lens.size, width)).astype(np.float32)
    scores[1] = torch.from_numpy(scores[1]).to(torch.bfloat16).float().numpy()
    scores[5] = 3.0
    pt = rng.permutation(lens.size * width).astype(np.int32).reshape(lens.size, width)
    inp = W.TopkInputs(scores, lens, pt, 1)
    _assert_equal(_run(inp, force_single=True), _oracle(inp), "mixed rows")
    _assert_equal(_run(inp), _oracle(inp), "mixed rows, split path")
