"""GPU parity of the fused index score (+ top-k) against the CPU oracle, for
the FP8 index cache and the bf16 one.

Scores: the oracle forms the FP8 dot products exactly, the kernel in FP32 on
the tensor cores; they must agree within 1e-3 relative (floored at the row's
k-th score). Integer-valued inputs make every score an exact integer on both
sides, so there the comparison is bit-exact and pins the MMA operand layout.
Selection: a GPU pick is accepted when its oracle score is at least the
oracle's k-th score minus that tolerance; the count, distinctness, order
(score descending, equal GPU scores by ascending index) and the slot
transform of the GPU's own indices are checked exactly. The full-size
workloads are checked on every row, in a pool of processes over the host
cores (tests/parity_pool.py).
"""

import time

import numpy as np
import pytest
import torch

import workloads as W
from oracle.score import index_scores
from parity_pool import TOL, check_fused_all_rows, check_fused_rows, kth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _t(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _dev_inputs(inp):
    if inp.dtype == "bf16":  # uint16 bit patterns -> torch.bfloat16
        def elem(a):
            return _t(a.view(np.int16)).view(torch.bfloat16)
    else:
        elem = _t
    return dict(q=elem(inp.q), w=_t(inp.w), kcache=elem(inp.kcache), kscale=_t(inp.kscale),
                block_table=_t(inp.block_table), seq_lens=_t(inp.seq_lens), row_to_batch=_t(inp.row_to_batch))


def _dense(inp, group_rows=1):
    import sparse_attention_indexer_top_gb300 as sai

    d = _dev_inputs(inp)
    max_len = int(inp.seq_lens.max()) if inp.rows else 0
    out = sai.index_score(d["q"], d["w"], d["kcache"], d["kscale"], d["block_table"], d["seq_lens"],
                          max_seq_len=max_len, row_to_batch=d["row_to_batch"], group_rows=group_rows)
    torch.cuda.synchronize()
    assert sai.device_status() == 0
    return out.cpu().numpy()


def _fused(inp, group_rows=1, block_size=None):
    """GPU (slots, indices, scores), plus (blocks, counts) built by the same
    call when block_size is given."""
    import sparse_attention_indexer_top_gb300 as sai

    d = _dev_inputs(inp)
    max_len = int(inp.seq_lens.max()) if inp.rows else 0
    out = sai.index_score_topk(d["q"], d["w"], d["kcache"], d["kscale"], d["block_table"], d["seq_lens"],
                               max_seq_len=max_len, row_to_batch=d["row_to_batch"], group_rows=group_rows,
                               want_blocks=block_size is not None, block_size=block_size or 128)
    torch.cuda.synchronize()
    assert sai.device_status() == 0
    return tuple(t.cpu().numpy() for t in out)


def _check_dense(got, inp, exact=False, rows=None):
    rows = list(range(inp.rows)) if rows is None else rows
    ref = index_scores(inp, rows)
    for j, i in enumerate(rows):
        n = int(inp.seq_lens[i])
        g = got[i, :n].astype(np.float64)
        r = ref[j].astype(np.float64)
        if exact:
            assert np.array_equal(g, r), f"row {i}: first diff at {np.flatnonzero(g != r)[:5]}"
        else:
            floor = abs(kth(ref[j], 512)) if n else 0.0
            err = np.abs(g - r) / np.maximum(np.maximum(np.abs(r), floor), 1e-30)
            assert err.max() <= TOL, f"row {i}: max rel err {err.max():.3e} at {int(err.argmax())}"


def _check_topk(got, inp, rows=None, k=512, block_size=128):
    slots, idx, scores = got[:3]
    blocks, counts = got[3:] if len(got) == 5 else (None, None)
    rows = list(range(inp.rows)) if rows is None else rows
    bad = check_fused_rows(inp, rows, index_scores(inp, rows), slots, idx, scores, k, blocks, counts, block_size)
    assert not bad, f"{len(bad)} rows fail: {bad[:5]}"


def _check_all_rows_in_pool(got, inp, block_size=128):
    """Every row against the oracle, the rows spread over the host cores."""
    slots, idx, scores = got[:3]
    blocks, counts = got[3:] if len(got) == 5 else (None, None)
    bad = check_fused_all_rows(inp, slots, idx, scores, blocks=blocks, counts=counts, block_size=block_size)
    assert not bad, f"{len(bad)} rows fail: {bad[:5]}"


def _small(kind="normal", rows=6, lens=(1, 127, 128, 300, 1000, 2500), seed=41, dtype="e4m3"):
    lens = np.asarray(lens[:rows], np.int32)
    per_row = int(-(-lens.max() // 128))
    return W.make_fused_inputs(seed, rows, 64, 128, rows * per_row + 3, lens, (rows, per_row), kind=kind,
                               dtype=dtype)


def test_dense_integer_inputs_exact():
    _check_dense(_dense(_small("int")), _small("int"), exact=True)


def test_dense_normal_inputs():
    inp = _small("normal")
    _check_dense(_dense(inp), inp)


def test_dense_grouped_rows_exact():
    # 8 rows of two requests (4 each), causal lengths, one block table row per request
    lens = np.array([997, 998, 999, 1000, 3001, 3002, 3003, 3004], np.int32)
    inp = W.make_fused_inputs(43, 8, 64, 128, 2 * 24 + 1, lens, (2, 24), row_to_batch=[0, 0, 0, 0, 1, 1, 1, 1],
                              kind="int")
    _check_dense(_dense(inp, group_rows=4), inp, exact=True)


def test_topk_small():
    inp = _small("normal")
    _check_topk(_fused(inp), inp)


def test_topk_zero_q_takes_lowest_indices():
    inp = _small("zero_q")
    slots, idx, scores = _fused(inp)
    for i in range(inp.rows):
        kk = min(int(inp.seq_lens[i]), 512)
        assert idx[i][:kk].tolist() == list(range(kk))


def test_topk_grouped_prefill_like():
    rows, kv = 64, 6000
    lens = (kv - rows + 1 + np.arange(rows)).astype(np.int32)
    blocks = -(-kv // 128)
    inp = W.make_fused_inputs(44, rows, 64, 128, blocks, lens, (1, blocks), row_to_batch=np.zeros(rows, np.int32))
    _check_topk(_fused(inp, group_rows=4), inp)


def test_topk_decode_many_chunks():
    inp = W.fused_decode(seed=45, rows=16, min_len=3000, max_len=20000)
    _check_topk(_fused(inp), inp)


def test_fused_decode_full_size():
    """The fused decode workload at full size (64 rows, 64 heads x 128,
    seq_lens U[4096, 32768], 16384-block pool), every row checked, with the
    per-row lists of 128-token KV blocks built by the same call (the merge)."""
    inp = W.fused_decode()
    _check_topk(_fused(inp), inp)
    _check_topk(_fused(inp, block_size=128), inp)


def test_fused_prefill_full_size():
    """The fused prefill workload at full size (4096 causal rows on a 32768-
    token KV, grouped by 4), in the launch configuration the benchmark times;
    every row against the oracle."""
    inp = W.fused_prefill()
    _check_all_rows_in_pool(_fused(inp, group_rows=4), inp)


def test_start_threshold_replay():
    """A unit whose sampled tiles hold far higher scores than the rest of it:
    the start threshold set from the sample then lets fewer than 512 of the
    unit's keys through, so the unit must be streamed again with no
    threshold. Four rows of 32768 keys are split into chunks as the host
    plan splits them (every unit of at least 16 tiles streams from its
    middle tile, so its first 8 tiles are the sample); in one chunk of each
    row the sampled tiles' keys get a 64x scale. The row's top 512 then lies
    among those 1024 keys, while without the replay that chunk would report
    only the few hundred that reached its threshold."""
    rows, n = 4, 32768
    per_row = n // 128
    inp = W.make_fused_inputs(48, rows, 64, 128, rows * per_row, np.full(rows, n, np.int32), (rows, per_row))
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    chunks = max(1, min(-(-4 * sms // rows), 12, per_row))  # the plan: about four units per SM, at most 12
    cb = -(-per_row // chunks)
    boosted = 0
    for r in range(rows):
        c = 1 + r  # a different chunk in each row
        start = c * cb
        tiles = min(cb, per_row - start)
        assert tiles >= 16 and tiles * 128 >= 2048, "the chunk must sample"
        for i in range(8):
            t = start + (i + tiles // 2) % tiles
            inp.kscale[inp.block_table[r, t]] *= np.float32(64.0)
            boosted += 1
    assert boosted == 8 * rows
    got = _fused(inp)
    _check_topk(got, inp)
    # every selected key comes from the boosted tiles
    for r in range(rows):
        c = 1 + r
        tiles = min(cb, per_row - c * cb)
        sampled = {c * cb + (i + tiles // 2) % tiles for i in range(8)}
        assert set((got[1][r] // 128).tolist()) <= sampled, f"row {r}: a pick outside the boosted tiles"


def test_start_threshold_replay_grouped_rows():
    """The replay in a four-row group where one row does not fail: the four
    rows share a request's 32768 keys, one chunk's sampled tiles get a 64x
    key scale (rows 0, 2 and 3 then let too few keys through and replay it),
    while row 1 has q = 0 (every score 0, so every key reaches its
    threshold): during the replay row 1 only frees the accumulator buffers,
    and all four rows must still come out exact."""
    rows, n = 4, 32768
    per_row = n // 128
    inp = W.make_fused_inputs(49, rows, 64, 128, per_row + 8, np.full(rows, n, np.int32), (1, per_row),
                              row_to_batch=np.zeros(rows, np.int32))
    inp.q[1] = 0  # e4m3 code 0 = +0
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    chunks = max(1, min(-(-4 * sms // 1), 12, per_row))  # one group of four rows
    cb = -(-per_row // chunks)
    c = 2
    tiles = min(cb, per_row - c * cb)
    assert tiles >= 16 and tiles * 128 >= 2048, "the chunk must sample"
    sampled = [c * cb + (i + tiles // 2) % tiles for i in range(8)]
    for t in sampled:
        inp.kscale[inp.block_table[0, t]] *= np.float32(64.0)
    got = _fused(inp, group_rows=4)
    _check_topk(got, inp)
    for r in (0, 2, 3):
        assert set((got[1][r] // 128).tolist()) <= set(sampled), f"row {r}: a pick outside the boosted tiles"
    assert np.array_equal(got[1][1], np.arange(512)), "row 1: equal scores go to the lowest indices"


@pytest.mark.parametrize("block_size", [128, 256, 1])
def test_fused_block_lists(block_size):
    """Block lists built by the fused call's last stage: the ranking path
    (one KV chunk per row: grouped prefill rows) and the merge path (decode
    rows over several chunks)."""
    rows, kv = 64, 6000
    lens = (kv - rows + 1 + np.arange(rows)).astype(np.int32)
    blocks = -(-kv // 128)
    inp = W.make_fused_inputs(44, rows, 64, 128, blocks, lens, (1, blocks), row_to_batch=np.zeros(rows, np.int32))
    _check_topk(_fused(inp, group_rows=4, block_size=block_size), inp, block_size=block_size)
    dec = W.fused_decode(seed=45, rows=16, min_len=3000, max_len=20000)
    _check_topk(_fused(dec, block_size=block_size), dec, block_size=block_size)


@pytest.mark.parametrize("kind", ["normal", "int"])
def test_topk_one_chunk_per_row(kind):
    """640 single rows give one KV chunk per row, so the fused kernel ranks
    each row's 512 and writes the outputs itself (no merge pass); integer
    inputs make many equal scores, which sends the ranking to its fallback."""
    rows, per_row = 640, 12
    lens = np.random.default_rng(47).integers(1, per_row * 128 + 1, size=rows).astype(np.int32)
    inp = W.make_fused_inputs(47, rows, 64, 128, rows * per_row + 1, lens, (rows, per_row), kind=kind)
    _check_topk(_fused(inp), inp)


def _packed_requests(seed, new_rows, prefixes, dtype="e4m3"):
    """Several requests packed into one call: request b contributes
    new_rows[b] query rows, causal on a KV of prefixes[b] + new_rows[b]
    tokens with its own block-table row (row_to_batch = b)."""
    kv = [p + n for p, n in zip(prefixes, new_rows)]
    per_row = -(-max(kv) // 128)
    lens, r2b = [], []
    for b, (p, n) in enumerate(zip(prefixes, new_rows)):
        lens += [p + i + 1 for i in range(n)]
        r2b += [b] * n
    rows = len(lens)
    return W.make_fused_inputs(seed, rows, 64, 128, len(kv) * per_row + 5, lens, (len(kv), per_row),
                               row_to_batch=r2b, dtype=dtype)


def test_topk_packed_requests_grouped():
    """Three requests with different prefixes, each a multiple of 4 rows, in
    one call with group_rows=4 (rows scored in pairs of one request)."""
    inp = _packed_requests(48, [36, 20, 44], [2900, 700, 5100])
    _check_topk(_fused(inp, group_rows=4), inp)


def test_topk_packed_requests_unaligned_single_rows():
    """Request boundaries that are not multiples of 4: group_rows=1."""
    inp = _packed_requests(49, [13, 7, 22], [3300, 100, 2000])
    _check_topk(_fused(inp, group_rows=1), inp)


# ---------------------------------------------------------------- bf16 index cache
# Same checks with q and the keys in bf16 (tcgen05 kind::f16, two 64-dim
# halves per key row); integer inputs pin the operand layout bit-exactly, and
# a cache without per-key scales (kscale = None) means scale 1.


def test_bf16_dense_integer_inputs_exact():
    inp = _small("int", dtype="bf16")
    _check_dense(_dense(inp), inp, exact=True)


@pytest.mark.parametrize("no_scale", [False, True])
def test_bf16_dense_normal_inputs(no_scale):
    inp = _small("normal", dtype="bf16", seed=51)
    if no_scale:
        inp.kscale = None
    _check_dense(_dense(inp), inp)


def test_bf16_dense_grouped_rows_exact():
    lens = np.array([997, 998, 999, 1000, 3001, 3002, 3003, 3004], np.int32)
    inp = W.make_fused_inputs(52, 8, 64, 128, 2 * 24 + 1, lens, (2, 24), row_to_batch=[0, 0, 0, 0, 1, 1, 1, 1],
                              kind="int", dtype="bf16")
    _check_dense(_dense(inp, group_rows=4), inp, exact=True)


def test_bf16_topk_small_and_zero_q():
    inp = _small("normal", dtype="bf16", seed=53)
    _check_topk(_fused(inp), inp)
    inp = _small("zero_q", dtype="bf16")
    slots, idx, scores = _fused(inp)
    for i in range(inp.rows):
        kk = min(int(inp.seq_lens[i]), 512)
        assert idx[i][:kk].tolist() == list(range(kk))


def test_bf16_topk_grouped_prefill_like_no_scale():
    rows, kv = 64, 6000
    lens = (kv - rows + 1 + np.arange(rows)).astype(np.int32)
    blocks = -(-kv // 128)
    inp = W.make_fused_inputs(54, rows, 64, 128, blocks, lens, (1, blocks), row_to_batch=np.zeros(rows, np.int32),
                              dtype="bf16")
    inp.kscale = None
    _check_topk(_fused(inp, group_rows=4), inp)


def test_bf16_topk_packed_requests():
    inp = _packed_requests(55, [36, 20, 44], [2900, 700, 5100], dtype="bf16")
    _check_topk(_fused(inp, group_rows=4), inp)
    inp = _packed_requests(56, [13, 7, 22], [3300, 100, 2000], dtype="bf16")
    _check_topk(_fused(inp, group_rows=1), inp)


def test_bf16_topk_one_chunk_per_row():
    rows, per_row = 640, 12
    lens = np.random.default_rng(57).integers(1, per_row * 128 + 1, size=rows).astype(np.int32)
    inp = W.make_fused_inputs(57, rows, 64, 128, rows * per_row + 1, lens, (rows, per_row), dtype="bf16")
    _check_topk(_fused(inp), inp)


def test_bf16_fused_decode_full_size():
    """The decode workload's shapes with a bf16 cache: 64 rows, seq_lens
    U[4096, 32768], a 16384-block pool; every row checked."""
    inp = W.fused_decode(dtype="bf16")
    _check_topk(_fused(inp), inp)


def test_bf16_fused_prefill_full_size():
    """The prefill workload's shapes with a bf16 cache; every row checked."""
    inp = W.fused_prefill(dtype="bf16")
    _check_all_rows_in_pool(_fused(inp, group_rows=4), inp)


@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
def test_chunked_prefix_calls_match_one_call(dtype):
    """A long extend processed as several calls, each holding one chunk of the
    query rows (causal over prefix + chunk, the same block table): every
    row's slots, indices and scores equal those of one call over all rows,
    bit for bit (a row's scores and selection do not depend on the other
    rows of the call or on how the keys are split into units)."""
    import sparse_attention_indexer_top_gb300 as sai

    rows, kv = 96, 9000
    lens = (kv - rows + 1 + np.arange(rows)).astype(np.int32)
    blocks = -(-kv // 128)
    inp = W.make_fused_inputs(58, rows, 64, 128, blocks + 3, lens, (1, blocks), row_to_batch=np.zeros(rows, np.int32),
                              dtype=dtype)
    whole = _fused(inp, group_rows=4)
    _check_topk(whole, inp, rows=[0, 1, 47, 94, 95])
    d = _dev_inputs(inp)
    for lo, hi in ((0, 32), (32, 40), (40, 96)):
        n = d["seq_lens"][lo:hi]
        s, i, sc = sai.index_score_topk(d["q"][lo:hi], d["w"][lo:hi], d["kcache"], d["kscale"], d["block_table"], n,
                                        max_seq_len=int(lens[hi - 1]), row_to_batch=d["row_to_batch"][lo:hi],
                                        group_rows=4)
        torch.cuda.synchronize()
        assert sai.device_status() == 0
        assert np.array_equal(s.cpu().numpy(), whole[0][lo:hi])
        assert np.array_equal(i.cpu().numpy(), whole[1][lo:hi])
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), whole[2][lo:hi].view(np.uint32))


def test_stalled_unit_wait_runs_out():
    """The bounded waits, exercised without a GPU fault: the test hook makes
    the next fused call stream no key tiles for its work unit 0 (row 0's
    first KV chunk), so every wait for those tiles gives up after about two
    seconds. The call must still finish, set status bit 2, leave the other
    rows exact, and leave the context usable (the same call without the hook
    is exact)."""
    import sparse_attention_indexer_top_gb300 as sai
    from sparse_attention_indexer_top_gb300 import _lib

    inp = W.fused_decode(seed=46, rows=4, min_len=3000, max_len=6000)
    d = _dev_inputs(inp)
    max_len = int(inp.seq_lens.max())
    _lib.load().sai_test_stall_next_fused(0)
    t0 = time.time()
    out = sai.index_score_topk(d["q"], d["w"], d["kcache"], d["kscale"], d["block_table"], d["seq_lens"],
                               max_seq_len=max_len)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    bits = sai.device_status(clear=True)
    assert bits & 2, f"status bits {bits}: no wait gave up"
    assert elapsed < 60
    got = tuple(t.cpu().numpy() for t in out)
    _check_topk(got, inp, rows=[1, 2, 3])
    _check_topk(_fused(inp), inp)  # the hook is consumed; the next call is exact
