"""The seeded synthetic workloads match the recipes the benchmark and the
parity tests rely on (CPU only): shapes, length laws, packed-extend
geometry, permutation page/block tables (distinct slots), value encodings,
and reproducibility from the seed alone."""

import numpy as np

import workloads as W


def test_tiny_decode_recipe():
    inp = W.tiny_decode()
    assert inp.seq_lens.tolist() == [100, 512, 1000, 4096]
    assert inp.scores.shape == (4, 4096) and inp.scores.dtype == np.float32
    assert inp.page_size == 1 and inp.page_tables.shape == (4, 4096)
    assert np.unique(inp.page_tables).size == inp.page_tables.size


def test_packed_extend_geometry():
    row_starts, seq_lens, r2b, width = W.packed_extend_meta()
    assert width == 140000 and seq_lens.size == 16384
    assert (row_starts[:8192] == 0).all() and (row_starts[8192:] == 70000).all()
    assert seq_lens[0] == 61809 and seq_lens[8191] == 70000 and seq_lens[8192] == 61809
    assert (r2b[:8192] == 0).all() and (r2b[8192:] == 1).all()
    # every window stays inside its request's columns of the shared buffer
    assert ((row_starts + seq_lens) <= (r2b.astype(np.int64) + 1) * 70000).all()
    pt = W.page_table_perm(3, (2, 70000))
    assert np.array_equal(np.sort(pt.ravel()), np.arange(140000))


def test_packed_extend_rows_regenerate_alone():
    inp = W.packed_extend(seed=3, reqs=2, new_tokens=16, kv_len=300)
    for i in (0, 7, 16, 31):
        n = int(inp.seq_lens[i])
        s0 = int(inp.row_starts[i])
        assert np.array_equal(inp.scores[i, s0:s0 + n], W.packed_extend_window(3, i, n))


def test_decode_topk_recipe():
    inp = W.decode_topk()
    assert inp.scores.shape == (128, 32768) and inp.page_size == 128
    assert inp.seq_lens.min() >= 8192 and inp.seq_lens.max() <= 32768
    assert inp.page_tables.shape == (128, 256)
    assert np.unique(inp.page_tables).size == inp.page_tables.size
    row = inp.scores[0, : int(inp.seq_lens[0])]
    # bf16-rounded values: the low 16 bits of every fp32 are zero, and ties are certain
    assert (row.view(np.uint32) & 0xFFFF == 0).all()
    assert np.unique(row).size < row.size


def test_fused_prefill_recipe():
    inp = W.fused_prefill()
    assert inp.rows == 4096 and inp.q.shape == (4096, 64, 128) and inp.q.dtype == np.uint8
    assert inp.seq_lens[0] == 28673 and inp.seq_lens[-1] == 32768
    assert (np.diff(inp.seq_lens) == 1).all()
    assert inp.kcache.shape == (256, 128, 128) and inp.block_table.shape == (1, 256)
    assert np.array_equal(np.sort(inp.block_table.ravel()), np.arange(256))
    assert (inp.row_to_batch == 0).all()
    assert inp.w.min() >= 0 and inp.w.max() <= 0.125
    assert inp.kscale.min() >= 0.5 and inp.kscale.max() <= 2.0


def test_fused_decode_recipe_small():
    inp = W.fused_decode(rows=6)
    assert inp.seq_lens.min() >= 4096 and inp.seq_lens.max() <= 32768
    assert inp.block_table.shape == (6, 256) and inp.kcache.shape[0] == 6 * 256
    assert np.unique(inp.block_table).size == inp.block_table.size
    a = W.fused_decode(rows=6)
    assert np.array_equal(a.q, inp.q) and np.array_equal(a.kcache, inp.kcache)


def test_bf16_variant_encodes_the_same_draws():
    e = W.make_fused_inputs(9, 2, 4, 8, 6, (20, 30), (2, 3), block_size=16)
    b = W.make_fused_inputs(9, 2, 4, 8, 6, (20, 30), (2, 3), block_size=16, dtype="bf16")
    assert b.q.dtype == np.uint16 and b.dtype == "bf16" and e.dtype == "e4m3"
    assert np.array_equal(e.w, b.w) and np.array_equal(e.kscale, b.kscale)
    assert np.array_equal(e.block_table, b.block_table)
