"""The C-ABI library loads, exports every symbol include/sai.h declares, and
rejects bad host arguments before touching the GPU (CPU only)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_top_gb300 import build, _lib

    build.build()
    return _lib.load()


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"\b(sai_\w+)\s*\(", txt)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    from sparse_attention_indexer_top_gb300._lib import SIGNATURES

    names = _declared()
    assert names, "no declarations found"
    for n in names:
        assert hasattr(lib, n), n
        assert n in SIGNATURES, f"{n} has no ctypes signature"


def test_status_strings(lib):
    from sparse_attention_indexer_top_gb300._lib import status_string

    assert status_string(0) == "ok"
    assert "NULL" in status_string(-1)
    assert status_string(12345) == "unknown status"


def _call(lib, **kw):
    a = dict(scores=1 << 20, rows=4, stride=4096, row_starts=None, seq_lens=1 << 21, pt=1 << 22, pt_rows=4,
             pt_stride=4096, r2b=None, ps=1, k=512, out_slots=1 << 23, out_idx=None, bs=128, out_blocks=None,
             out_counts=None, ws=None, ws_bytes=0)
    a.update(kw)
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.sai_topk_transform(v(a["scores"]), a["rows"], a["stride"], v(a["row_starts"]), v(a["seq_lens"]),
                                  v(a["pt"]), a["pt_rows"], a["pt_stride"], v(a["r2b"]), a["ps"], a["k"],
                                  v(a["out_slots"]), v(a["out_idx"]), a["bs"], v(a["out_blocks"]),
                                  v(a["out_counts"]), v(a["ws"]), a["ws_bytes"], None)


def test_host_validation(lib):
    # every case below is rejected before any CUDA call
    assert _call(lib, k=0) == -2
    assert _call(lib, k=256) == -3
    assert _call(lib, rows=-1) == -2
    assert _call(lib, out_slots=None, out_idx=None) == -1
    assert _call(lib, scores=None) == -1
    assert _call(lib, seq_lens=None) == -1
    assert _call(lib, pt=None) == -1  # slots requested without a page table
    assert _call(lib, ps=0) == -2
    assert _call(lib, pt_rows=3) == -2  # fewer page-table rows than rows, no row_to_batch
    assert _call(lib, stride=0) == -2
    assert _call(lib, scores=(1 << 20) + 2) == -7  # fp32 pointer not 4-byte aligned
    assert _call(lib, rows=0) == 0  # nothing to do
    # block lists: a block size of at least 1, counts only with blocks, a page table
    assert _call(lib, out_blocks=1 << 24, bs=0) == -2
    assert _call(lib, out_counts=1 << 24) == -1
    assert _call(lib, out_slots=None, out_idx=None, out_blocks=1 << 24, pt=None) == -1
    assert _call(lib, out_blocks=(1 << 24) + 2) == -7


def test_workspace_query_without_args(lib):
    assert lib.sai_topk_transform_workspace(0, 100, 512) == 0
    assert lib.sai_topk_transform_workspace(10, 100, 256) == 0


def test_sparse_blocks_argument_errors(lib):
    out = ctypes.c_void_p(1 << 20)
    slots = ctypes.c_void_p(1 << 20)
    assert lib.sai_sparse_blocks(slots, 4, 0, 128, out, None, None) == -2    # k < 1
    assert lib.sai_sparse_blocks(slots, 4, 513, 128, out, None, None) == -2  # k > 512
    assert lib.sai_sparse_blocks(slots, 4, 512, 0, out, None, None) == -2    # block_size < 1
    assert lib.sai_sparse_blocks(slots, -1, 512, 128, out, None, None) == -2
    assert lib.sai_sparse_blocks(None, 4, 512, 128, out, None, None) == -1
    assert lib.sai_sparse_blocks(slots, 4, 512, 128, None, None, None) == -1
    assert lib.sai_sparse_blocks(ctypes.c_void_p((1 << 20) + 2), 4, 512, 128, out, None, None) == -7
    assert lib.sai_sparse_blocks(None, 0, 512, 128, None, None, None) == 0  # nothing to do


def test_fused_argument_errors(lib):
    # (q, w, kcache, kscale, num_blocks, bt, bt_rows, bt_stride, r2b, seq_lens, rows, heads, dim, bs, max_len, group)
    p = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)

    def args(q=p, kscale=p, heads=64, group=1, rows=4):
        return (q, p, p, kscale, 8, p, 4, 8, None, p, rows, heads, 128, 128, 1024, group)

    for name in ("sai_index_score_topk", "sai_index_score_topk_bf16"):
        f = getattr(lib, name)
        tail = (512, p, p, p, 128, None, None, p, 1 << 20, None)
        assert f(*args(heads=32), *tail) == -3
        assert f(*args(group=2), *tail) == -3
        assert f(*args(rows=-1), *tail) == -2
        assert f(*args(q=None), *tail) == -1
        assert f(*args(rows=0), *tail) == 0
        assert f(*args(), 512, p, p, p, 0, p, None, p, 1 << 20, None) == -2  # block lists need a block size
        assert f(*args(), 512, p, p, p, 128, None, p, p, 1 << 20, None) == -1  # counts without blocks
    for name in ("sai_index_score", "sai_index_score_bf16"):
        f = getattr(lib, name)
        assert f(*args(heads=32), p, 1024, None) == -3
        assert f(*args(q=None), p, 1024, None) == -1
    # a missing key scale is an error for the FP8 cache only: the bf16 calls
    # get past the null check and stop at the misaligned q
    assert lib.sai_index_score_topk(*args(q=odd, kscale=None), 512, p, p, p, 128, None, None, p, 1 << 20, None) == -1
    assert lib.sai_index_score_topk_bf16(*args(q=odd, kscale=None), 512, p, p, p, 128, None, None, p, 1 << 20,
                                         None) == -7
    assert lib.sai_index_score(*args(q=odd, kscale=None), p, 1024, None) == -1
    assert lib.sai_index_score_bf16(*args(q=odd, kscale=None), p, 1024, None) == -7


def test_per_head_argument_errors(lib):
    p = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)

    def args(q=p, kscale=p, heads=64, rows=4):
        return (q, p, p, kscale, 8, p, 4, 8, None, p, rows, heads, 128, 128, 1024)

    for name in ("sai_index_score_topk_per_head", "sai_index_score_topk_per_head_bf16"):
        f = getattr(lib, name)
        tail = (512, p, p, p, 1 << 30, None)
        assert f(*args(heads=32), *tail) == -3
        assert f(*args(rows=-1), *tail) == -2
        assert f(*args(q=None), *tail) == -1
        assert f(*args(rows=0), *tail) == 0
        assert f(*args(), 256, p, p, p, 1 << 30, None) == -3  # k must be 512
        assert f(*args(), 512, None, None, p, 1 << 30, None) == -1  # no output
    for name in ("sai_index_score_per_head", "sai_index_score_per_head_bf16"):
        f = getattr(lib, name)
        assert f(*args(heads=32), p, 1024, None) == -3
        assert f(*args(), p, 1000, None) == -2  # out_stride < max_seq_len
    assert lib.sai_index_score_topk_per_head(*args(q=odd, kscale=None), 512, p, p, p, 1 << 30, None) == -1
    assert lib.sai_index_score_topk_per_head_bf16(*args(q=odd, kscale=None), 512, p, p, p, 1 << 30, None) == -7
    assert lib.sai_index_score_topk_per_head_workspace(0, 100, 512) == 0
