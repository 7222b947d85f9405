"""sai_topk_transform_noalloc: the allocation-free entry point.

Callers that cannot allocate device memory where they need a top-k (inside
an allocator callback, a pool owner with no memory left to hand out, code
with only fixed input/output buffers) use this entry point; its scratch is a
fixed array owned by the library. This file checks, through the C ABI, that
it returns exactly what sai_topk_transform returns with a caller-allocated
workspace, on two calls in a row (the second call finds the first call's
data still in the shared array), and that sizes needing more scratch than
the array holds are rejected before anything runs.

Kept in its own file, collected last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SAI_ERR_WORKSPACE = -4


def _t(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _args(inp):
    s, sl, pt = _t(inp.scores), _t(inp.seq_lens), _t(inp.page_tables)
    rs, rb = _t(inp.row_starts), _t(inp.row_to_batch)
    return s, sl, pt, rs, rb


def _with_workspace(lib, inp, stream):
    s, sl, pt, rs, rb = _args(inp)
    rows, stride = s.shape
    ws_bytes = lib.sai_topk_transform_workspace(rows, stride, 512)
    assert ws_bytes > 0, "this case must take the split path that uses scratch"
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    slots = torch.full((rows, 512), -7, dtype=torch.int32, device=DEV)
    idx = torch.full((rows, 512), -7, dtype=torch.int32, device=DEV)
    st = lib.sai_topk_transform(_p(s), rows, stride, _p(rs), _p(sl), _p(pt), pt.shape[0], pt.shape[1], _p(rb),
                                inp.page_size, 512, _p(slots), _p(idx), 0, None, None, _p(ws), ws_bytes, stream)
    assert st == 0
    return slots, idx


def _no_alloc(lib, inp, stream):
    s, sl, pt, rs, rb = _args(inp)
    rows, stride = s.shape
    slots = torch.full((rows, 512), -7, dtype=torch.int32, device=DEV)
    idx = torch.full((rows, 512), -7, dtype=torch.int32, device=DEV)
    st = lib.sai_topk_transform_noalloc(_p(s), rows, stride, _p(rs), _p(sl), _p(pt), pt.shape[0], pt.shape[1],
                                        _p(rb), inp.page_size, 512, _p(slots), _p(idx), stream)
    assert st == 0
    return slots, idx


def test_noalloc_matches_workspace_entry_on_two_calls():
    from sparse_attention_indexer_top_gb300 import _lib

    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    cases = [W.decode_topk(seed=2), W.decode_topk(seed=23, rows=60, min_len=9000, max_len=40000)]
    for inp in cases:  # two calls in a row on the shared scratch
        ref_s, ref_i = _with_workspace(lib, inp, stream)
        got_s, got_i = _no_alloc(lib, inp, stream)
        torch.cuda.synchronize()
        # integer outputs: the tolerance is exact equality
        assert torch.equal(got_i, ref_i)
        assert torch.equal(got_s, ref_s)
    bits = ctypes.c_int(0)
    assert lib.sai_device_status(ctypes.byref(bits), 1, stream) == 0 and bits.value == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from sparse_attention_indexer_top_gb300 import _lib

    lib = _lib.load()
    # fewer rows than two per SM, each 12 x 16384 scores long: the call
    # splits every row into 12 chunks, and on a part with at least 86 SMs
    # their partial lists (rows x 12 x 4100 bytes) outgrow the fixed array
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    rows, stride = 2 * sms - 1, 12 * 16384
    need = lib.sai_topk_transform_workspace(rows, stride, 512)
    if need <= (8 << 20):
        pytest.skip(f"{sms} SMs: {rows} split rows fit the fixed array")
    s = torch.zeros((rows, stride), dtype=torch.float32, device=DEV)
    sl = torch.full((rows,), stride, dtype=torch.int32, device=DEV)
    pt = torch.zeros((rows, stride), dtype=torch.int32, device=DEV)
    out = torch.empty((rows, 512), dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    st = lib.sai_topk_transform_noalloc(_p(s), rows, stride, None, _p(sl), _p(pt), rows, stride, None, 1, 512,
                                        _p(out), None, stream)
    assert st == SAI_ERR_WORKSPACE
