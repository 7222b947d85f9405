"""The Python binding refuses host (CPU) tensors and wrong dtypes before any
library call: the library has no CPU fallback, so a call with host memory
must fail loudly rather than compute anywhere else (CPU only)."""

import numpy as np
import pytest
import torch

import sparse_attention_indexer_top_gb300 as sai
import workloads as W


def _host_fused(dtype="e4m3"):
    inp = W.make_fused_inputs(81, 2, 64, 128, 8, (300, 200), (2, 3), dtype=dtype)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a))
    q = t(inp.q.view(np.int16)).view(torch.bfloat16) if dtype == "bf16" else t(inp.q)
    kc = t(inp.kcache.view(np.int16)).view(torch.bfloat16) if dtype == "bf16" else t(inp.kcache)
    return q, t(inp.w), kc, t(inp.kscale), t(inp.block_table), t(inp.seq_lens)


def test_topk_transform_refuses_host_tensors():
    scores = torch.zeros((2, 1024), dtype=torch.float32)
    lens = torch.tensor([1024, 600], dtype=torch.int32)
    pt = torch.zeros((2, 1024), dtype=torch.int32)
    with pytest.raises(ValueError, match="must be on"):
        sai.topk_transform(scores, lens, pt)


@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
def test_fused_calls_refuse_host_tensors(dtype):
    q, w, kc, ks, bt, lens = _host_fused(dtype)
    for fn in (sai.index_score_topk, sai.index_score, sai.index_score_per_head, sai.index_score_topk_per_head):
        with pytest.raises(ValueError, match="must be on"):
            fn(q, w, kc, ks, bt, lens, max_seq_len=300)


def test_sparse_blocks_refuses_host_tensors():
    with pytest.raises(ValueError, match="must be on"):
        sai.sparse_blocks(torch.zeros((2, 512), dtype=torch.int32))
