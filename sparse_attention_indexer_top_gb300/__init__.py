"""GB300-native sparse-attention indexer top-k (Python binding of libsai).

Every computation runs in the CUDA kernels of ``libsai.so``; this module only
checks tensor placement/dtypes, passes raw device pointers and the current
CUDA stream through the C ABI (include/sai.h), and uses torch to allocate
outputs and workspaces. There is no CPU fallback: without the built library
every call raises.
"""

from __future__ import annotations

import ctypes
from typing import Optional

import torch

from ._lib import SaiError, check, load, status_string  # noqa: F401

TOPK = 512


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: Optional[torch.Tensor], name: str, dtype, dev, ndim=None):
    if t is None:
        return
    if not t.is_cuda or t.device != dev:
        raise ValueError(f"{name} must be on {dev}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def device_status(clear: bool = True, stream=None) -> int:
    """Synchronize ``stream`` and return the device status bits (0 = clean)."""
    bits = ctypes.c_int(0)
    load().sai_device_status(ctypes.byref(bits), int(clear), _stream(stream))
    return bits.value


def topk_transform_workspace(rows: int, score_stride: int, k: int = TOPK) -> int:
    return int(load().sai_topk_transform_workspace(int(rows), int(score_stride), int(k)))


def _block_outputs(rows, k, dev, want_blocks, out_blocks, out_counts):
    if want_blocks or out_blocks is not None:
        if out_blocks is None:
            out_blocks = torch.empty((rows, k), dtype=torch.int32, device=dev)
        if out_counts is None:
            out_counts = torch.empty((rows,), dtype=torch.int32, device=dev)
        _need(out_blocks, "out_blocks", torch.int32, dev, 2)
        _need(out_counts, "out_counts", torch.int32, dev, 1)
    return out_blocks, out_counts


def topk_transform(scores: torch.Tensor, seq_lens: torch.Tensor, page_tables: Optional[torch.Tensor] = None, *,
                   page_size: int = 1, k: int = TOPK, row_starts: Optional[torch.Tensor] = None,
                   row_to_batch: Optional[torch.Tensor] = None, out_slots: Optional[torch.Tensor] = None,
                   out_indices: Optional[torch.Tensor] = None, want_indices: bool = False,
                   block_size: int = 128, want_blocks: bool = False, out_blocks: Optional[torch.Tensor] = None,
                   out_counts: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Top-k of each row's score window mapped through its page-table row.

    ``scores`` is fp32 ``[rows, stride]`` with unit column stride (any row
    stride); ``seq_lens``, ``row_starts``, ``row_to_batch`` are int32
    ``[rows]``; ``page_tables`` int32 ``[pt_rows, pt_stride]`` with unit
    column stride. Returns ``out_slots`` (int32 ``[rows, k]``), or
    ``(out_slots, out_indices)`` when indices are requested. With
    ``want_blocks`` (or ``out_blocks``) the same call also builds each row's
    ascending distinct blocks ``slot // block_size`` (int32 ``[rows, k]``, -1
    padded) and their counts (int32 ``[rows]``), appended to the result.
    """
    dev = scores.device
    _need(scores, "scores", torch.float32, dev, 2)
    _need(seq_lens, "seq_lens", torch.int32, dev, 1)
    _need(page_tables, "page_tables", torch.int32, dev, 2)
    _need(row_starts, "row_starts", torch.int32, dev, 1)
    _need(row_to_batch, "row_to_batch", torch.int32, dev, 1)
    if scores.stride(1) != 1 or (page_tables is not None and page_tables.stride(1) != 1):
        raise ValueError("scores and page_tables need unit column stride")
    rows = scores.shape[0]
    for name, t in (("seq_lens", seq_lens), ("row_starts", row_starts), ("row_to_batch", row_to_batch)):
        if t is not None and (t.shape[0] != rows or not t.is_contiguous()):
            raise ValueError(f"{name} must be contiguous [{rows}]")
    if out_slots is None and page_tables is not None:
        out_slots = torch.empty((rows, k), dtype=torch.int32, device=dev)
    if out_indices is None and (want_indices or page_tables is None):
        out_indices = torch.empty((rows, k), dtype=torch.int32, device=dev)
    stride = scores.stride(0) if rows > 1 else max(scores.shape[1], 1)
    ws_bytes = topk_transform_workspace(rows, stride, k) if rows else 0
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    pt_rows, pt_stride = (page_tables.shape[0], page_tables.stride(0)) if page_tables is not None else (0, 0)
    out_blocks, out_counts = _block_outputs(rows, k, dev, want_blocks, out_blocks, out_counts)
    st = load().sai_topk_transform(
        _ptr(scores), rows, stride, _ptr(row_starts), _ptr(seq_lens), _ptr(page_tables), pt_rows, pt_stride,
        _ptr(row_to_batch), int(page_size), int(k), _ptr(out_slots), _ptr(out_indices), int(block_size),
        _ptr(out_blocks), _ptr(out_counts), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))
    check(st, "sai_topk_transform")
    blocks = () if out_blocks is None else (out_blocks, out_counts)
    if out_slots is None:
        return (out_indices, *blocks) if blocks else out_indices
    if want_indices or out_indices is not None:
        return (out_slots, out_indices, *blocks)
    return (out_slots, *blocks) if blocks else out_slots


def topk_transform_noalloc(scores: torch.Tensor, seq_lens: torch.Tensor, page_tables: torch.Tensor, *,
                           out_slots: torch.Tensor, out_indices: Optional[torch.Tensor] = None, page_size: int = 1,
                           k: int = TOPK, row_starts: Optional[torch.Tensor] = None,
                           row_to_batch: Optional[torch.Tensor] = None, stream=None) -> None:
    """``topk_transform`` for callers that cannot allocate device memory.

    The caller supplies the output buffers; the split path's scratch is a
    fixed library-owned device array, so this wrapper allocates nothing.
    Calls that would need more scratch than that array holds raise
    ``SaiError`` (workspace). Calls that may overlap on the GPU share the
    array and must be serialized by the caller.
    """
    rows = scores.shape[0]
    stride = scores.stride(0) if rows > 1 else max(scores.shape[1], 1)
    st = load().sai_topk_transform_noalloc(
        _ptr(scores), rows, stride, _ptr(row_starts), _ptr(seq_lens), _ptr(page_tables), page_tables.shape[0],
        page_tables.stride(0), _ptr(row_to_batch), int(page_size), int(k), _ptr(out_slots), _ptr(out_indices),
        _stream(stream))
    check(st, "sai_topk_transform_noalloc")


def _fused_check(q, w, kcache, kscale, block_table, seq_lens, row_to_batch):
    """Argument checks of the fused calls; returns (device, bf16). The element
    type follows ``q``: uint8 e4m3 codes (FP8 index cache) or torch.bfloat16
    (bf16 index cache, where ``kscale`` may be None)."""
    dev = q.device
    bf16 = q.dtype == torch.bfloat16
    elem = torch.bfloat16 if bf16 else torch.uint8
    _need(q, "q", elem, dev, 3)
    _need(w, "w", torch.float32, dev, 2)
    _need(kcache, "kcache", elem, dev, 3)
    if kscale is None and not bf16:
        raise ValueError("kscale is required for an FP8 index cache")
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(seq_lens, "seq_lens", torch.int32, dev, 1)
    _need(row_to_batch, "row_to_batch", torch.int32, dev, 1)
    _need(kscale, "kscale", torch.float32, dev, 2)
    for name, t in (("q", q), ("w", w), ("kcache", kcache), ("kscale", kscale), ("seq_lens", seq_lens)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if block_table.stride(1) != 1:
        raise ValueError("block_table needs unit column stride")
    return dev, bf16


def index_score_topk_workspace(rows: int, max_seq_len: int, group_rows: int = 1, k: int = TOPK) -> int:
    return int(load().sai_index_score_topk_workspace(int(rows), int(max_seq_len), int(group_rows), int(k)))


def index_score_topk(q: torch.Tensor, w: torch.Tensor, kcache: torch.Tensor, kscale: Optional[torch.Tensor],
                     block_table: torch.Tensor, seq_lens: torch.Tensor, *, max_seq_len: int,
                     row_to_batch: Optional[torch.Tensor] = None, group_rows: int = 1, k: int = TOPK,
                     out_slots: Optional[torch.Tensor] = None, out_indices: Optional[torch.Tensor] = None,
                     out_scores: Optional[torch.Tensor] = None, block_size: int = 128, want_blocks: bool = False,
                     out_blocks: Optional[torch.Tensor] = None, out_counts: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None):
    """Fused index score + top-k. ``q`` e4m3 codes (uint8) ``[rows, 64,
    128]``, ``w`` fp32 ``[rows, 64]``, ``kcache`` uint8 ``[blocks, 128, 128]``,
    ``kscale`` fp32 ``[blocks, 128]``, ``block_table`` int32; or ``q`` and
    ``kcache`` torch.bfloat16 (bf16 index cache, ``kscale`` optional).
    Returns ``(slots, indices, scores)``, plus ``(blocks, counts)`` (each
    row's ascending distinct ``slot // block_size``, -1 padded) with
    ``want_blocks`` or ``out_blocks``."""
    dev, bf16 = _fused_check(q, w, kcache, kscale, block_table, seq_lens, row_to_batch)
    rows = q.shape[0]
    if out_slots is None:
        out_slots = torch.empty((rows, k), dtype=torch.int32, device=dev)
    if out_indices is None:
        out_indices = torch.empty((rows, k), dtype=torch.int32, device=dev)
    if out_scores is None:
        out_scores = torch.empty((rows, k), dtype=torch.float32, device=dev)
    ws = index_score_topk_workspace(rows, max_seq_len, group_rows, k) if rows else 0
    if workspace is None and ws:
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    out_blocks, out_counts = _block_outputs(rows, k, dev, want_blocks, out_blocks, out_counts)
    name = "sai_index_score_topk_bf16" if bf16 else "sai_index_score_topk"
    st = getattr(load(), name)(
        _ptr(q), _ptr(w), _ptr(kcache), _ptr(kscale), kcache.shape[0], _ptr(block_table), block_table.shape[0],
        block_table.stride(0), _ptr(row_to_batch), _ptr(seq_lens), rows, q.shape[1], q.shape[2], kcache.shape[1],
        int(max_seq_len), int(group_rows), int(k), _ptr(out_slots), _ptr(out_indices), _ptr(out_scores),
        int(block_size), _ptr(out_blocks), _ptr(out_counts), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream))
    check(st, name)
    if out_blocks is not None:
        return out_slots, out_indices, out_scores, out_blocks, out_counts
    return out_slots, out_indices, out_scores


def index_score(q: torch.Tensor, w: torch.Tensor, kcache: torch.Tensor, kscale: Optional[torch.Tensor],
                block_table: torch.Tensor, seq_lens: torch.Tensor, *, max_seq_len: int,
                row_to_batch: Optional[torch.Tensor] = None, group_rows: int = 1, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """Dense index scores ``[rows, max_seq_len]`` (FP8 or bf16 cache, as for
    ``index_score_topk``; cells past each row's length are left as they were;
    a new ``out`` starts as NaN)."""
    dev, bf16 = _fused_check(q, w, kcache, kscale, block_table, seq_lens, row_to_batch)
    rows = q.shape[0]
    if out is None:
        out = torch.full((rows, max(max_seq_len, 1)), float("nan"), dtype=torch.float32, device=dev)
    name = "sai_index_score_bf16" if bf16 else "sai_index_score"
    st = getattr(load(), name)(
        _ptr(q), _ptr(w), _ptr(kcache), _ptr(kscale), kcache.shape[0], _ptr(block_table), block_table.shape[0],
        block_table.stride(0), _ptr(row_to_batch), _ptr(seq_lens), rows, q.shape[1], q.shape[2], kcache.shape[1],
        int(max_seq_len), int(group_rows), _ptr(out), out.stride(0), _stream(stream))
    check(st, name)
    return out


def index_score_per_head(q: torch.Tensor, w: torch.Tensor, kcache: torch.Tensor, kscale: Optional[torch.Tensor],
                         block_table: torch.Tensor, seq_lens: torch.Tensor, *, max_seq_len: int,
                         row_to_batch: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """Dense per-index-head scores ``[rows, 64, max_seq_len]``: head h's
    summand ``kscale * w_h * relu(q_h . k)`` of the index score (FP8 or bf16
    cache, as for ``index_score_topk``; a new ``out`` starts as NaN)."""
    dev, bf16 = _fused_check(q, w, kcache, kscale, block_table, seq_lens, row_to_batch)
    rows, heads = q.shape[0], q.shape[1]
    if out is None:
        out = torch.full((rows, heads, max(max_seq_len, 1)), float("nan"), dtype=torch.float32, device=dev)
    if out.dim() != 3 or out.stride(2) != 1 or out.stride(0) != heads * out.stride(1):
        raise ValueError("out must be [rows, 64, stride] with rows of 64 contiguous head rows")
    name = "sai_index_score_per_head_bf16" if bf16 else "sai_index_score_per_head"
    st = getattr(load(), name)(
        _ptr(q), _ptr(w), _ptr(kcache), _ptr(kscale), kcache.shape[0], _ptr(block_table), block_table.shape[0],
        block_table.stride(0), _ptr(row_to_batch), _ptr(seq_lens), rows, heads, q.shape[2], kcache.shape[1],
        int(max_seq_len), _ptr(out), out.stride(1), _stream(stream))
    check(st, name)
    return out


def index_score_topk_per_head_workspace(rows: int, max_seq_len: int, k: int = TOPK) -> int:
    return int(load().sai_index_score_topk_per_head_workspace(int(rows), int(max_seq_len), int(k)))


def index_score_topk_per_head(q: torch.Tensor, w: torch.Tensor, kcache: torch.Tensor, kscale: Optional[torch.Tensor],
                              block_table: torch.Tensor, seq_lens: torch.Tensor, *, max_seq_len: int,
                              row_to_batch: Optional[torch.Tensor] = None, k: int = TOPK,
                              out_slots: Optional[torch.Tensor] = None, out_indices: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None, stream=None):
    """Top-k per (row, index head) of the per-head scores: ``(slots,
    indices)``, int32 ``[rows, 64, k]`` (-1 padded)."""
    dev, bf16 = _fused_check(q, w, kcache, kscale, block_table, seq_lens, row_to_batch)
    rows, heads = q.shape[0], q.shape[1]
    if out_slots is None:
        out_slots = torch.empty((rows, heads, k), dtype=torch.int32, device=dev)
    if out_indices is None:
        out_indices = torch.empty((rows, heads, k), dtype=torch.int32, device=dev)
    ws = index_score_topk_per_head_workspace(rows, max_seq_len, k) if rows else 0
    if workspace is None and ws:
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    name = "sai_index_score_topk_per_head_bf16" if bf16 else "sai_index_score_topk_per_head"
    st = getattr(load(), name)(
        _ptr(q), _ptr(w), _ptr(kcache), _ptr(kscale), kcache.shape[0], _ptr(block_table), block_table.shape[0],
        block_table.stride(0), _ptr(row_to_batch), _ptr(seq_lens), rows, heads, q.shape[2], kcache.shape[1],
        int(max_seq_len), int(k), _ptr(out_slots), _ptr(out_indices), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream))
    check(st, name)
    return out_slots, out_indices


def sparse_blocks(slots: torch.Tensor, block_size: int = 128, *, out_blocks: Optional[torch.Tensor] = None,
                  out_counts: Optional[torch.Tensor] = None, stream=None):
    """Per-row distinct KV blocks of top-k slots: ``(blocks [rows, k] int32,
    ascending, -1 padded; counts [rows] int32)``. Slots < 0 are padding."""
    dev = slots.device
    _need(slots, "slots", torch.int32, dev, 2)
    if not slots.is_contiguous():
        raise ValueError("slots must be contiguous")
    rows, k = slots.shape
    if out_blocks is None:
        out_blocks = torch.empty((rows, k), dtype=torch.int32, device=dev)
    if out_counts is None:
        out_counts = torch.empty((rows,), dtype=torch.int32, device=dev)
    _need(out_blocks, "out_blocks", torch.int32, dev, 2)
    _need(out_counts, "out_counts", torch.int32, dev, 1)
    st = load().sai_sparse_blocks(_ptr(slots), rows, int(k), int(block_size), _ptr(out_blocks), _ptr(out_counts),
                                  _stream(stream))
    check(st, "sai_sparse_blocks")
    return out_blocks, out_counts
