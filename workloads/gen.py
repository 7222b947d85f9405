"""Seeded input generators for the five indexer workloads.

The shapes are the ones the pages measure or launch with:

* k = 512 and a 16384-row prefill chunk at ISL 70000 with two requests packed
  into one score buffer (sglang PR #37889 "[AMD] Enable GLM DSA prefill top-k
  to the v2 kernel", Motivation and the kernel-level table in "Speed Tests and
  Profiling");
* 128-token KV blocks and an FP8 (e4m3) index-key cache (ROCm/ATOM PR #1473
  "enable minimax m3 fp8 index cache and fuse index_score_kernel with
  partial_topk kernel", launch script in Motivation).

Every array is drawn on the host from ``numpy.random.Generator(PCG64)`` with a
``SeedSequence`` that names the config and the array, so any single array (or
any single score row) can be regenerated alone. FP8 and bf16 values are
produced by torch's round-to-nearest-even casts (a library routine); this
module does no indexer arithmetic.
"""

from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

K_TOP = 512
KV_BLOCK = 128
HEAD_DIM = 128
IDX_HEADS = 64

# Human-readable names of the five workloads, in order.
CONFIGS = (
    "tiny decode-layout top-k transform: 4 rows, seq_lens {100,512,1000,4096}, "
    "fp32 N(0,1), page_size 1",
    "decode top-k transform: 128 rows, seq_lens U[8192,32768], bf16-rounded "
    "N(0,1) in [128,32768], page_size 128",
    "packed-extend prefill top-k: 2 requests x 8192 new tokens on a 70000-token "
    "KV each, scores [16384,140000] fp32 N(0,1), page_size 1",
    "fused decode FP8 index-score + top-512: 64 rows, 64 heads x 128, "
    "seq_lens U[4096,32768], 128-token blocks",
    "fused prefill FP8 index-score + top-512: 4096 causal rows on a "
    "32768-token KV, 64 heads x 128, 128-token blocks",
)


def _rng(*words: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(words))))


def e4m3fn_encode(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to OCP E4M3FN codes (uint8) with torch's RNE cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 bit patterns (uint16) with torch's RNE cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _bf16_round(x: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy().copy()


def _row_values(seed: int, row: int, n: int, kind: str) -> np.ndarray:
    """Values of one score window; regenerable from (seed, row) alone."""
    g = _rng(seed, 101, row)
    if kind == "normal":
        return g.standard_normal(n, dtype=np.float32)
    if kind == "bf16":
        return _bf16_round(g.standard_normal(n, dtype=np.float32))
    if kind == "int":  # small integers: many exact ties
        return g.integers(-8, 9, size=n).astype(np.float32)
    if kind == "const":
        return np.full(n, 0.5, np.float32)
    if kind == "signed_zero":  # +0 / -0 mixed with a few non-zero values
        v = np.where(g.random(n) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
        hot = g.random(n) < 0.01
        v[hot] = g.standard_normal(int(hot.sum()), dtype=np.float32)
        return v
    if kind == "inf":  # finite values with some +-inf mixed in
        v = g.standard_normal(n, dtype=np.float32)
        u = g.random(n)
        v[u < 0.002] = np.inf
        v[(u >= 0.002) & (u < 0.004)] = -np.inf
        return v
    if kind == "scaled":  # N(0,1) times 1e-3, 1 or 1e3, varying from row to row
        return g.standard_normal(n, dtype=np.float32) * np.float32(10.0 ** (3 * ((row * 7919) % 3 - 1)))
    if kind == "ascending":  # worst order for a streaming filter
        return np.sort(g.standard_normal(n, dtype=np.float32))
    if kind == "descending":
        return np.sort(g.standard_normal(n, dtype=np.float32))[::-1].copy()
    raise ValueError(kind)


@dataclass
class TopkInputs:
    """Inputs of one ``topk_transform`` call (host arrays)."""

    scores: np.ndarray  # [rows, stride] float32
    seq_lens: np.ndarray  # [rows] int32
    page_tables: np.ndarray  # [pt_rows, pt_stride] int32
    page_size: int
    k: int = K_TOP
    row_starts: Optional[np.ndarray] = None  # [rows] int32 or None
    row_to_batch: Optional[np.ndarray] = None  # [rows] int32 or None
    name: str = ""

    @property
    def rows(self) -> int:
        return int(self.seq_lens.shape[0])


def make_topk_inputs(
    seed: int,
    seq_lens,
    score_stride: int,
    page_size: int,
    pt_shape,
    row_starts=None,
    row_to_batch=None,
    kind: str = "normal",
    fill: float = 0.0,
    k: int = K_TOP,
    name: str = "",
    threads: int = 0,
    scores_out: Optional[np.ndarray] = None,
) -> TopkInputs:
    """Build a score buffer whose row ``i`` holds a window of ``seq_lens[i]``
    values starting at column ``row_starts[i]`` (0 if absent); every other cell
    is ``fill`` (``+inf`` poisons any read outside the windows).

    The page table is one random permutation of ``0 .. pt_rows*pt_stride-1``
    reshaped to ``pt_shape``, so physical slots are distinct across requests.
    ``scores_out`` (optional, e.g. a pinned host buffer) receives the scores.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    rows = int(seq_lens.shape[0])
    if scores_out is None:
        scores = np.empty((rows, score_stride), dtype=np.float32)
    else:
        scores = scores_out
        assert scores.shape == (rows, score_stride) and scores.dtype == np.float32
    starts = None if row_starts is None else np.asarray(row_starts, dtype=np.int32)

    def fill_row(i: int) -> None:
        n = int(seq_lens[i])
        s = 0 if starts is None else int(starts[i])
        row = scores[i]
        row[:s] = fill
        row[s + max(n, 0):] = fill
        if n > 0:
            row[s : s + n] = _row_values(seed, i, n, kind)

    nthreads = threads or min(16, os.cpu_count() or 1)
    if rows * score_stride > (1 << 24) and nthreads > 1:
        with _cf.ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(fill_row, range(rows)))
    else:
        for i in range(rows):
            fill_row(i)
    pt = page_table_perm(seed, pt_shape)
    r2b = None if row_to_batch is None else np.asarray(row_to_batch, dtype=np.int32)
    return TopkInputs(scores, seq_lens, pt, page_size, k, starts, r2b, name)


def page_table_perm(seed: int, pt_shape) -> np.ndarray:
    """One random permutation of the slot ids, reshaped to ``pt_shape``."""
    pt_rows, pt_stride = pt_shape
    return _rng(seed, 202).permutation(pt_rows * pt_stride).astype(np.int32).reshape(pt_rows, pt_stride)


def fill_rows(dst: np.ndarray, r0: int, seed: int, row_starts, seq_lens, kind: str = "normal",
              fill: float = 0.0, threads: int = 0) -> None:
    """Write score rows ``r0 .. r0 + len(dst) - 1`` of a buffer into ``dst``
    (same values as ``make_topk_inputs`` gives those rows)."""
    def one(j: int) -> None:
        i = r0 + j
        n = int(seq_lens[i])
        s = 0 if row_starts is None else int(row_starts[i])
        dst[j, :s] = fill
        dst[j, s + max(n, 0):] = fill
        if n > 0:
            dst[j, s:s + n] = _row_values(seed, i, n, kind)

    nthreads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(one, range(dst.shape[0])))


def tiny_decode(seed: int = 1) -> TopkInputs:
    """4 decode rows of lengths {100, 512, 1000, 4096}; page_size 1."""
    return make_topk_inputs(seed, [100, 512, 1000, 4096], 4096, 1, (4, 4096), name="tiny_decode")


def decode_topk(seed: int = 2, rows: int = 128, max_len: int = 32768, min_len: int = 8192) -> TopkInputs:
    """Decode rows with lengths U[min_len, max_len] and bf16-rounded N(0,1)
    scores (ties are certain); 128-token pages."""
    lens = _rng(seed, 303).integers(min_len, max_len + 1, size=rows).astype(np.int32)
    blocks = -(-max_len // KV_BLOCK)
    return make_topk_inputs(seed, lens, max_len, KV_BLOCK, (rows, blocks), kind="bf16", name="decode_topk")


def packed_extend_meta(reqs: int = 2, new_tokens: int = 8192, kv_len: int = 70000):
    """Row metadata of a packed extend batch: ``reqs`` requests, each adding
    ``new_tokens`` query rows whose KV totals ``kv_len`` tokens (a prefix of
    ``kv_len - new_tokens``). Row ``i = new_tokens*r + p`` reads request ``r``'s
    window of the shared buffer at column ``kv_len*r`` with causal length
    ``kv_len - new_tokens + p + 1`` and uses page-table row ``r``."""
    rows = reqs * new_tokens
    r = np.arange(rows, dtype=np.int64) // new_tokens
    p = np.arange(rows, dtype=np.int64) % new_tokens
    row_starts = (kv_len * r).astype(np.int32)
    seq_lens = (kv_len - new_tokens + p + 1).astype(np.int32)
    row_to_batch = r.astype(np.int32)
    return row_starts, seq_lens, row_to_batch, reqs * kv_len


def packed_extend_window(seed: int, row: int, n: int, kind: str = "normal") -> np.ndarray:
    """Regenerate the score window of one row."""
    return _row_values(seed, row, n, kind)


def packed_extend(seed: int = 3, reqs: int = 2, new_tokens: int = 8192, kv_len: int = 70000,
                  fill: float = 0.0, kind: str = "normal", stride_pad: int = 0,
                  scores_out: Optional[np.ndarray] = None) -> TopkInputs:
    """Packed-extend prefill top-k inputs (all requests share one buffer)."""
    row_starts, seq_lens, r2b, width = packed_extend_meta(reqs, new_tokens, kv_len)
    return make_topk_inputs(seed, seq_lens, width + stride_pad, 1, (reqs, kv_len),
                            row_starts=row_starts, row_to_batch=r2b, fill=fill, kind=kind,
                            name="packed_extend", scores_out=scores_out)


@dataclass
class FusedInputs:
    """Inputs of one ``index_score_topk`` call (host arrays)."""

    q: np.ndarray  # [rows, heads, dim] uint8 e4m3fn codes (or uint16 bf16 bits)
    w: np.ndarray  # [rows, heads] float32
    kcache: np.ndarray  # [blocks, block_size, dim] uint8 e4m3fn codes (or uint16 bf16 bits)
    kscale: np.ndarray  # [blocks, block_size] float32
    block_table: np.ndarray  # [bt_rows, bt_stride] int32
    seq_lens: np.ndarray  # [rows] int32 (causal length per query row)
    row_to_batch: Optional[np.ndarray] = None
    k: int = K_TOP
    name: str = ""
    extra: dict = field(default_factory=dict)
    dtype: str = "e4m3"  # element type of q and kcache: "e4m3" or "bf16"

    @property
    def rows(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def block_size(self) -> int:
        return int(self.kcache.shape[1])


def make_fused_inputs(seed: int, rows: int, heads: int, dim: int, num_blocks: int,
                      seq_lens, block_table_shape, row_to_batch=None, block_size: int = KV_BLOCK,
                      q_std: float = 0.25, k_std: float = 0.25, k: int = K_TOP,
                      name: str = "", kind: str = "normal", dtype: str = "e4m3") -> FusedInputs:
    """q, k ~ e4m3(N(0,1)*std) (or bf16 with ``dtype="bf16"``); w ~ U(0,1)/8;
    kscale ~ U(0.5,2); block table = a permutation of the pool's block ids
    reshaped to ``block_table_shape``.

    ``kind="int"`` draws small integer-valued q and k (exact in e4m3) with
    w = 1 and kscale = 1, so every score is an exact integer.
    ``kind="zero_q"`` makes q all zero (every score 0).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    enc = {"e4m3": e4m3fn_encode, "bf16": bf16_encode}[dtype]
    if kind == "int":
        q = enc(_rng(seed, 401).integers(-3, 4, size=(rows, heads, dim)).astype(np.float32))
        kc = enc(_rng(seed, 402).integers(-3, 4, size=(num_blocks, block_size, dim)).astype(np.float32))
        w = np.ones((rows, heads), np.float32)
        ks = np.ones((num_blocks, block_size), np.float32)
    else:
        q = enc(_rng(seed, 401).standard_normal((rows, heads, dim), dtype=np.float32) * np.float32(q_std))
        kc = enc(_rng(seed, 402).standard_normal((num_blocks, block_size, dim), dtype=np.float32) * np.float32(k_std))
        w = (_rng(seed, 403).random((rows, heads), dtype=np.float32) / np.float32(8.0)).astype(np.float32)
        ks = (np.float32(0.5) + np.float32(1.5) * _rng(seed, 404).random((num_blocks, block_size), dtype=np.float32)).astype(np.float32)
        if kind == "zero_q":
            q[:] = 0
    bt_rows, bt_stride = block_table_shape
    perm = _rng(seed, 405).permutation(num_blocks).astype(np.int32)
    need = bt_rows * bt_stride
    if need > num_blocks:
        raise ValueError("block table larger than the block pool")
    bt = perm[:need].reshape(bt_rows, bt_stride).copy()
    r2b = None if row_to_batch is None else np.asarray(row_to_batch, dtype=np.int32)
    return FusedInputs(q, w, kc, ks, bt, seq_lens, r2b, k, name, dtype=dtype)


def fused_decode(seed: int = 4, rows: int = 64, min_len: int = 4096, max_len: int = 32768,
                 heads: int = IDX_HEADS, dim: int = HEAD_DIM, dtype: str = "e4m3") -> FusedInputs:
    """Decode: one query row per request, each with its own block-table row."""
    lens = _rng(seed, 303).integers(min_len, max_len + 1, size=rows).astype(np.int32)
    per_row = -(-max_len // KV_BLOCK)
    return make_fused_inputs(seed, rows, heads, dim, rows * per_row, lens, (rows, per_row),
                             name="fused_decode", dtype=dtype)


def fused_prefill(seed: int = 5, rows: int = 4096, kv_len: int = 32768,
                  heads: int = IDX_HEADS, dim: int = HEAD_DIM, dtype: str = "e4m3") -> FusedInputs:
    """Prefill of one request: the query rows are the last ``rows`` positions
    of a ``kv_len``-token KV, so row r sees ``kv_len - rows + r + 1`` keys."""
    blocks = -(-kv_len // KV_BLOCK)
    lens = (kv_len - rows + 1 + np.arange(rows)).astype(np.int32)
    r2b = np.zeros(rows, np.int32)
    return make_fused_inputs(seed, rows, heads, dim, blocks, lens, (1, blocks), row_to_batch=r2b,
                             name="fused_prefill", dtype=dtype)
