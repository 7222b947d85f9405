"""CPU oracle for the sparse-attention indexer top-k path.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, obviously correct
restatement of what the indexer computes, used to check the CUDA library. Only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it. The library in
``sparse_attention_indexer_top_gb300`` never imports it and shares no code with
it; only the seeded input generators in ``workloads`` serve both.

Modules
-------
``fp8``    OCP E4M3FN decoding written from the format's bit definition.
``bf16``   bfloat16 decoding written from the format's bit definition.
``topk``   per-row window top-k (stable sort) and the page-table transform.
``score``  the index score (FP8 or bf16 cache), the fused score + top-k, and
           the per-index-head scores and top-k.
``brute``  O(n^2) rank-rule selection, used only to pin ``topk``.
``blocks`` per-row distinct KV blocks of the selected slots.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
brute force, invariants or library routines; none is "parity unpinned".
"""

from .fp8 import e4m3fn_decode, e4m3fn_units  # noqa: F401
from .bf16 import bf16_decode  # noqa: F401
from .topk import topk_row, page_transform, topk_transform  # noqa: F401
from .score import index_scores_row, index_scores, index_score_topk  # noqa: F401
from .score import index_scores_per_head, index_score_topk_per_head  # noqa: F401
from .brute import rank_select_bruteforce  # noqa: F401
from .blocks import sparse_blocks  # noqa: F401
