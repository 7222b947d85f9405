"""Seeded synthetic inputs shared by the tests, the oracle runs and ``bench.py``.

Only random draws and array layout live here; none of the indexer's arithmetic
(no ordering keys, no selection, no dot products, no page transform).
"""

from .gen import (  # noqa: F401
    CONFIGS,
    TopkInputs,
    FusedInputs,
    e4m3fn_encode,
    bf16_encode,
    make_topk_inputs,
    make_fused_inputs,
    tiny_decode,
    decode_topk,
    packed_extend,
    packed_extend_meta,
    packed_extend_window,
    fused_decode,
    fused_prefill,
    page_table_perm,
    fill_rows,
)
