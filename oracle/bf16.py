"""bfloat16 decoding, written from the format definition.

The index cache of the sparse-attention indexer may also be kept at the
model's own dtype: ROCm/ATOM PR #1473 "enable minimax m3 fp8 index cache and
fuse index_score_kernel with partial_topk kernel" adds an index-cache type
option whose default "auto" means the model dtype (review of the ``--index-
cache-dtype`` help text, and the commit "convert auto for bf16 type"); the
FP8 cache is used only when the KV cache dtype is an fp8 one. For the model
served there the "auto" type is bfloat16, whose encoding is the upper 16 bits
of an IEEE-754 binary32:

* 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits;
* exponent field 0: subnormal, value = mantissa * 2^-133;
* exponent field 1..254: value = (1 + mantissa/128) * 2^(e-127);
* exponent field 255: infinity (mantissa 0) or NaN.
"""

from __future__ import annotations

import numpy as np


def _fields(bits: np.ndarray):
    c = np.asarray(bits).astype(np.int64) & 0xFFFF
    return c >> 15, (c >> 7) & 0xFF, c & 0x7F


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """float64 value of each bfloat16 bit pattern (uint16)."""
    sign, exp, man = _fields(bits)
    m = man.astype(np.float64)
    e = exp.astype(np.float64)
    mag = np.where(exp == 0, m * 2.0**-133, (1.0 + m / 128.0) * np.exp2(np.minimum(e, 254.0) - 127.0))
    mag = np.where(exp == 255, np.where(man == 0, np.inf, np.nan), mag)
    return np.where(sign == 1, -mag, mag)


def bf16_finite(bits: np.ndarray) -> np.ndarray:
    """float64 values of finite bfloat16 patterns; ``ValueError`` on inf/NaN."""
    _, exp, _ = _fields(bits)
    if np.any(exp == 255):
        raise ValueError("non-finite bfloat16 value")
    return bf16_decode(bits)
