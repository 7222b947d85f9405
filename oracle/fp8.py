"""OCP E4M3FN decoding, written from the format definition.

The FP8 index-key cache of the fused path stores e4m3 codes (ROCm/ATOM PR
#1473 "enable minimax m3 fp8 index cache and fuse index_score_kernel with
partial_topk kernel": the pull request overview's "Enable FP8 dtype for the
MiniMax-M3 index cache" and the commit "fp8 index score calculate in fp8").
The pages name the dtype but not its encoding; the encoding is the OCP 8-bit
floating point format E4M3 in its "FN" variant:

* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
* exponent field 0: subnormal, value = mantissa * 2^-9;
* exponent field e > 0: value = (1 + mantissa/8) * 2^(e-7);
* no infinities; S.1111.111 is NaN; the largest finite value is 448.

Every finite code is an integer multiple of 2^-9 ("units"), which lets the
score oracle form dot products exactly.
"""

from __future__ import annotations

import numpy as np

UNIT_EXP = -9  # one unit = 2^-9


def _fields(codes: np.ndarray):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = c >> 7
    exp = (c >> 3) & 0xF
    man = c & 0x7
    return sign, exp, man


def e4m3fn_units(codes: np.ndarray) -> np.ndarray:
    """Signed integer value of each code in units of 2^-9 (int64).

    Raises ``ValueError`` on a NaN code (S.1111.111).
    """
    sign, exp, man = _fields(codes)
    if np.any((exp == 15) & (man == 7)):
        raise ValueError("NaN e4m3fn code")
    # subnormal: man units; normal: (8 + man) * 2^(exp-1) units
    mag = np.where(exp == 0, man, (8 + man) << np.maximum(exp - 1, 0))
    return np.where(sign == 1, -mag, mag).astype(np.int64)


def e4m3fn_decode(codes: np.ndarray) -> np.ndarray:
    """float64 value of each code; NaN codes decode to NaN."""
    sign, exp, man = _fields(codes)
    nan = (exp == 15) & (man == 7)
    mag = np.where(exp == 0, man.astype(np.float64) * 2.0**UNIT_EXP,
                   (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0))
    val = np.where(sign == 1, -mag, mag)
    return np.where(nan, np.nan, val)
