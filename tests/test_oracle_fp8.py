"""Pins of the oracle's E4M3FN decoder (CPU only)."""

import os

import numpy as np
import pytest
import torch

from oracle.fp8 import e4m3fn_decode, e4m3fn_units

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3fn_spec_values.txt")


def _spec_table():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            rows.append((int(code, 16), float(val)))
    return rows


def test_spec_values():
    """Values printed by the OCP OFP8 specification for E4M3."""
    for code, val in _spec_table():
        got = float(e4m3fn_decode(np.array([code], np.uint8))[0])
        if np.isnan(val):
            assert np.isnan(got), hex(code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)


def test_all_codes_match_torch():
    """All 256 codes against torch's float8_e4m3fn -> float32 conversion."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = e4m3fn_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}


def test_units_are_exact_multiples():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    units = e4m3fn_units(codes)
    assert np.array_equal(units.astype(np.float64) * 2.0**-9, e4m3fn_decode(codes))
    assert units.max() == 229376 and units.min() == -229376  # +-448


def test_units_reject_nan():
    with pytest.raises(ValueError):
        e4m3fn_units(np.array([0x7F], np.uint8))
