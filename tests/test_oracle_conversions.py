"""Pins for the oracle's 16-bit float handling.

The oracle widens f16 and bf16 exactly and rounds f32 to bf16 to nearest
even.  These are checked against independent library implementations
(NumPy's binary16, PyTorch's bfloat16 cast) over every 16-bit pattern and
over a sample of f32 values that covers ties, overflow, subnormals and
signed zeros.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _same(a: float, b: float) -> bool:
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def test_widen_f16_every_pattern_matches_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in range(0, 1 << 16, 1):
        if not _same(oracle.widen16(int(bits[b]), "f16"), float(ref[b])):
            pytest.fail(f"f16 pattern {b:#06x}: oracle {oracle.widen16(int(bits[b]), 'f16')} "
                        f"numpy {ref[b]}")


def test_widen_bf16_every_pattern_matches_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b in range(1 << 16):
        if not _same(oracle.widen16(int(bits[b]), "bf16"), float(ref[b])):
            pytest.fail(f"bf16 pattern {b:#06x}")


def _torch_bf16(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_f32_to_bf16_rounds_like_torch():
    rng = np.random.default_rng(1)
    # random bit patterns across the whole exponent range (NaNs removed)
    raw = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = raw.view(np.float32)
    vals = vals[~np.isnan(vals)]
    # exact ties: low half exactly 0x8000, with even and odd kept halves
    hi = rng.integers(0, 1 << 16, size=2000, dtype=np.uint32)
    ties = ((hi << 16) | 0x8000).astype(np.uint32).view(np.float32)
    ties = ties[~np.isnan(ties)]
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.finfo(np.float32).max,
                        -np.finfo(np.float32).max, np.finfo(np.float32).tiny,
                        1e-45, -1e-45, 1.0, -1.0, 3.0, 1.00390625, 1.01171875,
                        65504.0, 3.3895314e38], dtype=np.float32)
    sample = np.concatenate([vals, ties, special]).astype(np.float32)
    ours = oracle.f32_to_bf16_array(sample)
    ref = _torch_bf16(sample)
    mismatch = np.nonzero(ours != ref)[0]
    assert mismatch.size == 0, (
        f"{mismatch.size} mismatches, first {sample[mismatch[0]]!r}: "
        f"{ours[mismatch[0]]:#06x} vs {ref[mismatch[0]]:#06x}")


def test_f32_to_bf16_nan_stays_nan_with_sign():
    for pattern in (0x7fc00000, 0x7f800001, 0xffc00000, 0x7fffffff):
        x = np.array([pattern], dtype=np.uint32).view(np.float32)[0]
        out = oracle.f32_to_bf16(float(x))
        assert (out & 0x7f80) == 0x7f80 and (out & 0x7f) != 0, hex(out)
        assert (out >> 15) == (pattern >> 31)
