"""Pins for the oracle's binary16 / bfloat16 codecs against numpy and torch's own conversions.

The block-format specification (section 4) fixes f16() and bf16() as round-to-nearest-even; numpy's
float32 -> float16 cast and torch's float32 -> bfloat16 cast are both that rounding, and numpy's float16
and float32 interpretations define the decoded values.
"""
import numpy as np
import pytest
import torch


def test_f16_decode_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signs of zeros too
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_decode_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint32)
    want = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([orc.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _f32_probe_values():
    g = np.random.default_rng(1234)
    vals = [g.standard_normal(4000).astype(np.float32) * np.float32(s) for s in (1e-6, 1e-3, 0.02, 1, 300, 6e4)]
    # every binary16 value and every midpoint between neighbours (ties), as float32
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2
    vals += [h.astype(np.float32), mids.astype(np.float32), -mids.astype(np.float32)]
    # neighbours of the ties
    m32 = mids.astype(np.float32)
    vals += [np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(0))]
    vals.append(np.array([0.0, -0.0, 65504, 65519.99, 65520, 70000, -65520, 5.96e-8, 2.98e-8, 2.99e-8,
                          1e-9, np.inf, -np.inf], dtype=np.float32))
    return np.concatenate(vals).astype(np.float32)


def test_f16_encode_matches_numpy(orc):
    v = _f32_probe_values()
    want = v.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16(x) for x in v], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_f16_encode_nan(orc):
    h = orc.f32_to_f16(np.float32(np.nan))
    assert np.isnan(np.uint16(h).view(np.float16))


def test_bf16_encode_matches_torch(orc):
    g = np.random.default_rng(99)
    v = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(0.02),
        g.standard_normal(20000).astype(np.float32) * np.float32(1e30),
        # ties: float32 patterns whose low 16 bits are exactly 0x8000, both parities of bit 16
        (g.integers(0, 0x7F00, 5000).astype(np.uint32) << 16 | 0x8000).view(np.float32),
        # subnormal float32 inputs
        (g.integers(1, 0x007FFFFF, 5000).astype(np.uint32)).view(np.float32),
        np.array([0.0, -0.0, 3.3895314e38, 3.4028235e38, np.inf, -np.inf], dtype=np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16(x) for x in v], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]
