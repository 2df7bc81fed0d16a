"""Pins of the oracle's number-format conversions against independent routines.

The oracle writes its binary16 and bfloat16 conversions from the format
definitions.  Here they are checked against numpy's float16 type (ordering and
exact widening) and against torch's bfloat16 conversion, which are separate
implementations of the same IEEE formats.
"""
import numpy as np
import pytest
import torch

import oracle


def _sweep_f32(stride=4099, seed=0):
    """Positive and negative binary32 patterns spread over the whole range,
    plus the edges of binary16's range and its subnormals."""
    pos = np.arange(0, 0x7F800000, stride, dtype=np.uint32)
    rng = np.random.default_rng(seed)
    extra = rng.integers(0, 0x7F800000, 200_000, dtype=np.uint32)
    edges = np.array([65504.0, 65505.0, 65519.0, 65520.0, 65536.0, 1e30, 6.1035156e-05,
                      6.0975552e-05, 5.9604645e-08, 2.9802322e-08, 1e-30, 1.0, 0.2, 2.0 / 15,
                      np.finfo(np.float32).tiny, np.finfo(np.float32).max],
                     dtype=np.float32).view(np.uint32)
    # every binary16 value and its two binary32 neighbours
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    hb = h.view(np.uint32)
    around = np.concatenate([hb, hb + 1, np.maximum(hb, 1) - 1])
    allpos = np.concatenate([pos, extra, edges, around]).astype(np.uint32)
    return np.concatenate([allpos, allpos | np.uint32(0x80000000)]).view(np.float32)


def test_f16_round_nearest_even_matches_numpy():
    """Round to nearest, ties to even (the compensator's fp16 state), against
    numpy's float16 cast; the sweep adds every exact midpoint between
    consecutive binary16 values (the ties) and the overflow threshold 65520."""
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = ((h[:-1] + h[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (h[:-1] + h[1:]) / 2)      # exact in fp32
    x = np.concatenate([_sweep_f32(), mids, -mids,
                        np.array([65520.0, -65520.0, 65519.996, np.inf, -np.inf], np.float32)])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16_rn(x)
    assert np.array_equal(got, want)
    assert np.isnan(oracle.f32_to_f16_rn(np.array([np.nan], np.float32)).view(np.float16)[0])


def test_f16_round_up_is_least_upper_bound():
    x = _sweep_f32()
    r = oracle.f32_to_f16_ru(x).view(np.float16)
    xd = x.astype(np.float64)
    rd = r.astype(np.float64)
    # r is a binary16 value not below x ...
    assert np.all(rd >= xd), x[rd < xd][:5]
    # ... and the binary16 value just below r is below x (so r is the least one).
    with np.errstate(over="ignore"):
        below = np.nextafter(r, np.float16(-np.inf)).astype(np.float64)
    assert np.all(below < xd), x[below >= xd][:5]
    # beyond the largest finite binary16 a positive value goes to +inf
    assert np.all(np.isinf(rd[xd > 65504.0]))
    assert np.all(rd[xd < -65504.0] == -65504.0)


def test_f16_round_up_specials():
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0], dtype=np.float32)
    r = oracle.f32_to_f16_ru(specials)
    assert r[0] == 0x7C00 and r[1] == 0xFC00
    assert np.isnan(r[2:3].view(np.float16))[0]
    assert r[3] == 0x0000 and r[4] == 0x8000


def test_f16_to_f32_exact_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_bf16_round_nearest_even_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    # exact ties: low 16 bits 0x8000, with both parities of the kept bit
    ties = (rng.integers(0, 2**16, 100_000, dtype=np.uint32) << 16) | 0x8000
    x = np.concatenate([bits, ties]).view(np.float32)
    x = x[~np.isnan(x)]
    got = oracle.f32_to_bf16_rn(x)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_nan_stays_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    got = oracle.f32_to_bf16_rn(x)
    assert np.all(np.isnan(oracle.bf16_to_f32(got)))


@pytest.mark.parametrize("v", [0.2, 2.0 / 15, 3.0, 1e-3, 7.5e-5, 1234.5])
def test_f16_round_up_small_examples(v):
    r = oracle.f32_to_f16_ru(np.array([v], np.float32)).view(np.float16)[0]
    assert float(r) >= float(np.float32(v))
    assert float(np.nextafter(r, np.float16(-np.inf))) < float(np.float32(v))
