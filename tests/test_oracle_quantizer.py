"""Pins of the oracle's group quantizer Q_b.

The pages name the quantizer ("zero-aware asymmetric, g=128", Table 8 of "Echo:
Error-Compensated 4-Bit Tensor-Parallel Communication", formula "Eqn. (8)" not
printed) and its transport format (article "Your All-Reduce Is 4x Overpriced",
section "The cancellation rule": 4-bit integers with half-precision parameters
per group).  The reading the oracle implements: range [min(0, min v), max(0,
max v)], fp16 step rounded up, integer zero point, codes rint(v/s) + z.

The checks below use properties, not the formula retyped: brute-force
optimality of every code over all 2^b codes, the least-upper-bound property of
the step, exact decoding of 0, the half-step error bound, scale invariance and
closed-form special cases.
"""
import numpy as np
import pytest

import oracle


def _groups(rng, bits, count=300, g=128):
    """Groups of the shapes that stress the quantizer."""
    out = []
    for k in range(count):
        kind = k % 10
        if kind == 0:
            v = rng.standard_normal(g)
        elif kind == 1:
            v = np.abs(rng.standard_normal(g)) + 0.5          # all positive
        elif kind == 2:
            v = -np.abs(rng.standard_normal(g)) - 0.5         # all negative
        elif kind == 3:
            v = np.full(g, rng.standard_normal())             # constant
        elif kind == 4:
            v = np.zeros(g)
            v[rng.integers(g)] = rng.standard_normal() * 10    # single nonzero
        elif kind == 5:
            v = rng.standard_normal(g) * 1e-3                  # small
        elif kind == 6:
            v = rng.standard_t(4, g) * 50                      # heavy tails
        elif kind == 7:
            v = rng.standard_normal(g)
            v[rng.integers(g, size=8)] = 0.0                   # exact zeros inside
        elif kind == 8:
            L = (1 << bits) - 1                                # on-grid values: exact ties inside
            s = 2.0 ** rng.integers(-6, 3)
            v = (rng.integers(0, 2 * L + 1, g) * 0.5 - L / 3) * s
        else:
            v = rng.uniform(-3, 7, g)
        out.append(np.asarray(v, dtype=np.float32))
    return out


@pytest.mark.parametrize("g", [64, 128, 256])
@pytest.mark.parametrize("bits", [4, 8])
def test_codes_are_brute_force_optimal(bits, g):
    """Each code minimises |v - s(q - z)| over all 2^b codes for the chosen (s, z),
    up to the rounding of the fp32 quotient v/s; exact ties go to the even q - z."""
    L = (1 << bits) - 1
    rng = np.random.default_rng(10 + bits + g)
    ties_seen = 0
    for v in _groups(rng, bits, g=g):
        q, sb, zb, bad, _ = oracle.quantize_group(v, bits)
        assert bad == 0
        s = float(oracle.f16_to_f32([sb])[0])
        z = float(oracle.f16_to_f32([zb])[0])
        assert z == int(z) and 0 <= z <= L
        codes = np.arange(L + 1, dtype=np.float64)
        err = np.abs(v.astype(np.float64)[:, None] - s * (codes[None, :] - z))
        best = err.min(axis=1)
        chosen = err[np.arange(v.size), q.astype(np.int64)]
        assert np.all(chosen <= best + s * 2.0 ** -20), (v, q, s, z)
        # exact ties between two codes: the chosen q - z is even (half-to-even)
        second = np.sort(err, axis=1)[:, 1]
        tie = (np.abs(best - second) == 0) & (best > 0)
        for i in np.nonzero(tie)[0]:
            ties_seen += 1
            assert (int(q[i]) - int(z)) % 2 == 0, (v[i], q[i], z, s)
    if bits == 4:
        assert ties_seen > 0  # the on-grid groups do produce exact ties


@pytest.mark.parametrize("g", [64, 128, 256])
@pytest.mark.parametrize("bits", [4, 8])
def test_step_is_least_fp16_above_range_over_levels(bits, g):
    """s is the smallest fp16 value >= fl32((hi - lo) / (2^b - 1)), with the range
    widened to contain 0; an all-zero group gets s = 1."""
    L = (1 << bits) - 1
    rng = np.random.default_rng(20 + bits + g)
    for v in _groups(rng, bits, g=g):
        _, sb, _, _, _ = oracle.quantize_group(v, bits)
        s = np.array([sb], np.uint16).view(np.float16)[0]
        lo = np.float32(min(0.0, float(v.min())))
        hi = np.float32(max(0.0, float(v.max())))
        s32 = np.float32(hi - lo) / np.float32(L)
        if s32 == 0:
            assert sb == 0x3C00
            continue
        assert float(s) >= float(s32)
        assert float(np.nextafter(s, np.float16(-np.inf))) < float(s32)


@pytest.mark.parametrize("bits", [4, 8])
def test_zero_decodes_exactly_and_bottom_code_covers_min(bits):
    rng = np.random.default_rng(30 + bits)
    for v in _groups(rng, bits):
        q, sb, zb, _, _ = oracle.quantize_group(v, bits)
        s = float(oracle.f16_to_f32([sb])[0])
        z = int(oracle.f16_to_f32([zb])[0])
        deq = oracle.dequantize_group(q, sb, zb)
        # code z decodes to exactly 0, and every 0 input is sent as code z
        assert oracle.dequantize_group(np.array([z], np.uint8), sb, zb)[0] == 0.0
        zeros = v == 0
        assert np.all(q[zeros] == z) and np.all(deq[zeros] == 0.0)
        # code 0 decodes to within half a step of lo = min(0, min v)
        lo = min(0.0, float(v.min()))
        assert abs(lo - (-z * s)) <= s / 2 * (1 + 2.0 ** -20)


@pytest.mark.parametrize("bits", [4, 8])
def test_error_at_most_half_step(bits):
    rng = np.random.default_rng(40 + bits)
    for v in _groups(rng, bits, count=600):
        q, sb, zb, _, _ = oracle.quantize_group(v, bits)
        s = float(oracle.f16_to_f32([sb])[0])
        deq = oracle.dequantize_group(q, sb, zb).astype(np.float64)
        assert np.max(np.abs(v - deq)) <= s / 2 * (1 + 2.0 ** -20)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("k", [-5, -1, 1, 4])
def test_scale_invariance_by_powers_of_two(bits, k):
    """Scaling a group by 2^k (inside fp16's normal range) keeps codes and zero
    point and scales the step exactly."""
    rng = np.random.default_rng(50 + bits)
    for v in _groups(rng, bits, count=120):
        if not np.any(v):
            continue
        q, sb, zb, _, _ = oracle.quantize_group(v, bits)
        s = float(oracle.f16_to_f32([sb])[0])
        # both steps must be fp16 normal numbers for the scaling to be exact
        if not (2.0 ** -14 <= min(s, s * 2.0 ** k) and max(s, s * 2.0 ** k) < 2.0 ** 15):
            continue
        q2, sb2, zb2, _, _ = oracle.quantize_group(v * np.float32(2.0 ** k), bits)
        assert np.array_equal(q, q2) and zb == zb2
        assert float(oracle.f16_to_f32([sb2])[0]) == s * 2.0 ** k


@pytest.mark.parametrize("bits", [4, 8])
def test_closed_form_special_groups(bits):
    L = (1 << bits) - 1
    g = 128
    # all zero: step 1, zero point 0, every code 0
    q, sb, zb, bad, _ = oracle.quantize_group(np.zeros(g, np.float32), bits)
    assert (sb, zb, bad) == (0x3C00, 0, 0) and not q.any()
    # constant positive c: range [0, c]; every code is the top code, zero point 0
    q, sb, zb, _, _ = oracle.quantize_group(np.full(g, 3.7, np.float32), bits)
    assert zb == 0 and np.all(q == L)
    # constant negative: range [c, 0]; zero point is the top code, every code 0
    q, sb, zb, _, _ = oracle.quantize_group(np.full(g, -3.7, np.float32), bits)
    assert oracle.f16_to_f32([zb])[0] == L and not q.any()
    # values already on the grid {0..L} * 2^-3 with both ends present: lossless
    v = (np.arange(g) % (L + 1)).astype(np.float32) * np.float32(0.125)
    v[-1] = L * 0.125
    q, sb, zb, _, _ = oracle.quantize_group(v, bits)
    assert oracle.f16_to_f32([sb])[0] == 0.125 and zb == 0
    assert np.array_equal(oracle.dequantize_group(q, sb, zb), v)


def test_worked_single_groups():
    """Two groups worked by hand from the definition (4-bit, L = 15).

    [3.0, 0.0]: range [0, 3]; 3/15 = 0.2 in fp32 (0.200000003); the fp16 values
    around it are 1638/8192 = 0.19995 and 1639/8192 = 0.20007, so s = 1639/8192
    (bits 0x3267), z = 0, codes rint(3/s) = rint(14.9945) = 15 and 0.

    [0.25, 2.0]: range [0, 2]; 2/15 = 0.13333334 in fp32, rounded up to fp16 is
    1093/8192 (bits 0x3045); codes rint(2048/1093) = 2 and rint(16384/1093) = 15.
    """
    q, sb, zb, _, _ = oracle.quantize_group(np.array([3.0, 0.0], np.float32), 4)
    assert (sb, zb, list(q)) == (0x3267, 0, [15, 0])
    q, sb, zb, _, _ = oracle.quantize_group(np.array([0.25, 2.0], np.float32), 4)
    assert (sb, zb, list(q)) == (0x3045, 0, [2, 15])
    # decoding: 15 * 1639/8192 = 24585/8192, exact in fp32
    assert oracle.dequantize_group(np.array([15], np.uint8), 0x3267, 0)[0] == 24585 / 8192


def test_flags_non_finite_and_scale_overflow():
    v = np.ones(128, np.float32)
    v[5] = np.inf
    assert oracle.quantize_group(v, 4)[3] == 1
    v[5] = np.nan
    assert oracle.quantize_group(v, 4)[3] == 1
    # range 1e6 / 15 > 65504: the fp16 step overflows
    v = np.linspace(0, 1e6, 128).astype(np.float32)
    assert oracle.quantize_group(v, 4)[3] == 1
    # just inside: 65504 * 15
    v = np.linspace(0, 65504 * 15, 128).astype(np.float32)
    assert oracle.quantize_group(v, 4)[3] == 0


def test_packing_nibble_order():
    """Element 2i in the low nibble of byte i, element 2i+1 in the high nibble."""
    q = np.array([1, 2, 3, 4, 15, 0], np.uint8)
    assert list(oracle.pack_codes(q, 4)) == [0x21, 0x43, 0x0F]
    assert list(oracle.pack_codes(np.array([5, 6, 7], np.uint8), 4)) == [0x65, 0x07]
    assert list(oracle.pack_codes(np.array([200, 7, 255], np.uint8), 8)) == [200, 7, 255]
