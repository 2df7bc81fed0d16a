"""Pins of the oracle's two ablation quantizers ("Echo: Error-Compensated 4-Bit
Tensor-Parallel Communication", Table 8: "naive zero-point" and "symmetric
grid"; their formulas are not printed).  The readings:

  naive zero-point  range [min v, max v] without 0; offset m = fp16 rounding of
                    min v toward -inf, stored where the zero point goes; step
                    (max v - m)/(2^b - 1) rounded up to fp16; codes
                    rint((v - m)/s) in [0, 2^b - 1]; decoded m + s*q.
  symmetric grid    step max|v|/(2^(b-1) - 1) rounded up to fp16; zero point
                    2^(b-1); codes rint(v/s) in +-(2^(b-1) - 1) plus the zero
                    point; decoded s*(q - z).

Checked as for the main quantizer: brute-force optimality over all codes, the
bounds that define s and m, symmetry, exact zero (or its absence), groups
worked by hand, and the error-feedback identity of a whole call.
"""
import numpy as np
import pytest

import oracle
from test_oracle_call import bf16_bits, random_x
from test_oracle_quantizer import _groups

NAIVE, SYM = oracle.NAIVE_ZERO_POINT, oracle.SYMMETRIC


def _f16(bits):
    return float(np.array([bits], np.uint16).view(np.float16)[0])


def test_f16_round_down_is_greatest_lower_bound():
    rng = np.random.default_rng(3)
    pos = rng.integers(0, 0x7F800000, 400_000, dtype=np.uint32)
    x = np.concatenate([pos, pos | np.uint32(0x80000000)]).view(np.float32)
    r = oracle.f32_to_f16_rd(x).view(np.float16)
    xd, rd = x.astype(np.float64), r.astype(np.float64)
    assert np.all(rd <= xd)
    with np.errstate(over="ignore"):
        above = np.nextafter(r, np.float16(np.inf)).astype(np.float64)
    assert np.all(above > xd)
    assert oracle.f32_to_f16_rd(np.array([0.0], np.float32))[0] == 0


@pytest.mark.parametrize("bits", [4, 8])
def test_naive_offset_and_step_bounds(bits):
    L = (1 << bits) - 1
    rng = np.random.default_rng(60 + bits)
    for v in _groups(rng, bits):
        q, sb, mb, bad, _ = oracle.quantize_group(v, bits, mode=NAIVE)
        assert bad == 0
        m = _f16(mb)
        lo, hi = float(v.min()), float(v.max())
        # m is the greatest fp16 value not above min v
        assert m <= lo
        assert float(np.nextafter(np.float16(m), np.float16(np.inf))) > lo
        s32 = (np.float32(hi) - np.float32(m)) / np.float32(L)
        s = _f16(sb)
        if s32 == 0:
            assert sb == 0x3C00
        else:
            assert s >= float(s32)
            assert float(np.nextafter(np.float16(s), np.float16(-np.inf))) < float(s32)


@pytest.mark.parametrize("bits", [4, 8])
def test_naive_codes_brute_force_and_error(bits):
    L = (1 << bits) - 1
    rng = np.random.default_rng(70 + bits)
    for v in _groups(rng, bits):
        q, sb, mb, _, _ = oracle.quantize_group(v, bits, mode=NAIVE)
        s, m = _f16(sb), _f16(mb)
        deq = oracle.dequantize_group(q, sb, mb, mode=NAIVE).astype(np.float64)
        # decoding is m + s*q in fp32 (one multiply, one add)
        want = (np.float32(s) * q.astype(np.float32) + np.float32(m)).astype(np.float64)
        assert np.array_equal(deq, want)
        codes = np.arange(L + 1, dtype=np.float64)
        err = np.abs(v.astype(np.float64)[:, None] - (m + s * codes[None, :]))
        chosen = err[np.arange(v.size), q.astype(np.int64)]
        slack = s * 2.0 ** -18 + np.abs(v) * 2.0 ** -22
        assert np.all(chosen <= err.min(axis=1) + slack)
        assert np.max(np.abs(v - deq) - slack) <= s / 2


@pytest.mark.parametrize("bits", [4, 8])
def test_symmetric_step_codes_and_mirror(bits):
    half = 1 << (bits - 1)
    Lh = half - 1
    rng = np.random.default_rng(80 + bits)
    for v in _groups(rng, bits):
        q, sb, zb, bad, _ = oracle.quantize_group(v, bits, mode=SYM)
        assert bad == 0 and _f16(zb) == half
        s = _f16(sb)
        a = np.float32(np.max(np.abs(v)))
        s32 = a / np.float32(Lh)
        if s32 == 0:
            assert sb == 0x3C00
        else:
            assert s >= float(s32)
            assert float(np.nextafter(np.float16(s), np.float16(-np.inf))) < float(s32)
        assert q.min() >= 1 and q.max() <= 2 * half - 1       # code 0 is never used
        # brute force over the usable codes
        codes = np.arange(1, 2 * half, dtype=np.float64)
        err = np.abs(v.astype(np.float64)[:, None] - s * (codes[None, :] - half))
        chosen = err[np.arange(v.size), q.astype(np.int64) - 1]
        assert np.all(chosen <= err.min(axis=1) + s * 2.0 ** -20)
        # odd symmetry: negating the group mirrors the codes about the zero point
        q2, sb2, _, _, _ = oracle.quantize_group(-v, bits, mode=SYM)
        assert sb2 == sb and np.array_equal(q2.astype(int) - half, -(q.astype(int) - half))
        # zero is exact
        zeros = v == 0
        assert np.all(q[zeros] == half)


def test_worked_groups_by_hand():
    """Naive zero-point, 4-bit, [-1, 0, 1, 2]: m = -1 (fp16 0xBC00); step
    3/15 = 0.2 rounded up to fp16 is 1639/8192 (0x3267); codes rint((v+1)/s) =
    0, 5, 10, 15; 0 decodes to -1 + 5*1639/8192 = 3/8192, not 0.

    Symmetric, 4-bit, [-1.5, 0, 0.5, 3]: step 3/7 = 0.4285714 rounded up to fp16
    is 439/1024 (0x36DC); codes rint(v/s) + 8 = 5, 8, 9, 15."""
    q, sb, mb, _, _ = oracle.quantize_group(np.array([-1, 0, 1, 2], np.float32), 4, mode=NAIVE)
    assert (sb, mb, list(q)) == (0x3267, 0xBC00, [0, 5, 10, 15])
    d = oracle.dequantize_group(q, sb, mb, mode=NAIVE)
    assert list(d) == [-1.0, 3 / 8192, 8198 / 8192, 16393 / 8192]
    q, sb, zb, _, _ = oracle.quantize_group(np.array([-1.5, 0, 0.5, 3], np.float32), 4, mode=SYM)
    assert (sb, zb, list(q)) == (0x36DC, 0x4800, [5, 8, 9, 15])
    d = oracle.dequantize_group(q, sb, zb, mode=SYM)
    assert list(d) == [-3 * 439 / 1024, 0.0, 439 / 1024, 7 * 439 / 1024]


@pytest.mark.parametrize("mode", [NAIVE, SYM])
def test_whole_call_invariants_and_error_feedback(mode):
    """Any quantizer keeps the call's structure: identical outputs, at most two
    quantizations, and error feedback's identity D_N = -E_N."""
    P, n, g, bits, N = 4, 4 * 256, 128, 4, 100
    rng = np.random.default_rng(90 + mode)
    e = np.zeros((P, n), np.float32)
    D = np.zeros(n)
    for k in range(N):
        x = random_x(rng, P, n)
        r = oracle.allreduce(x, g, bits, e=e, mode=mode, want_nq=True)
        assert r["flagged"] == 0 and r["nq"].max() <= 2
        assert all(np.array_equal(r["out"][p], r["out"][0]) for p in range(P))
        D += oracle.bf16_to_f32(r["out"][0]) - oracle.bf16_to_f32(x).astype(np.float64).sum(0)
    assert np.max(np.abs(D + e.astype(np.float64).sum(0))) <= N * P * 2.0 ** -22 * 8


def test_zero_handling_distinguishes_the_quantizers():
    """A group holding exact zeros: the zero-aware and symmetric quantizers send
    0 exactly, the naive zero-point one in general does not (Table 8's point)."""
    v = np.array([-0.3, 0.0, 0.7, 0.0, 1.1, -0.05], np.float32)
    for mode, exact in [(oracle.ZERO_AWARE, True), (SYM, True), (NAIVE, False)]:
        q, sb, zb, _, _ = oracle.quantize_group(v, 4, mode=mode)
        d = oracle.dequantize_group(q, sb, zb, mode=mode)
        assert (np.all(d[v == 0] == 0)) == exact, mode
