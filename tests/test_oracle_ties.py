"""Pins of the oracle's count of exact rounding ties.

Codes are rint (half to even) of v/s plus an integer zero point, itself a rint
of -lo/s (the zero-aware quantizer's reading of "Echo: Error-Compensated 4-Bit
Tensor-Parallel Communication", Table 8, formula not printed).  An exact tie is
a rint whose fp32 argument lies exactly on a half-integer, where both
neighbouring codes are equally near and half-to-even decides; such ties must be
counted and reported, since they are the only places where a code of another
implementation could differ by one.

The inputs below fix the number of ties by construction, independently of the
oracle's arithmetic:
  * a group holding its two extreme values -k0*s and (L - k0)*s, s a power of
    two, has step s and zero point k0 exactly (range L*s, exact in fp32 and
    fp16), so every value h*s/2 gives v/s = h/2 exactly: a tie iff h is odd,
    whatever its sign;
  * a group whose extremes are -(k0 + 1/2)*s and (L - k0 - 1/2)*s has the same
    step and a zero point -lo/s = k0 + 1/2: one more tie;
  * values (h + 1/2 +- 2^-t)*s, t = 10..22, exact in fp32, are near ties: they
    must not count.
Stage 1 (the push) and stage 2 (the owner's requantization) are checked apart:
groups of all zeros produce no tie, so a call whose senders hold zeros counts
only the owner's stage-2 ties, and a call whose one nonzero sender holds a
grid group with integer extremes (decoded exactly, so the owner's sum is back
on the integer grid of the same step) counts only that sender's stage-1 ties.
"""
import numpy as np
import pytest

import oracle

PLAIN, ZP = "plain", "zero-point tie"


def _near(rng, h_half, s):
    """A value (h_half +- 2^-t)*s, exact in fp32, with t as large as fits in
    10..22 (h_half a half-integer)."""
    sign = 1.0 if rng.random() < 0.5 else -1.0
    for t in range(int(rng.integers(10, 23)), 9, -1):
        val = (h_half + sign * 2.0 ** -t) * s
        if float(np.float32(val)) == val:
            return val
    raise AssertionError("no exact near tie")


def tie_group(rng, bits, g, kind, near_frac=0.25):
    """A group of g fp32 values with a known number of exact rounding ties.

    Returns (v, ties, near, negative_ties): v float32 [g]; ties the exact ties
    the quantizer meets (codes and zero point); near the planted near ties;
    negative_ties the exact code ties at negative v."""
    L = (1 << bits) - 1
    s = 2.0 ** int(rng.integers(-6, 2))
    if kind == PLAIN:
        k0 = int(rng.integers(0, L + 1))
        lo_h, hi_h = -2 * k0, 2 * (L - k0)             # v = h*s/2 for h in [lo_h, hi_h]
        zp_tie = 0
    else:
        k0 = int(rng.integers(0, L))
        lo_h, hi_h = -(2 * k0 + 1), 2 * (L - k0) - 1   # extremes on half-integers
        zp_tie = 1
    h = rng.integers(lo_h, hi_h + 1, g)
    h[0], h[1] = lo_h, hi_h                            # both extremes present
    v = h * (s / 2)
    near = np.zeros(g, bool)
    inner = np.nonzero((h % 2 == 1) & (h > lo_h) & (h < hi_h))[0]
    inner = inner[inner >= 2]
    pick = inner[rng.random(inner.size) < near_frac]
    for i in pick:
        v[i] = _near(rng, h[i] / 2, s)
        near[i] = True
    exact = (h % 2 == 1) & ~near
    assert np.array_equal(v.astype(np.float32).astype(np.float64), v)   # all exact in fp32
    return (v.astype(np.float32), int(exact.sum()) + zp_tie, int(near.sum()),
            int((exact & (h < 0)).sum()))


@pytest.mark.parametrize("g", [64, 128, 256])
@pytest.mark.parametrize("bits", [4, 8])
def test_group_tie_count_by_construction(bits, g):
    rng = np.random.default_rng(700 + bits + g)
    L = (1 << bits) - 1
    tot_near = tot_neg = tot_zp = 0
    for k in range(240):
        kind = ZP if k % 3 == 2 else PLAIN
        v, ties, near, neg = tie_group(rng, bits, g, kind)
        q, sb, zb, bad, got = oracle.quantize_group(v, bits)
        assert bad == 0
        s = float(oracle.f16_to_f32([sb])[0])
        assert s == float(np.max(v) - np.min(v)) / L     # the step the construction fixes
        assert got == ties, (kind, got, ties)
        tot_near += near
        tot_neg += neg
        tot_zp += kind == ZP
    # the construction exercises what a wrong counter would get wrong
    assert tot_near > 500 and tot_neg > 500 and tot_zp == 80


@pytest.mark.parametrize("bits", [4, 8])
def test_near_ties_integers_and_zero_groups_count_nothing(bits):
    """Groups with no value on a half-integer quotient and an integer zero point:
    the count must stay 0, near ties (down to 2^-22 of a step) included."""
    rng = np.random.default_rng(710 + bits)
    L = (1 << bits) - 1
    for k in range(200):
        s = 2.0 ** int(rng.integers(-6, 2))
        k0 = int(rng.integers(0, L + 1))
        h = 2 * rng.integers(-k0, L - k0 + 1, 128)            # integers only
        h[0], h[1] = -2 * k0, 2 * (L - k0)
        v = h * (s / 2)
        odd = rng.integers(-k0, L - k0, 128) + 0.5          # half-integers strictly inside
        for i in range(2, 128, 2):
            v[i] = _near(rng, odd[i], s)
        assert oracle.quantize_group(v.astype(np.float32), bits)[4] == 0
    for v in (np.zeros(128, np.float32), np.full(128, 3.0, np.float32)):
        assert oracle.quantize_group(v, bits)[4] == 0


def _call_inputs(rng, P, bits, g, npos, stage):
    """Inputs for oracle.group_positions: x all +0 (bf16), the values carried in
    the compensator state e, so that v = 0 + e = e exactly.  For stage 1 one
    sender per position holds a PLAIN group, everything else is 0; for stage 2
    the owner holds a PLAIN or ZP group and every sender 0."""
    owners = (np.arange(npos) % P).astype(np.int32)
    x = np.zeros((npos, P, g), np.uint16)
    e = np.zeros((npos, P, g), np.float32)
    expected = 0
    for k in range(npos):
        o = int(owners[k])
        if stage == 1:
            p = (o + 1 + k // P) % P
            if p == o:
                p = (p + 1) % P
            v, ties, _, _ = tie_group(rng, bits, g, PLAIN)
        else:
            p = o
            v, ties, _, _ = tie_group(rng, bits, g, ZP if k % 2 else PLAIN)
        e[k, p] = v
        expected += ties
    return owners, x, e, expected


@pytest.mark.parametrize("P", [2, 3, 4, 8])
@pytest.mark.parametrize("bits", [4, 8])
def test_stage1_ties_counted_through_a_call(P, bits):
    rng = np.random.default_rng(720 + P + bits)
    owners, x, e, expected = _call_inputs(rng, P, bits, 128, 96, stage=1)
    e_sender = e.copy()
    r = oracle.group_positions(P, owners, bits, x, e, want_wire=True)
    assert r["flagged"] == 0
    assert r["ties"] == expected and expected > 1000
    # the owner's sum is the sender's decoded group, back on the step's integer
    # grid: it is quantized losslessly, with the sender's step
    for k in range(owners.size):
        o = int(owners[k])
        p = int(np.nonzero(e_sender[k].any(axis=1))[0][0])
        assert p != o and r["m2"][k] == r["m1"][k, p]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("bits", [4, 8])
def test_stage2_ties_counted_through_a_call(P, bits):
    rng = np.random.default_rng(730 + P + bits)
    owners, x, e, expected = _call_inputs(rng, P, bits, 128, 96, stage=2)
    r = oracle.group_positions(P, owners, bits, x, e, want_wire=True)
    assert r["flagged"] == 0
    assert r["ties"] == expected and expected > 1000
    # every sender held zeros: step 1, zero point 0, all codes 0
    for k in range(owners.size):
        for p in range(P):
            if p != owners[k]:
                assert r["m1"][k, p] == 0x3C00 and not r["q1"][k, p].any()


def _whole_call_values(rng, P, bits, g, Gs, near_frac):
    """[P, n] values for one call: even-numbered groups of each segment tie at
    stage 1 (one sender holds a PLAIN group), odd-numbered ones at stage 2 (the
    owner holds a PLAIN or ZP group); everything else is 0."""
    n = P * g * Gs
    vals = np.zeros((P, n), np.float32)
    expected = 0
    for o in range(P):
        for j in range(Gs):
            sl = slice(o * Gs * g + j * g, o * Gs * g + (j + 1) * g)
            if j % 2 == 0:
                p = (o + 1 + j // 2) % P
                p = p if p != o else (p + 1) % P
                v, ties, _, _ = tie_group(rng, bits, g, PLAIN, near_frac)
            else:
                p = o
                v, ties, _, _ = tie_group(rng, bits, g, ZP if j % 4 == 1 else PLAIN, near_frac)
            vals[p, sl] = v
            expected += ties
    return vals, expected


@pytest.mark.parametrize("bits", [4, 8])
def test_whole_call_counts_both_stages(bits):
    """The construction through oracle.allreduce on a [P, n] call, with the values
    in the compensator state; the total is the sum over both stages."""
    P, g, Gs = 4, 128, 12
    rng = np.random.default_rng(740 + bits)
    e, expected = _whole_call_values(rng, P, bits, g, Gs, 0.25)
    x = np.zeros(e.shape, np.uint16)
    r = oracle.allreduce(x, g, bits, e=e)
    assert r["flagged"] == 0 and r["ties"] == expected


def test_whole_call_counts_ties_of_bf16_inputs_uncompensated():
    """Uncompensated, with the values carried by the bf16 inputs themselves (a
    4-bit half-step grid needs at most 6 significant bits, exact in bf16)."""
    P, g, Gs, bits = 3, 128, 10, 4
    rng = np.random.default_rng(750)
    vals, expected = _whole_call_values(rng, P, bits, g, Gs, 0.0)
    x = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(oracle.bf16_to_f32(x), vals)
    r = oracle.allreduce(x, g, bits)
    assert r["flagged"] == 0 and r["ties"] == expected and expected > 500
