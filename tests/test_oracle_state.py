"""Pins of the compensator's options in the oracle: the held error stored in
bf16 or fp16 instead of fp32, and a decay applied to each revealed error
before it is kept.  (The pages describe a "two-timescale compensator" but print none of
its equations or constants; fp32 storage with decay 1 is the plain error
feedback every other test pins.)

Checked against: a one-rank call sequence recomputed step by step from the
group quantizer (pinned elsewhere), which fixes where the decay and the bf16
rounding enter; and drift over long sequences, which must stay far below the
uncompensated random walk.
"""
import numpy as np
import pytest

import oracle
from test_oracle_call import random_x


def _one_rank_reference(xs, bits, g, decay, fmt):
    """P = 1: the call quantizes v = x + e once per group; the new state is
    decay * (v - y), rounded to bf16 or fp16 when so stored."""
    n = xs[0].shape[1]
    e = np.zeros(n, np.float32)
    outs, states = [], []
    for x in xs:
        v = (oracle.bf16_to_f32(x[0]) + e).astype(np.float32)
        y = np.zeros(n, np.uint16)
        for j in range(n // g):
            sl = slice(j * g, (j + 1) * g)
            q, sb, zb, _, _ = oracle.quantize_group(v[sl], bits)
            y[sl] = oracle.f32_to_bf16_rn(oracle.dequantize_group(q, sb, zb))
        r = (v - oracle.bf16_to_f32(y)).astype(np.float32)
        t = (np.float32(decay) * r).astype(np.float32)
        if fmt == oracle.STATE_BF16:
            e = oracle.bf16_to_f32(oracle.f32_to_bf16_rn(t))
        elif fmt == oracle.STATE_F16:
            e = oracle.f16_to_f32(oracle.f32_to_f16_rn(t))
        else:
            e = t
        outs.append(y)
        states.append(e.copy())
    return outs, states


@pytest.mark.parametrize("fmt,decay", [(0, 0.75), (1, 1.0), (1, 0.5), (2, 1.0), (2, 0.5)])
def test_one_rank_sequence_recomputed_step_by_step(fmt, decay):
    rng = np.random.default_rng(5)
    g, bits, n = 128, 4, 128 * 6
    xs = [random_x(rng, 1, n) for _ in range(6)]
    want_y, want_e = _one_rank_reference(xs, bits, g, decay, fmt)
    e = np.zeros((1, n), np.float32)
    for k, x in enumerate(xs):
        r = oracle.allreduce(x, g, bits, e=e, state_fmt=fmt, decay=decay)
        assert np.array_equal(r["out"][0], want_y[k]), k
        assert np.array_equal(e[0].view(np.uint32), want_e[k].view(np.uint32)), k


def test_bf16_state_holds_bf16_values_on_every_rank():
    rng = np.random.default_rng(6)
    P, n = 4, 4 * 128 * 3
    e = np.zeros((P, n), np.float32)
    for _ in range(3):
        oracle.allreduce(random_x(rng, P, n), 128, 4, e=e, bf16_state=True)
    assert np.array_equal(oracle.bf16_to_f32(oracle.f32_to_bf16_rn(e)).reshape(P, n), e)
    assert np.any(e != 0)


def test_f16_state_holds_f16_values_on_every_rank():
    rng = np.random.default_rng(7)
    P, n = 4, 4 * 128 * 3
    e = np.zeros((P, n), np.float32)
    for _ in range(3):
        oracle.allreduce(random_x(rng, P, n), 128, 4, e=e, state_fmt=oracle.STATE_F16)
    assert np.array_equal(e.astype(np.float16).astype(np.float32), e)
    assert np.any(e != 0)


def _drift(P, n, N, seed, scale=1.0, **kw):
    rng = np.random.default_rng(seed)
    e = np.zeros((P, n), np.float32) if kw.pop("compensated", True) else None
    D = np.zeros(n)
    D1 = None
    for k in range(N):
        x = random_x(rng, P, n)
        if scale != 1.0:
            xf = (oracle.bf16_to_f32(x).reshape(P, n) * np.float32(scale)).astype(np.float32)
            x = oracle.f32_to_bf16_rn(xf).reshape(P, n)
        r = oracle.allreduce(x, 128, 4, e=e, **kw)
        D += oracle.bf16_to_f32(r["out"][0]) - oracle.bf16_to_f32(x).astype(np.float64).sum(0)
        if k == 0:
            D1 = D.copy()
    rms = lambda a: float(np.sqrt(np.mean(a * a)))
    return rms(D), rms(D1)


def test_drift_of_the_state_options():
    """Over 600 calls: bf16 storage adds only its rounding (drift stays near the
    fp32 one); a decay below 1 feeds back only part of each error, so the drift
    grows like a random walk of size (1 - decay), between the exact feedback
    and no feedback at all."""
    P, n, N = 2, 4096, 600
    f32, d1 = _drift(P, n, N, 9)
    b16, _ = _drift(P, n, N, 9, bf16_state=True)
    f16, _ = _drift(P, n, N, 9, state_fmt=oracle.STATE_F16)
    dec, _ = _drift(P, n, N, 9, decay=0.9)
    none, _ = _drift(P, n, N, 9, compensated=False)
    assert f32 <= 3.0 * d1
    assert b16 <= 2.0 * f32
    assert f16 <= 2.0 * f32
    assert 2.0 * f32 < dec < 0.5 * none


def test_f16_state_loses_tiny_errors_bf16_keeps():
    """fp16's range ends near 6e-5 (subnormals below, 2^-24 apart), bf16's
    does not: with inputs around 1e-6 the revealed errors are in fp16's
    subnormal range, so an fp16 state keeps them only coarsely and the drift
    grows well beyond the bf16 state's, though far below no feedback."""
    P, n, N = 2, 4096, 300
    b16, b1 = _drift(P, n, N, 9, scale=1e-6, bf16_state=True)
    f16, f1 = _drift(P, n, N, 9, scale=1e-6, state_fmt=oracle.STATE_F16)
    none, n1 = _drift(P, n, N, 9, scale=1e-6, compensated=False)
    assert f16 / f1 > 1.5 * (b16 / b1)
    assert f16 / f1 < 0.5 * (none / n1)
