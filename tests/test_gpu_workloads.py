"""The five workloads at their full sizes, in the launch configuration the bench
times, checked against the oracle over their whole call sequences.

p2_n4096, p4_2048x4096 and p4_8192x4096 are compared in full: every output of
every rank, the whole compensator state and the wire codes.  p8_1gib and
p4_32768x1024 are compared on a fixed 1/64 sample of group positions carried
through every call (positions are independent, so the oracle on a sample is
exactly the oracle's whole call restricted to it); every sample includes the
first and last group of every owner segment.  Shorter runs check the options
(quantizers, state formats, group sizes, the persistent kernel) at full size.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import (STATE_DTYPES, SampledOracle, assert_state_close, assert_wire_equal, bits,
                     sample_groups, sampled_wire, wire_to_canonical)
from bit_error_compensated_gb300.workloads import WORKLOADS, call_sequence, rank_inputs

pytestmark = pytest.mark.gpu
G = 128


@pytest.fixture(scope="module")
def echo():
    from bit_error_compensated_gb300 import echo as mod
    return mod


def test_p2_n4096_full(echo):
    w = WORKLOADS[1]
    plan = echo.echo_plan(w.P, w.n, G, 4)
    lay = echo.echo_wire_layout(plan)
    comp = torch.zeros((w.P, w.n), device="cuda")
    e_ref = np.zeros((w.P, w.n), np.float32)
    ties = 0
    for c in call_sequence(1):
        x = rank_inputs(1, c, "cuda")
        out = torch.empty_like(x)
        compensated = c.state != "none"
        echo.echo_allreduce(plan, list(x), list(out), comp if compensated else None)
        ref = oracle.allreduce(bits(x), G, 4, e=e_ref if compensated else None, want_wire=True)
        ties += ref["ties"]
        assert np.array_equal(bits(out), ref["out"])
        assert_wire_equal(wire_to_canonical(echo.echo_debug_wire(plan), lay, w.P, w.n, 4), ref, w.P)
        assert_state_close(comp.cpu().numpy(), e_ref)
    print(f"p2_n4096: exact rounding ties in the oracle: {ties}; code mismatches: 0")


def _full_sequence(echo, number, bits_, wire_every=1):
    """Every call of workload `number` compared in full with the oracle."""
    w = WORKLOADS[number]
    P, n = w.P, w.n
    plan = echo.echo_plan(P, n, G, bits_)
    lay = echo.echo_wire_layout(plan)
    states, refs = {}, {}
    x = torch.empty((P, n), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    seq = call_sequence(number)
    ties = 0
    for k, c in enumerate(seq):
        rank_inputs(number, c, "cuda", out=x)
        comp = None
        if c.state != "none":
            comp = states.setdefault(c.state, torch.zeros((P, n), device="cuda"))
            refs.setdefault(c.state, np.zeros((P, n), np.float32))
        echo.echo_allreduce(plan, list(x), list(out), comp)
        check_wire = k % wire_every == 0 or k == len(seq) - 1
        ref = oracle.allreduce(bits(x), G, bits_, e=refs.get(c.state), want_wire=check_wire)
        ties += ref["ties"]
        assert np.array_equal(bits(out), ref["out"]), f"outputs, call {k}"
        if comp is not None:
            assert_state_close(comp.cpu().numpy(), refs[c.state], f"state, call {k}")
        if check_wire:
            assert_wire_equal(wire_to_canonical(echo.echo_debug_wire(plan), lay, P, n, bits_), ref, P)
    print(f"{w.name} ({bits_}-bit): {len(seq)} calls compared in full; exact rounding ties in "
          f"the oracle: {ties}; mismatches: 0")


def _sampled_sequence(echo, number, bits_, sample, calls=None, wire_calls=(0,), quant=0,
                      fmt=0, decay=1.0, g=G, persistent=False, fused=True, tile=1):
    """The workload's calls compared with the oracle on sampled group positions.
    The schedule defaults to the library's (tile kernel, form chosen by size);
    tile=0 with fused True/False gives the two- and three-kernel schedules."""
    w = WORKLOADS[number]
    P, n = w.P, w.n
    plan = echo.echo_plan(P, n, g, bits_)
    echo.echo_set_persistent(plan, persistent)
    echo.echo_set_tile_fused(plan, tile)
    echo.echo_set_fused(plan, fused)
    echo.echo_set_quantizer(plan, quant)
    echo.echo_set_state(plan, fmt, decay)
    sdt = STATE_DTYPES[fmt]
    lay = echo.echo_wire_layout(plan)
    Gs = lay["Gs"]
    groups = sample_groups(P, Gs, sample, seed=number)
    so = SampledOracle(P, Gs, groups, bits_, g=g, mode=quant, state_fmt=fmt, decay=decay)
    states = {}
    x = torch.empty((P, n), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    seq = call_sequence(number)
    if calls is not None:
        seq = seq[:calls]
    ties = 0
    for k, c in enumerate(seq):
        rank_inputs(number, c, "cuda", out=x)
        comp = None
        if c.state != "none":
            comp = states.setdefault(c.state, torch.zeros((P, n), dtype=sdt, device="cuda"))
        echo.echo_allreduce(plan, list(x), list(out), comp)
        xs = bits(so.gather(x))
        check_wire = k in wire_calls or k == len(seq) - 1
        ref = so.call(xs, c.state if comp is not None else None, want_wire=check_wire)
        ties += ref["ties"]
        got = bits(so.gather(out))
        for p in range(P):
            assert np.array_equal(got[p], ref["y_rows"]), f"call {k} rank {p}"
        if comp is not None:
            assert_state_close(so.gather(comp).float().numpy(), so.state_rows(c.state),
                               f"state call {k}")
        if check_wire:
            wire = sampled_wire(echo.echo_debug_wire(plan), lay, P, groups, bits_)
            for p in range(P):
                mask = so.owners != p
                assert np.array_equal(wire["q1"][mask, p], ref["q1"][mask, p]), f"push codes, call {k}"
                assert np.array_equal(wire["m1"][mask, p], ref["m1"][mask, p]), f"push meta, call {k}"
            assert np.array_equal(wire["q2"], ref["q2"]), f"gather codes, call {k}"
            assert np.array_equal(wire["m2"], ref["m2"]), f"gather meta, call {k}"
    print(f"workload {number} ({bits_}-bit): {len(seq)} calls, {groups.size} sampled positions, "
          f"exact rounding ties in the oracle: {ties}; code mismatches: 0")


def test_p4_2048x4096_full(echo):
    _full_sequence(echo, 2, 4)


@pytest.mark.parametrize("bits_", [4, 8])
def test_p8_1gib_sampled(echo, bits_):
    """The default schedule, as the bench times it, on 1/64 of the positions."""
    w = WORKLOADS[3]
    _sampled_sequence(echo, 3, bits_, sample=w.n // G // 64)


@pytest.mark.parametrize("fused", [True, False], ids=["two_kernels", "three_kernels"])
def test_p8_1gib_kernel_schedules_sampled(echo, fused):
    """Push and reduce (fused gather), or push, reduce and gather, at 1 GiB per rank."""
    _sampled_sequence(echo, 3, 4, sample=2048, calls=1, tile=0, fused=fused)


def test_p4_8192x4096_full(echo):
    _full_sequence(echo, 4, 4, wire_every=8)


def test_p4_32768x1024_sampled(echo):
    """All 1 120 calls (10 steps of 56 forward and 56 backward sites, two
    states) on 1/64 of the positions."""
    w = WORKLOADS[5]
    _sampled_sequence(echo, 5, 4, sample=w.n // G // 64)


@pytest.mark.parametrize("quant", [1, 2])
def test_p4_2048x4096_ablation_quantizers_sampled(echo, quant):
    """The Table 8 ablation quantizers over the first 16 calls of the 64-call
    workload, at full size."""
    _sampled_sequence(echo, 2, 4, sample=512, calls=16, quant=quant)


@pytest.mark.parametrize("state", [(1, 1.0), (0, 0.9), (1, 0.9), (2, 1.0)])
def test_p4_2048x4096_state_options_sampled(echo, state):
    """The compensator state in bf16 or fp16 and/or decayed, over the first 16
    calls of the 64-call workload, at full size."""
    _sampled_sequence(echo, 2, 4, sample=512, calls=16, fmt=state[0], decay=state[1])


def test_p8_1gib_bf16_state_sampled(echo):
    _sampled_sequence(echo, 3, 4, sample=2048, calls=4, fmt=1)


@pytest.mark.parametrize("g", [64, 256])
def test_p4_2048x4096_group_sizes_sampled(echo, g):
    """Groups of 64 and 256 over the first 16 calls of the 64-call workload."""
    _sampled_sequence(echo, 2, 4, sample=512 * 128 // g, calls=16, g=g)


@pytest.mark.parametrize("fused", [False, True])
def test_p4_2048x4096_persistent_sampled(echo, fused):
    """The persistent kernel over the first 16 calls of the 64-call workload."""
    _sampled_sequence(echo, 2, 4, sample=512, calls=16, persistent=True, fused=fused)


def test_p8_1gib_persistent_sampled(echo):
    _sampled_sequence(echo, 3, 4, sample=2048, calls=1, persistent=True)


def test_p4_32768x1024_persistent_sampled(echo):
    """Two states (forward and backward sites) through the persistent kernel."""
    _sampled_sequence(echo, 5, 4, sample=256, calls=24, persistent=True)


def test_p8_1gib_tile_rank_parallel_sampled(echo):
    """The tile kernel's rank-parallel form (which the default takes only for
    small grids) at 1 GiB per rank, 4- and 8-bit codes."""
    _sampled_sequence(echo, 3, 4, sample=2048, calls=1, tile=3)
    _sampled_sequence(echo, 3, 8, sample=2048, calls=1, tile=3)


def test_p4_32768x1024_tile_rank_parallel_sampled(echo):
    """Two states (forward and backward sites) through the rank-parallel form."""
    _sampled_sequence(echo, 5, 4, sample=1024, calls=224, tile=3)


@pytest.mark.parametrize("form", [2, 3], ids=["rank_loop", "rank_parallel"])
def test_p4_2048x4096_tile_forms_sampled(echo, form):
    _sampled_sequence(echo, 2, 4, sample=512, calls=16, tile=form)


@pytest.mark.parametrize("fused", [True, False], ids=["two_kernels", "three_kernels"])
def test_p4_2048x4096_kernel_schedules_sampled(echo, fused):
    """The two- and three-kernel schedules over the first 16 calls, with bf16 state."""
    _sampled_sequence(echo, 2, 4, sample=512, calls=16, tile=0, fused=fused, fmt=1)
