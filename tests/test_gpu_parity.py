"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Small and mid sizes, compared element by element: outputs of every rank, the
compensator state, and every push and gather code and meta word.  Sizes span
several reduce tiles (32 groups each) with a ragged last tile (37 groups per
segment), P from 1 to 16, 4- and 8-bit codes, the three compensator modes and
both gather variants, over a sequence of calls that carries the state.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import STATE_DTYPES, assert_state_close, assert_wire_equal, bits, wire_to_canonical

pytestmark = pytest.mark.gpu

G = 128


@pytest.fixture(scope="module")
def echo():
    from bit_error_compensated_gb300 import echo as mod
    return mod


def _inputs(P, n, seed, scale=1.0):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    x = torch.randn((P, n), generator=gen, device="cuda") * scale
    # a per-element spread shared by the ranks, like the channel scales of a
    # TP partial sum
    spread = torch.exp(torch.randn(n, generator=gen, device="cuda"))
    return (x * spread).to(torch.bfloat16)


SCHEDULES = ["fused", "unfused", "persistent", "tile", "tile_rp"]
# the tile schedule's forms, forced (the default, ECHO_TILE_AUTO, picks one by size)
TILE_FORMS = {"tile": 2, "tile_rp": 3}


def _set_schedule(echo, plan, schedule):
    echo.echo_set_fused(plan, schedule != "unfused")
    echo.echo_set_persistent(plan, schedule == "persistent")
    echo.echo_set_tile_fused(plan, TILE_FORMS.get(schedule, 0))


def _run_sequence(echo, P, Gs, bits_, mode, fused, calls=3, seed=0, inplace=False, quant=0,
                  fmt=0, decay=1.0, g=G, persistent=False, tile=False):
    n = P * g * Gs
    plan = echo.echo_plan(P, n, g, bits_)
    echo.echo_set_fused(plan, fused)
    echo.echo_set_persistent(plan, persistent)
    echo.echo_set_tile_fused(plan, tile)
    echo.echo_set_quantizer(plan, quant)
    echo.echo_set_state(plan, fmt, decay)
    assert echo.echo_comp_bytes(plan) == P * n * (4 if fmt == 0 else 2)
    lay = echo.echo_wire_layout(plan)
    sdt = STATE_DTYPES[fmt]
    comp_t = torch.zeros((P, n), dtype=sdt, device="cuda") if mode == "caller" else None
    comp_arg = {"none": None, "default": echo.COMP_DEFAULT, "caller": comp_t}[mode]
    e_ref = None if mode == "none" else np.zeros((P, n), np.float32)
    for k in range(calls):
        x = _inputs(P, n, seed * 100 + k)
        xb = bits(x)
        out = x if inplace else torch.empty_like(x)
        echo.echo_allreduce(plan, list(x), list(out), comp_arg)
        torch.cuda.synchronize()
        assert echo.echo_get_status(plan) == 0
        ref = oracle.allreduce(xb, g, bits_, e=e_ref, want_wire=True, mode=quant,
                               state_fmt=fmt, decay=decay)
        got = bits(out)
        assert np.array_equal(got, ref["out"]), f"outputs differ at call {k}"
        wire = wire_to_canonical(echo.echo_debug_wire(plan), lay, P, n, bits_)
        assert_wire_equal(wire, ref, P)
        if mode == "caller":
            # a bf16 or fp16 state widens to fp32 exactly
            assert_state_close(comp_t.float().cpu().numpy(), e_ref, f"state after call {k}")
    return plan


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("mode", ["none", "default", "caller"])
@pytest.mark.parametrize("bits_", [4, 8])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
def test_matches_oracle(echo, P, bits_, mode, fused):
    _run_sequence(echo, P, 37, bits_, mode, fused, seed=P * 10 + bits_)


@pytest.mark.parametrize("quant", [1, 2])
@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("mode", ["none", "caller"])
@pytest.mark.parametrize("bits_", [4, 8])
@pytest.mark.parametrize("P", [1, 3, 4, 8])
def test_ablation_quantizers_match_oracle(echo, P, bits_, mode, fused, quant):
    """The two quantizers of the paper's Table 8 ablation ("naive zero-point",
    "symmetric grid"), selected with echo_set_quantizer."""
    _run_sequence(echo, P, 37, bits_, mode, fused, seed=500 + 10 * P + bits_, quant=quant)


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("state", [(1, 1.0), (0, 0.75), (1, 0.5), (2, 1.0), (2, 0.5)])
@pytest.mark.parametrize("bits_", [4, 8])
@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_state_options_match_oracle(echo, P, bits_, state, fused):
    """The compensator state kept in bf16 or fp16 and/or decayed (echo_set_state)."""
    fmt, decay = state
    _run_sequence(echo, P, 37, bits_, "caller", fused, calls=4, seed=700 + 10 * P + bits_,
                  fmt=fmt, decay=decay)


@pytest.mark.parametrize("quant", [1, 2])
def test_state_options_with_ablation_quantizers(echo, quant):
    _run_sequence(echo, 4, 37, 4, "caller", 0, seed=800 + quant, quant=quant,
                  fmt=quant, decay=0.9)   # bf16 state with the naive quantizer, fp16 with the symmetric


def test_state_format_switch(echo):
    """Changing the format zeroes the plan's own state; changing only the decay
    keeps it.  Checked through the outputs, which depend on the held state."""
    P, Gs = 4, 37
    n = P * G * Gs
    plan = echo.echo_plan(P, n, G, 4)
    e = np.zeros((P, n), np.float32)
    steps = [(0, 1.0), (0, 1.0), (1, 1.0), (1, 1.0), (1, 0.5), (2, 0.5), (2, 1.0),
             (0, 0.5), (0, 1.0)]
    prev = steps[0]
    for k, (fmt, decay) in enumerate(steps):
        echo.echo_set_state(plan, fmt, decay)
        if fmt != prev[0]:
            e[:] = 0
        prev = (fmt, decay)
        x = _inputs(P, n, 900 + k)
        out = torch.empty_like(x)
        echo.echo_allreduce(plan, list(x), list(out), echo.COMP_DEFAULT)
        torch.cuda.synchronize()
        ref = oracle.allreduce(bits(x), G, 4, e=e, state_fmt=fmt, decay=decay)
        assert np.array_equal(bits(out), ref["out"]), f"call {k}"


# Groups per owner segment that leave a ragged last reduce tile (64 groups of
# 64, 16 groups of 256), a ragged last push unit (8 groups of 64; 2 of 256)
# and, for 64, a ragged last gather run (4 groups).
GS_RAGGED = {64: 75, 256: 37}


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("mode", ["none", "caller"])
@pytest.mark.parametrize("bits_", [4, 8])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("g", [64, 256])
def test_group_sizes_match_oracle(echo, g, P, bits_, mode, fused):
    """Groups of 64 and 256 elements (the group-size rows of the paper's
    Table 8 ablation)."""
    _run_sequence(echo, P, GS_RAGGED[g], bits_, mode, fused, seed=1000 + g + 10 * P + bits_, g=g)


@pytest.mark.parametrize("opts", [dict(quant=1), dict(quant=2), dict(fmt=1), dict(fmt=2),
                                  dict(fmt=1, decay=0.5, quant=2), dict(fmt=2, decay=0.5, quant=1)])
@pytest.mark.parametrize("g", [64, 256])
def test_group_sizes_with_options(echo, g, opts):
    _run_sequence(echo, 4, GS_RAGGED[g], 4, "caller", 0, seed=1100 + g, g=g, **opts)


@pytest.mark.parametrize("g,Gs", [(64, 1), (64, 7), (64, 8), (64, 63), (64, 64), (64, 65),
                                  (64, 129), (256, 1), (256, 2), (256, 3), (256, 15), (256, 16),
                                  (256, 17), (256, 33)])
def test_group_size_tile_boundaries(echo, g, Gs):
    _run_sequence(echo, 4, Gs, 4, "caller", 0, calls=2, seed=Gs, g=g)


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("mode", ["none", "default", "caller"])
@pytest.mark.parametrize("bits_", [4, 8])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
def test_persistent_matches_oracle(echo, P, bits_, mode, fused):
    """The whole call as one persistent kernel (echo_set_persistent)."""
    _run_sequence(echo, P, 37, bits_, mode, fused, seed=2000 + P * 10 + bits_, persistent=True)


@pytest.mark.parametrize("opts", [dict(g=64), dict(g=256), dict(quant=1), dict(quant=2),
                                  dict(fmt=1, decay=0.5), dict(g=64, quant=2, fused=1),
                                  dict(g=256, fmt=1, fused=1), dict(fmt=2), dict(inplace=True),
                                  dict(inplace=True, fused=1)])
def test_persistent_with_options(echo, opts):
    opts = dict(opts)
    g = opts.pop("g", G)
    fused = opts.pop("fused", 0)
    _run_sequence(echo, 4, {64: 75, 128: 37, 256: 37}[g], 4, "caller", fused, seed=2100, g=g,
                  persistent=True, **opts)


@pytest.mark.parametrize("Gs", [1, 2, 31, 32, 33, 64, 129, 300])
def test_persistent_tile_boundaries(echo, Gs):
    _run_sequence(echo, 3, Gs, 4, "caller", 0, calls=2, seed=Gs, persistent=True)


@pytest.mark.parametrize("form", [2, 3], ids=["rank_loop", "rank_parallel"])
@pytest.mark.parametrize("mode", ["none", "default", "caller"])
@pytest.mark.parametrize("bits_", [4, 8])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
def test_tile_fused_matches_oracle(echo, P, bits_, mode, form):
    """The whole call as one kernel, a block per owner tile (echo_set_tile_fused),
    in each of its two forms."""
    _run_sequence(echo, P, 37, bits_, mode, 1, seed=2200 + P * 10 + bits_, tile=form)


@pytest.mark.parametrize("opts", [dict(g=64), dict(g=256), dict(quant=1), dict(quant=2),
                                  dict(fmt=1, decay=0.5), dict(fmt=2), dict(g=64, quant=2),
                                  dict(g=256, fmt=1), dict(inplace=True), dict(decay=0.75)])
@pytest.mark.parametrize("form", [2, 3], ids=["rank_loop", "rank_parallel"])
def test_tile_fused_with_options(echo, opts, form):
    opts = dict(opts)
    g = opts.pop("g", G)
    _run_sequence(echo, 4, {64: 75, 128: 37, 256: 37}[g], 4, "caller", 1, seed=2300, g=g,
                  tile=form, **opts)


@pytest.mark.parametrize("P,Gs", [(3, 1), (3, 7), (3, 8), (3, 9), (5, 15), (5, 16), (5, 17),
                                  (2, 300)])
@pytest.mark.parametrize("form", [2, 3], ids=["rank_loop", "rank_parallel"])
def test_tile_fused_tile_boundaries(echo, P, Gs, form):
    """Segments of a few groups up to several tiles, with short last tiles."""
    _run_sequence(echo, P, Gs, 4, "caller", 1, calls=2, seed=Gs, tile=form)


@pytest.mark.parametrize("P,Gs", [(8, 8), (8, 608), (8, 609), (4, 1216), (4, 1217), (2, 9)])
def test_tile_fused_automatic_form(echo, P, Gs):
    """The default picks the rank-parallel form for grids of at most four times
    the SMs and P >= 2, the rank loop otherwise; both sides of that bound (608
    blocks of 8 groups on a 152-SM GB300) match the oracle."""
    _run_sequence(echo, P, Gs, 4, "default", 1, calls=2, seed=Gs + P, tile=1)


def _fuzz_cases(count, seed):
    """Seeded random configurations of the call: ranks, segment length in
    groups (short, one tile, several tiles with a ragged end), code width,
    group size, quantizer, state format and decay, compensation mode, in-place
    outputs, and the schedule (the tile kernel's two forms weighted up)."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(count):
        P = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 11, 16]))
        g = int(rng.choice([64, 128, 256]))
        per_tile = 1024 // g
        Gs = int(rng.choice([1, per_tile - 1, per_tile, per_tile + 1, 3 * per_tile + 5,
                             int(rng.integers(1, 6 * per_tile))]))
        Gs = max(Gs, 1)
        fmt = int(rng.integers(0, 3))
        cases.append(dict(P=P, Gs=Gs, g=g, bits_=int(rng.choice([4, 8])),
                          quant=int(rng.integers(0, 3)), fmt=fmt,
                          decay=float(rng.choice([1.0, 1.0, 0.75])),
                          mode=str(rng.choice(["none", "default", "caller", "caller"])),
                          inplace=bool(rng.integers(0, 4) == 0),
                          schedule=str(rng.choice(["tile", "tile_rp", "tile", "tile_rp",
                                                   "fused", "unfused", "persistent",
                                                   "default"])),
                          seed=9000 + i))
    return cases


@pytest.mark.parametrize("case", _fuzz_cases(96, 20261203), ids=lambda c: (
    f"P{c['P']}-Gs{c['Gs']}-g{c['g']}-b{c['bits_']}-q{c['quant']}-s{c['fmt']}-"
    f"{c['mode']}-{c['schedule']}"))
def test_random_configurations_match_oracle(echo, case):
    """Random combinations of every option against the oracle, two calls each."""
    c = dict(case)
    schedule = c.pop("schedule")
    mode = c.pop("mode")
    P, Gs, bits_ = c.pop("P"), c.pop("Gs"), c.pop("bits_")
    tile = {"tile": 2, "tile_rp": 3, "default": 1}.get(schedule, 0)
    fused = 0 if schedule == "unfused" else 1
    _run_sequence(echo, P, Gs, bits_, mode, fused, calls=2, tile=tile,
                  persistent=schedule == "persistent", **c)


def test_every_schedule_gives_the_same_bits(echo):
    """Outputs, state and every wire byte of a call sequence agree between the
    schedules: one kernel a block per owner tile (the default, and each of its
    two forms forced), push and reduce, push, reduce and gather, and the
    persistent kernel."""
    P, Gs = 4, 70
    n = P * G * Gs
    res = []
    for schedule in ("default", "tile", "tile_rp", "fused", "unfused", "persistent"):
        plan = echo.echo_plan(P, n, G, 4)
        if schedule != "default":              # the default needs no call
            _set_schedule(echo, plan, schedule)
        comp = torch.zeros((P, n), device="cuda")
        outs = []
        for k in range(4):
            x = _inputs(P, n, 3000 + k)
            out = torch.empty_like(x)
            echo.echo_allreduce(plan, list(x), list(out), comp)
            outs.append(bits(out))
        torch.cuda.synchronize()
        res.append((outs, comp.cpu().numpy().view(np.uint32), echo.echo_debug_wire(plan)))
    for other in res[1:]:
        assert all(np.array_equal(a, b) for a, b in zip(res[0][0], other[0]))
        assert np.array_equal(res[0][1], other[1])
        assert res[0][2] == other[2]


def test_persistent_bounded_wait_reports_timeout(echo):
    """A push that never reports completion (the hold hook) makes the reduce
    of its tile wait until its 1 s bound: the call ends with ECHO_ERR_TIMEOUT
    instead of hanging, echo_get_status clears the schedule, and the next call
    is correct again."""
    import time
    P, Gs = 4, 37
    n = P * G * Gs
    plan = echo.echo_plan(P, n, G, 4)
    echo.echo_set_persistent(plan, True)
    x = _inputs(P, n, 77)
    out = torch.empty_like(x)
    echo.echo_debug_hold_push(plan, 5)
    t0 = time.monotonic()
    echo.echo_allreduce(plan, list(x), list(out), None)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert echo.echo_get_status(plan) == echo.ECHO_ERR_TIMEOUT
    assert 0.5 < waited < 10.0
    echo.echo_debug_hold_push(plan, -1)
    for k in range(2):
        xk = _inputs(P, n, 78 + k)
        echo.echo_allreduce(plan, list(xk), list(out), None)
        torch.cuda.synchronize()
        assert echo.echo_get_status(plan) == 0
        assert np.array_equal(bits(out), oracle.allreduce(bits(xk), G, 4)["out"])


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_calls_captured_in_a_cuda_graph(echo, schedule):
    """A sequence of calls captured once by stream capture and replayed: every
    replay continues the state, and outputs match the oracle's calls."""
    P, Gs = 4, 37
    n = P * G * Gs
    plan = echo.echo_plan(P, n, G, 4)
    _set_schedule(echo, plan, schedule)
    xs = [_inputs(P, n, 4000 + k) for k in range(3)]
    outs = [torch.empty_like(x) for x in xs]
    echo.echo_allreduce(plan, list(xs[0]), list(outs[0]), None)      # first use outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        for x, out in zip(xs, outs):
            echo.echo_allreduce(plan, list(x), list(out), echo.COMP_DEFAULT, side)
    e = np.zeros((P, n), np.float32)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        for x, out in zip(xs, outs):
            ref = oracle.allreduce(bits(x), G, 4, e=e)
            assert np.array_equal(bits(out), ref["out"])
    assert echo.echo_get_status(plan) == 0


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("fmt", [0, 1, None])          # fp32 state, bf16 state, none
def test_any_grid_size_gives_the_same_bits(echo, schedule, fmt):
    """The kernels stride over their work, so a 1-, 3- or 7-block grid must give
    the same outputs, state and codes as the launchers' own grid (where a push
    warp takes one unit with fp32 state and up to four, two in flight, with a
    2-byte state or none)."""
    P, Gs = 4, 70
    n = P * G * Gs
    res = []
    for cap in (0, 1, 3, 7):
        plan = echo.echo_plan(P, n, G, 4)
        _set_schedule(echo, plan, schedule)
        echo.echo_debug_set_grid(plan, cap)
        comp = None
        if fmt is not None:
            echo.echo_set_state(plan, fmt, 1.0)
            comp = torch.zeros((P, n), dtype=STATE_DTYPES[fmt], device="cuda")
        outs = []
        for k in range(3):
            x = _inputs(P, n, 5000 + k)
            out = torch.empty_like(x)
            echo.echo_allreduce(plan, list(x), list(out), comp)
            outs.append(bits(out))
        torch.cuda.synchronize()
        state = None if comp is None else comp.cpu().view(torch.uint8).numpy()
        res.append((outs, state, echo.echo_debug_wire(plan)))
    for other in res[1:]:
        assert all(np.array_equal(a, b) for a, b in zip(res[0][0], other[0]))
        assert (res[0][1] is None) == (other[1] is None)
        assert res[0][1] is None or np.array_equal(res[0][1], other[1])
        assert res[0][2] == other[2]


@pytest.mark.parametrize("case", [(1, 128, 4, 5), (2, 64, 8, 9), (3, 256, 4, 7), (4, 128, 8, 37),
                                  (8, 64, 4, 75), (16, 256, 8, 3), (5, 128, 4, 33)])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_guard_bands_stay_intact(echo, case, schedule):
    """Nothing is written outside the receive slots or the plan's state: the
    guard bands around both still hold their fill after calls of ragged shapes
    in every state format."""
    P, g, bits_, Gs = case
    n = P * g * Gs
    plan = echo.echo_plan(P, n, g, bits_)
    _set_schedule(echo, plan, schedule)
    for fmt in (0, 1, 2):
        echo.echo_set_state(plan, fmt, 0.5 if fmt else 1.0)
        for k in range(2):
            x = _inputs(P, n, 6000 + k)
            echo.echo_allreduce(plan, list(x), list(torch.empty_like(x)), echo.COMP_DEFAULT)
    torch.cuda.synchronize()
    assert echo.echo_debug_check_guards(plan)


@pytest.mark.parametrize("Gs", [1, 4, 7, 8, 9, 31, 32, 33, 64, 129])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("fused", [0, 1])
def test_tile_boundaries(echo, Gs, fmt, fused):
    """Segments of one group up to past several reduce tiles (8 groups of 128)
    and push blocks (8 groups with fp32 state, 16 with a 2-byte state), ending
    on and beside their edges."""
    _run_sequence(echo, 4, Gs, 4, "caller", fused, calls=2, seed=Gs, fmt=fmt)


@pytest.mark.parametrize("fused", [0, 1])
def test_in_place(echo, fused):
    _run_sequence(echo, 4, 40, 4, "caller", fused, calls=3, seed=7, inplace=True)


def test_fused_and_unfused_identical(echo):
    P, Gs, n = 4, 50, 4 * G * 50
    outs = []
    for fused in (0, 1):
        plan = echo.echo_plan(P, n, G, 4)
        echo.echo_set_fused(plan, fused)
        comp = torch.zeros((P, n), device="cuda")
        o = []
        for k in range(4):
            x = _inputs(P, n, 900 + k)
            out = torch.empty_like(x)
            echo.echo_allreduce(plan, list(x), list(out), comp)
            o.append(bits(out))
        outs.append((o, comp.cpu().numpy(), echo.echo_debug_wire(plan)))
    assert all(np.array_equal(a, b) for a, b in zip(outs[0][0], outs[1][0]))
    assert np.array_equal(outs[0][1].view(np.uint32), outs[1][1].view(np.uint32))
    assert outs[0][2] == outs[1][2]


def test_deterministic_run_twice(echo):
    P, n = 8, 8 * G * 45
    res = []
    for _ in range(2):
        plan = echo.echo_plan(P, n, G, 4)
        comp = torch.zeros((P, n), device="cuda")
        for k in range(3):
            x = _inputs(P, n, 50 + k)
            out = torch.empty_like(x)
            echo.echo_allreduce(plan, list(x), list(out), comp)
        res.append((bits(out), comp.cpu().numpy().view(np.uint32), echo.echo_debug_wire(plan)))
    assert np.array_equal(res[0][0], res[1][0])
    assert np.array_equal(res[0][1], res[1][1])
    assert res[0][2] == res[1][2]


def test_all_outputs_identical_across_ranks(echo):
    P, n = 8, 8 * G * 33
    plan = echo.echo_plan(P, n, G, 4)
    x = _inputs(P, n, 3)
    out = torch.empty_like(x)
    echo.echo_allreduce(plan, list(x), list(out), echo.COMP_DEFAULT)
    o = bits(out)
    assert all(np.array_equal(o[p], o[0]) for p in range(P))


def test_reset_and_resume(echo):
    """Checkpoint/resume of the only cross-call state: K calls, save the state,
    M more calls; then restore and replay the M calls -- bitwise equal."""
    P, n = 4, 4 * G * 34
    plan = echo.echo_plan(P, n, G, 4)
    comp = torch.zeros((P, n), device="cuda")
    for k in range(3):
        x = _inputs(P, n, 200 + k)
        echo.echo_allreduce(plan, list(x), list(torch.empty_like(x)), comp)
    saved = comp.clone()
    outs_a = []
    for k in range(3, 6):
        x = _inputs(P, n, 200 + k)
        out = torch.empty_like(x)
        echo.echo_allreduce(plan, list(x), list(out), comp)
        outs_a.append(bits(out))
    state_a = comp.clone()
    comp.copy_(saved)
    for i, k in enumerate(range(3, 6)):
        x = _inputs(P, n, 200 + k)
        out = torch.empty_like(x)
        echo.echo_allreduce(plan, list(x), list(out), comp)
        assert np.array_equal(bits(out), outs_a[i])
    assert torch.equal(comp.view(torch.int32), state_a.view(torch.int32))
    # reset: the plan's own state back to zero gives a fresh start
    echo.echo_allreduce(plan, list(x), list(torch.empty_like(x)), echo.COMP_DEFAULT)
    echo.echo_reset_comp(plan)
    out1 = torch.empty_like(x)
    echo.echo_allreduce(plan, list(x), list(out1), echo.COMP_DEFAULT)
    out2 = torch.empty_like(x)
    echo.echo_allreduce(plan, list(x), list(out2), torch.zeros((P, n), device="cuda"))
    assert torch.equal(out1, out2)
    comp.zero_()
    echo.echo_reset_comp_async(plan, comp)
    assert not comp.any()


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_overflow_flag(echo, schedule):
    P, n = 2, 2 * G * 4
    plan = echo.echo_plan(P, n, G, 4)
    _set_schedule(echo, plan, schedule)
    x = _inputs(P, n, 1)
    x[1, 300] = float("inf")
    echo.echo_allreduce(plan, list(x), list(torch.empty_like(x)), None)
    assert echo.echo_get_status(plan) == echo.ECHO_ERR_OVERFLOW
    assert echo.echo_get_status(plan) == 0          # read-and-clear
    x = _inputs(P, n, 1) * 1e6                       # step beyond fp16
    x = x.to(torch.bfloat16)
    echo.echo_allreduce(plan, list(x), list(torch.empty_like(x)), None)
    assert echo.echo_get_status(plan) == echo.ECHO_ERR_OVERFLOW
    assert oracle.allreduce(bits(x), G, 4)["flagged"] > 0


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_empty_and_degenerate(echo, schedule):
    plan = echo.echo_plan(4, 0, G, 4)
    _set_schedule(echo, plan, schedule)
    e = torch.empty((4, 0), dtype=torch.bfloat16, device="cuda")
    ptrs = [torch.empty(8, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    echo.echo_allreduce(plan, ptrs, [torch.empty(8, dtype=torch.bfloat16, device="cuda")
                                     for _ in range(4)], echo.COMP_DEFAULT)
    assert echo.echo_comp_bytes(plan) == 0 and e.numel() == 0
    # all-zero input: step 1, zero point 0, outputs exactly zero
    P, n = 4, 4 * G * 3
    plan = echo.echo_plan(P, n, G, 4)
    _set_schedule(echo, plan, schedule)
    x = torch.zeros((P, n), dtype=torch.bfloat16, device="cuda")
    out = torch.ones_like(x)
    echo.echo_allreduce(plan, list(x), list(out), echo.COMP_DEFAULT)
    assert not out.any()


def test_argument_errors(echo):
    P, n = 2, 2 * G * 2
    plan = echo.echo_plan(P, n, G, 4)
    x = torch.zeros((P, n + 8), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((P, n + 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(echo.EchoError) as ei:          # misaligned by 2 bytes
        echo.echo_allreduce(plan, [x[0, 1:], x[1]], [out[0], out[1]], None)
    assert ei.value.status == echo.ECHO_ERR_ALIGN
    # a compensator state must be 32-byte aligned: 16 bytes off is rejected
    state = torch.zeros(P * n + 8, dtype=torch.float32, device="cuda")
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_allreduce(plan, [x[0, :n], x[1, :n]], [out[0, :n], out[1, :n]], state[4:])
    assert ei.value.status == echo.ECHO_ERR_ALIGN
    echo.echo_allreduce(plan, [x[0, :n], x[1, :n]], [out[0, :n], out[1, :n]], state[8:])
    torch.cuda.synchronize()
    with pytest.raises(echo.EchoError) as ei:          # out[0] overlaps in[1]
        echo.echo_allreduce(plan, [x[0], x[1]], [x[1], out[1]], None)
    assert ei.value.status == echo.ECHO_ERR_ARG
    with pytest.raises(echo.EchoError) as ei:          # two outputs overlap
        echo.echo_allreduce(plan, [x[0], x[1]], [out[0], out[0]], None)
    assert ei.value.status == echo.ECHO_ERR_ARG
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_plan(3, 3 * G * 2 + 1, G, 4)
    assert ei.value.status == echo.ECHO_ERR_SHAPE
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_plan(2, 2 * G, G, 6)
    assert ei.value.status == echo.ECHO_ERR_UNSUPPORTED
    for g in (32, 96, 512):                             # group sizes the GPU does not take
        with pytest.raises(echo.EchoError) as ei:
            echo.echo_plan(2, 2 * 512 * 3, g, 4)
        assert ei.value.status == echo.ECHO_ERR_UNSUPPORTED
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_set_quantizer(plan, 3)
    assert ei.value.status == echo.ECHO_ERR_ARG
    for fmt, decay in [(3, 1.0), (-1, 1.0), (0, 0.0), (0, -0.5), (1, 1.5), (0, float("nan")),
                       (0, float("inf"))]:
        with pytest.raises(echo.EchoError) as ei:
            echo.echo_set_state(plan, fmt, decay)
        assert ei.value.status == echo.ECHO_ERR_ARG
    assert echo.echo_comp_bytes(plan) == plan.P * plan.n * 4       # unchanged
    for bad in (2, -1):                                 # the C call takes 0 or 1 only
        assert echo._lib.echo_set_persistent(plan, bad) == echo.ECHO_ERR_ARG
    for bad in (4, -1):                                 # ECHO_TILE_OFF .. RANK_PARALLEL
        assert echo._lib.echo_set_tile_fused(plan, bad) == echo.ECHO_ERR_ARG
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_debug_hold_push(plan, -2)
    assert ei.value.status == echo.ECHO_ERR_ARG
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_debug_set_grid(plan, -1)
    assert ei.value.status == echo.ECHO_ERR_ARG


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("bits_", [4, 8])
def test_exact_and_near_rounding_ties(echo, bits_, schedule):
    """Inputs on a half-step grid make v/s land exactly on half-integers (ties
    to even) or, with a tiny held error added, within 2^-10..2^-22 of them --
    the cases where the kernels' reciprocal fast path must defer to the exact
    quotient.  Outputs, state and codes must still equal the oracle's."""
    P, Gs = 2, 64
    n = P * G * Gs
    L = (1 << bits_) - 1
    rng = np.random.default_rng(bits_)
    s = 0.125                                     # the step every group gets
    i = rng.integers(0, min(2 * L, 255) + 1, (P, n)).astype(np.float64)
    vals = i * (s / 2)
    vals[:, ::G] = L * s                          # each group's maximum: range [0, L*s]
    x = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(x.float().numpy(), vals.astype(np.float32))   # exact in bf16
    near = rng.random((P, n)) < 0.5
    delta = (2.0 ** -rng.integers(10, 23, (P, n))) * s
    e0 = np.where(near & (vals < L * s), delta, 0.0).astype(np.float32)
    x = x.cuda()
    comp = torch.from_numpy(e0.copy()).cuda()
    plan = echo.echo_plan(P, n, G, bits_)
    _set_schedule(echo, plan, schedule)
    lay = echo.echo_wire_layout(plan)
    out = torch.empty_like(x)
    echo.echo_allreduce(plan, list(x), list(out), comp)
    e_ref = e0.copy()
    ref = oracle.allreduce(bits(x), G, bits_, e=e_ref, want_wire=True)
    assert ref["ties"] > 100                      # the grid does produce exact ties
    assert np.array_equal(bits(out), ref["out"])
    assert_wire_equal(wire_to_canonical(echo.echo_debug_wire(plan), lay, P, n, bits_), ref, P)
    assert_state_close(comp.cpu().numpy(), e_ref)


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("P", [2, 4])
@pytest.mark.parametrize("bits_", [4, 8])
def test_tie_count_by_construction(echo, bits_, P, schedule):
    """Inputs whose number of exact rounding ties is fixed by construction
    (tests/test_oracle_ties.py): half-step grids at stage 1 in some groups and
    at stage 2 in others, zero-point ties, and near ties within 2^-10..2^-22 of
    a step.  The values ride in the caller's fp32 state over bf16 zeros, so
    v = x + e is exact.  The oracle must count exactly the constructed ties,
    and the GPU must produce the same codes, outputs and state on them."""
    from test_oracle_ties import _whole_call_values
    Gs = 36                                      # more than one reduce tile, ragged
    n = P * G * Gs
    rng = np.random.default_rng(60 + 10 * P + bits_)
    e0, expected = _whole_call_values(rng, P, bits_, G, Gs, 0.25)
    x = torch.zeros((P, n), dtype=torch.bfloat16, device="cuda")
    comp = torch.from_numpy(e0.copy()).cuda()
    plan = echo.echo_plan(P, n, G, bits_)
    _set_schedule(echo, plan, schedule)
    lay = echo.echo_wire_layout(plan)
    out = torch.empty_like(x)
    echo.echo_allreduce(plan, list(x), list(out), comp)
    torch.cuda.synchronize()
    assert echo.echo_get_status(plan) == 0
    e_ref = e0.copy()
    ref = oracle.allreduce(bits(x), G, bits_, e=e_ref, want_wire=True)
    assert ref["ties"] == expected
    assert np.array_equal(bits(out), ref["out"])
    assert_wire_equal(wire_to_canonical(echo.echo_debug_wire(plan), lay, P, n, bits_), ref, P)
    assert_state_close(comp.cpu().numpy(), e_ref)


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_subnormal_inputs_and_state(echo, fmt, schedule):
    """The entry pass, the quantizers and the state update keep subnormal
    numbers exactly as the oracle's IEEE fp32 arithmetic does (no flush to
    zero): bf16 inputs and held errors that are subnormal, values that cancel
    exactly (x + e = +0), and groups whose whole range is subnormal, over three
    compensated calls, against the oracle bit for bit."""
    P, Gs = 2, 40
    n = P * G * Gs
    rng = np.random.default_rng(90 + fmt)
    tiny = np.float32(2.0 ** -130)                     # fp32 subnormal
    x32 = (rng.standard_normal((P, n)) * 2.0 ** -128).astype(np.float32)   # bf16 subnormals
    x32[:, ::3] = rng.standard_normal((P, -(-n // 3))).astype(np.float32)  # mixed with normals
    groups = x32.reshape(P, -1, G)
    groups[:, ::4] = (rng.standard_normal((P, groups[:, ::4].shape[1], G)) * 2.0 ** -132
                      ).astype(np.float32)             # all-subnormal groups
    x = torch.from_numpy(x32).to(torch.bfloat16)
    xf = x.float().numpy()
    e0 = (rng.standard_normal((P, n)) * tiny).astype(np.float32)
    cancel = rng.random((P, n)) < 0.1
    e0[cancel] = -xf[cancel]                           # x + e = +0 exactly
    if fmt != 0:                                       # a 2-byte state holds only its own values
        e0 = torch.from_numpy(e0).to(STATE_DTYPES[fmt]).float().numpy()
        assert (np.abs(e0[e0 != 0]) < 2.0 ** -126).any() or fmt == 2
    plan = echo.echo_plan(P, n, G, 4)
    _set_schedule(echo, plan, schedule)
    echo.echo_set_state(plan, fmt, 1.0)
    comp = torch.from_numpy(e0).to(STATE_DTYPES[fmt]).cuda()
    e_ref = e0.copy()
    x = x.cuda()
    for k in range(3):
        xk = x if k == 0 else torch.roll(x, k, dims=1)
        out = torch.empty_like(xk)
        echo.echo_allreduce(plan, list(xk), list(out), comp)
        torch.cuda.synchronize()
        assert echo.echo_get_status(plan) == 0
        ref = oracle.allreduce(bits(xk), G, 4, e=e_ref, state_fmt=fmt)
        assert np.array_equal(bits(out), ref["out"]), f"outputs differ at call {k}"
        assert_state_close(comp.float().cpu().numpy(), e_ref, f"state after call {k}")


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_prepared_call_matches_oracle(echo, schedule):
    """echo.prepare_allreduce marshals the buffers once; calling it three times
    on inputs rewritten in place between calls gives the oracle's results
    (outputs bit for bit, the carried state within STATE_RTOL)."""
    P, Gs = 4, 37
    n = P * G * Gs
    plan = echo.echo_plan(P, n, G, 4)
    _set_schedule(echo, plan, schedule)
    x = torch.empty((P, n), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    comp = torch.zeros((P, n), device="cuda")
    call = echo.prepare_allreduce(plan, list(x), list(out), comp)
    e_ref = np.zeros((P, n), np.float32)
    for k in range(3):
        x.copy_(_inputs(P, n, 300 + k))              # new inputs, same buffers
        call()
        torch.cuda.synchronize()
        ref = oracle.allreduce(bits(x), G, 4, e=e_ref)
        assert np.array_equal(bits(out), ref["out"]), f"outputs differ at call {k}"
        assert_state_close(comp.cpu().numpy(), e_ref, f"state after call {k}")
    assert echo.echo_get_status(plan) == 0
