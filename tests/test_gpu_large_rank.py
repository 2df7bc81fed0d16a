"""A rank tensor longer than 2^31 elements: every element offset, state offset
and receive-slot offset needs 64-bit arithmetic past that point.  P = 2 ranks
of n = 2^31 + 2*128*64 bf16 elements (4 GiB each; about 36 GB on the device
with the outputs, the plan's fp32 state and its receive slots), two
compensated calls, for each schedule; compared with the oracle on sampled
group positions that include every group past element 2^31 of a rank, the
groups around that boundary and the first and last group of each segment
(positions are independent, so the oracle on them is exactly its whole call
restricted to them)."""
import numpy as np
import pytest
import torch

from _parity import SampledOracle, assert_state_close, assert_wire_equal, bits, sampled_wire

pytestmark = pytest.mark.gpu
G = 128
P = 2
N = 2 ** 31 + P * G * 64


@pytest.fixture(scope="module")
def big_inputs():
    x = torch.empty((P, N), dtype=torch.bfloat16, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(31)
    for p in range(P):
        x[p] = torch.randn(N, generator=gen, device="cuda").to(torch.bfloat16)
    yield x
    del x
    torch.cuda.empty_cache()


def _sample(Gs):
    first_past = 2 ** 31 // G                    # first global group past element 2^31
    groups = set(range(first_past - 8, P * Gs))  # the boundary and everything past it
    for o in range(P):
        groups.update(range(o * Gs, o * Gs + 4))
        groups.update(range(o * Gs + Gs - 4, o * Gs + Gs))
    rng = np.random.default_rng(31)
    groups.update(int(v) for v in rng.choice(P * Gs, size=1024, replace=False))
    return np.array(sorted(groups), np.int64)


@pytest.mark.parametrize("schedule", ["fused", "unfused", "persistent", "tile", "tile_rp"])
def test_rank_longer_than_2_31_elements(big_inputs, schedule):
    from bit_error_compensated_gb300 import echo
    x = big_inputs
    Gs = N // P // G
    groups = _sample(Gs)
    assert (groups * G >= 2 ** 31).sum() >= 64
    so = SampledOracle(P, Gs, groups, 4)
    xs = bits(so.gather(x))
    plan = echo.echo_plan(P, N, G, 4)
    echo.echo_set_fused(plan, schedule != "unfused")
    echo.echo_set_persistent(plan, schedule == "persistent")
    echo.echo_set_tile_fused(plan, {"tile": 2, "tile_rp": 3}.get(schedule, 0))
    lay = echo.echo_wire_layout(plan)
    out = torch.empty_like(x)
    for k in range(2):
        echo.echo_allreduce(plan, list(x), list(out), echo.COMP_DEFAULT)
        torch.cuda.synchronize()
        assert echo.echo_get_status(plan) == 0
        ref = so.call(xs, "fwd", want_wire=True)
        got = bits(so.gather(out))
        for r in range(P):
            assert np.array_equal(got[r], ref["y_rows"]), f"rank {r} outputs, call {k}"
        assert_wire_equal(sampled_wire(echo.echo_debug_wire(plan), lay, P, groups, 4), ref, P)
    # the plan's own state, read back through a caller-visible copy of the call:
    # one more call with a caller state started from the oracle's carried state
    comp = torch.zeros((P, N), device="cuda")
    idx = torch.from_numpy(so.idx).cuda()
    comp[:, idx] = torch.from_numpy(so.state_rows("fwd")).cuda()
    echo.echo_allreduce(plan, list(x), list(out), comp)
    torch.cuda.synchronize()
    ref = so.call(xs, "fwd")
    assert np.array_equal(bits(so.gather(out))[0], ref["y_rows"])
    assert_state_close(so.gather(comp).numpy(), so.state_rows("fwd"), "state past 2^31")
    del plan, comp, out
    torch.cuda.empty_cache()
