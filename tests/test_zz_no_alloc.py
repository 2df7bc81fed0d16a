"""echo_allreduce_noalloc, the entry point for callers that cannot allocate
device memory (for example code hosted by a runtime that owns the memory
budget and forbids allocation on its execution path).  Its receive slots live
in the library's fixed device array instead of a plan's cudaMalloc'd
workspace; its results must equal echo_allreduce's.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh
process.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import STATE_RTOL, assert_state_close, bits

pytestmark = pytest.mark.gpu
G = 128
SCRATCH = 32 << 20                       # ECHO_NOALLOC_SCRATCH_BYTES


def _r256(x):
    return (x + 255) // 256 * 256


def _slot_bytes(P, Gs, bits_):
    """Bytes the call needs in the fixed array: a 256-byte status word, then the
    receive slots in the layout echo_wire_layout describes, each section
    rounded up to 256 bytes."""
    CB, Gs_pad = G * bits_ // 8, (Gs + 3) // 4 * 4
    end = 256 + P * (P - 1) * Gs * CB
    end = _r256(end) + P * (P - 1) * Gs_pad * 4
    end = _r256(end) + P * Gs * CB
    end = _r256(end) + P * Gs_pad * 4
    return _r256(end)


def _largest_groups(P, bits_):
    """The most groups per segment whose slots fit the array."""
    lo, hi = 1, SCRATCH
    while lo < hi:
        mid = (lo + hi + 1) // 2
        lo, hi = (mid, hi) if _slot_bytes(P, mid, bits_) <= SCRATCH else (lo, mid - 1)
    return lo


def _inputs(P, n, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    x = torch.randn((P, n), generator=gen, device="cuda")
    spread = torch.exp(torch.randn(n, generator=gen, device="cuda"))
    return (x * spread).to(torch.bfloat16)


@pytest.mark.parametrize("bits_", [4, 8])
@pytest.mark.parametrize("compensated", [True, False])
def test_noalloc_matches_the_plan_call_on_two_calls_in_a_row(bits_, compensated):
    from bit_error_compensated_gb300 import echo
    P, n = 4, 4 * G * 100
    plan = echo.echo_plan(P, n, G, bits_)
    comp_plan = torch.zeros((P, n), device="cuda") if compensated else None
    comp_free = torch.zeros((P, n), device="cuda") if compensated else None
    for k in range(2):
        x = _inputs(P, n, 40 + k)
        out_plan = torch.empty_like(x)
        out_free = torch.full_like(x, 7.0)          # stale contents must not leak through
        echo.echo_allreduce(plan, list(x), list(out_plan), comp_plan)
        echo.echo_allreduce_noalloc(P, n, bits_, list(x), list(out_free), comp_free)
        torch.cuda.synchronize()
        # the same tolerance as every other parity test: outputs bit for bit,
        # state within STATE_RTOL relative
        assert np.array_equal(bits(out_free), bits(out_plan)), f"outputs differ at call {k}"
        if compensated:
            assert STATE_RTOL == 1e-6
            assert_state_close(comp_free.cpu().numpy(), comp_plan.cpu().numpy(), f"state, call {k}")


def test_noalloc_allocates_nothing_per_call():
    from bit_error_compensated_gb300 import echo
    P, n = 2, 2 * G * 64
    x = _inputs(P, n, 5)
    out = torch.empty_like(x)
    comp = torch.zeros((P, n), device="cuda")
    echo.echo_allreduce_noalloc(P, n, 4, list(x), list(out), comp)   # first call: set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        echo.echo_allreduce_noalloc(P, n, 4, list(x), list(out), comp)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_sizes_beyond_its_scratch_and_the_plan_state():
    from bit_error_compensated_gb300 import echo
    P, n = 4, 4 * G * 16384 * 2          # 4096 x 4096 per rank: slots ~36 MB > 32 MiB
    keep = [torch.empty(8, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dummy = [t.data_ptr() for t in keep]   # raw addresses: the library's own check decides
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_allreduce_noalloc(P, n, 4, dummy, dummy, None)
    assert ei.value.status == echo.ECHO_ERR_TOO_LARGE
    assert "no-allocation" in echo.echo_strerror(echo.ECHO_ERR_TOO_LARGE)
    x = _inputs(2, 2 * G * 4, 1)
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_allreduce_noalloc(2, 2 * G * 4, 4, list(x), list(torch.empty_like(x)),
                                    echo.COMP_DEFAULT)
    assert ei.value.status == echo.ECHO_ERR_ARG


@pytest.mark.parametrize("P,bits_,size", [(4, 4, "2048x4096"), (4, 4, "largest"), (4, 8, "largest"),
                                          (2, 8, "largest"), (1, 4, "small"), (8, 4, "small")])
def test_noalloc_matches_the_oracle_up_to_its_largest_size(P, bits_, size):
    """Three compensated calls in a row, compared in full with the CPU oracle:
    every output bit for bit, the state within STATE_RTOL.  Sizes: the
    2048 x 4096 per rank that the header names as fitting at P=4 with 4-bit
    codes, the largest n whose receive slots fit the fixed array (4- and 8-bit),
    and small P=1 and P=8 calls.  The plan-based call on the same inputs must
    give the same outputs too."""
    from bit_error_compensated_gb300 import echo
    if size == "2048x4096":
        n = 2048 * 4096
        assert _slot_bytes(P, n // P // G, bits_) <= SCRATCH
    elif size == "largest":
        n = P * G * _largest_groups(P, bits_)
    else:
        n = P * G * 37
    plan = echo.echo_plan(P, n, G, bits_)
    comp_free = torch.zeros((P, n), device="cuda")
    comp_plan = torch.zeros((P, n), device="cuda")
    e_ref = np.zeros((P, n), np.float32)
    for k in range(3):
        x = _inputs(P, n, 70 + k)
        out_free = torch.full_like(x, 3.0)
        out_plan = torch.empty_like(x)
        echo.echo_allreduce_noalloc(P, n, bits_, list(x), list(out_free), comp_free)
        echo.echo_allreduce(plan, list(x), list(out_plan), comp_plan)
        torch.cuda.synchronize()
        ref = oracle.allreduce(bits(x), G, bits_, e=e_ref)
        got = bits(out_free)
        assert np.array_equal(got, ref["out"]), f"outputs differ from the oracle at call {k}"
        assert_state_close(comp_free.cpu().numpy(), e_ref, f"state, call {k}")
        assert np.array_equal(bits(out_plan), got), f"plan call differs at call {k}"
    assert echo.echo_get_status(plan) == 0


@pytest.mark.parametrize("P,bits_", [(4, 4), (4, 8), (2, 8), (16, 4)])
def test_noalloc_rejects_one_tile_past_its_largest_size(P, bits_):
    """The smallest n past the largest that fits -- one more group per segment
    -- returns ECHO_ERR_TOO_LARGE before touching any buffer."""
    from bit_error_compensated_gb300 import echo
    Gs = _largest_groups(P, bits_)
    assert _slot_bytes(P, Gs + 1, bits_) > SCRATCH
    keep = [torch.empty(8, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dummy = [t.data_ptr() for t in keep]
    with pytest.raises(echo.EchoError) as ei:
        echo.echo_allreduce_noalloc(P, P * G * (Gs + 1), bits_, dummy, dummy, None)
    assert ei.value.status == echo.ECHO_ERR_TOO_LARGE
