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

from _parity import STATE_RTOL, assert_state_close, bits

pytestmark = pytest.mark.gpu
G = 128


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
