"""Plans used at the same time from several host threads, each on its own
stream: the library's one-time kernel set-up and launch caches are shared by
all threads, while every plan owns its receive slots, so calls of different
plans may overlap on the GPU.  Each thread creates its plan and issues its
calls while the others do; afterwards every call's outputs and the final
state are compared with the oracle replaying that thread's sequence alone
(outputs bit for bit, state within STATE_RTOL).

The persistent schedule is left out: its launch is cooperative, and whether
its blocks become resident at once beside other streams' kernels is the
driver's to decide.
"""
import threading

import numpy as np
import pytest
import torch

import oracle
from _parity import STATE_DTYPES, assert_state_close, bits

pytestmark = pytest.mark.gpu

# name: (P, g, groups per segment, bits, state format or None, tile, fused)
WORKERS = {
    "p4_rank_parallel_f32": (4, 128, 37, 4, 0, 1, 1),
    "p8_rank_loop_8bit_bf16": (8, 128, 1000, 8, 1, 1, 1),
    "p2_two_kernels_uncompensated": (2, 128, 300, 4, None, 0, 1),
    "p3_three_kernels_g64_f32": (3, 64, 75, 4, 0, 0, 0),
    "p16_g256_f16": (16, 256, 9, 4, 2, 1, 1),
}
CALLS = 6


def _inputs(P, n, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    x = torch.randn((P, n), generator=gen, device="cuda")
    return (x * torch.exp(torch.randn(n, generator=gen, device="cuda"))).to(torch.bfloat16)


def test_plans_on_concurrent_threads_and_streams():
    from bit_error_compensated_gb300 import echo
    inputs = {}
    for i, (name, (P, g, Gs, _, _, _, _)) in enumerate(WORKERS.items()):
        n = P * g * Gs
        inputs[name] = [_inputs(P, n, 3000 + 100 * i + k) for k in range(CALLS)]
    torch.cuda.synchronize()
    start = threading.Barrier(len(WORKERS))
    results, errors = {}, []

    def worker(name):
        try:
            P, g, Gs, bits_, fmt, tile, fused = WORKERS[name]
            n = P * g * Gs
            stream = torch.cuda.Stream()
            start.wait()                                   # plans created concurrently
            plan = echo.echo_plan(P, n, g, bits_)
            echo.echo_set_tile_fused(plan, tile)
            echo.echo_set_fused(plan, bool(fused))
            comp = None
            if fmt is not None:
                echo.echo_set_state(plan, fmt, 1.0)
                comp = torch.zeros((P, n), dtype=STATE_DTYPES[fmt], device="cuda")
            outs = []
            with torch.cuda.stream(stream):
                for x in inputs[name]:
                    out = torch.empty_like(x)
                    echo.echo_allreduce(plan, list(x), list(out), comp, stream=stream)
                    outs.append(out)
            stream.synchronize()
            assert echo.echo_get_status(plan, stream) == 0
            results[name] = (outs, comp)
        except BaseException as exc:                       # reported by the main thread
            errors.append((name, exc))
            start.abort()

    threads = [threading.Thread(target=worker, args=(name,)) for name in WORKERS]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    assert not errors, errors
    torch.cuda.synchronize()

    for name, (P, g, Gs, bits_, fmt, _, _) in WORKERS.items():
        n = P * g * Gs
        outs, comp = results[name]
        e = None if fmt is None else np.zeros((P, n), np.float32)
        for k, x in enumerate(inputs[name]):
            ref = oracle.allreduce(bits(x), g, bits_, e=e, state_fmt=fmt)
            assert np.array_equal(bits(outs[k]), ref["out"]), f"{name}: outputs differ at call {k}"
        if fmt is not None:
            assert_state_close(comp.float().cpu().numpy(), e, f"{name}: state")
