"""Every element of the five workloads at full size, in the launch
configuration the bench times, checked against the identity that error
feedback makes exact ("Echo: Error-Compensated 4-Bit Tensor-Parallel
Communication", abstract and Fig. 2(a); "Your All-Reduce Is 4x Overpriced",
"The cancellation rule": the sum reveals each injected error, and the error is
fed into the next call).

The sampled and full comparisons with the oracle (test_gpu_workloads.py) fix
the values bit for bit; this file adds a check of EVERY element of every call
at sizes where the oracle only sees a sample.  For one call, with E(i) the sum
over ranks of the held errors at element position i:

    y(i) = sum_p x_p(i) + E_before(i) - E_after(i)

up to the fp32 roundings of the call's own adds (the entry pass v = x + e, the
senders' residuals v - deq(q), the P - 1 adds of the owner's sum and its
residual S - y): each is at most 2^-24 of its result, so the residual of the
identity is bounded by (P + 2) * 2^-23 * (sum |x| + sum |e_before| +
sum |e_after|) per position.  A dropped state write, a wrong rank or segment
index, an output written to the wrong place or a missed add breaks it by
about a quantization step, orders of magnitude above that bound.  Summed over
a sequence it telescopes: the accumulated error sum_k (y_k - sum_p x_pk)
equals -E_N (E_0 = 0), so it is set by the state alone and does not grow with
the number of calls, while without compensation it grows like a random walk.
All P outputs of every call are also compared bit for bit.
"""
import math

import pytest
import torch

from bit_error_compensated_gb300.workloads import WORKLOADS, Call, call_sequence, rank_inputs

pytestmark = pytest.mark.gpu
G = 128
CHUNK = 1 << 24                  # element positions per fp64 pass
ULP2 = 2.0 ** -23                # twice the unit roundoff of fp32
TINY = 2.0 ** -140               # absolute slack per position for subnormal results


@pytest.fixture(scope="module")
def echo():
    from bit_error_compensated_gb300 import echo as mod
    return mod


def _rank_sums(t: torch.Tensor, c0: int, c1: int):
    """fp64 sum over ranks of t[:, c0:c1] and of its magnitudes."""
    d = t[:, c0:c1].double()
    return d.sum(0), d.abs().sum(0)


class IdentityCheck:
    """Per-call check of the identity above, and the accumulated error of a
    sequence of calls on one compensator state."""

    def __init__(self, P: int, n: int):
        self.P, self.n = P, n
        dev = "cuda"
        self.t = torch.empty(n, dtype=torch.float64, device=dev)      # sum x + E_before
        self.mag = torch.empty(n, dtype=torch.float64, device=dev)    # sum |x| + sum |e_before|
        self.sx = torch.empty(n, dtype=torch.float64, device=dev)     # sum x
        self.worst = 0.0

    def before(self, x: torch.Tensor, comp: torch.Tensor):
        for c0 in range(0, self.n, CHUNK):
            c1 = min(self.n, c0 + CHUNK)
            sx, ax = _rank_sums(x, c0, c1)
            se, ae = _rank_sums(comp, c0, c1)
            self.sx[c0:c1] = sx
            self.t[c0:c1] = sx + se
            self.mag[c0:c1] = ax + ae

    def after(self, out: torch.Tensor, comp: torch.Tensor, drift: torch.Tensor,
              bounds: torch.Tensor, what: str):
        """Checks the call just made; adds y - sum x to `drift` and the call's
        rounding bound to `bounds`."""
        y16 = out.view(torch.int16)
        for r in range(1, self.P):
            assert torch.equal(y16[r], y16[0]), f"{what}: output of rank {r} differs from rank 0's"
        for c0 in range(0, self.n, CHUNK):
            c1 = min(self.n, c0 + CHUNK)
            y = out[0, c0:c1].double()
            se, ae = _rank_sums(comp, c0, c1)
            resid = (y - self.t[c0:c1] + se).abs()
            bound = (self.P + 2) * ULP2 * (self.mag[c0:c1] + ae) + self.P * TINY
            ratio = float((resid / bound).max())
            self.worst = max(self.worst, ratio)
            if ratio > 1.0:
                i = int((resid / bound).argmax()) + c0
                raise AssertionError(
                    f"{what}: identity broken at element {i}: residual {float(resid.max()):.3e}"
                    f" against a rounding bound of {float(bound[i - c0]):.3e}")
            drift[c0:c1] += y - self.sx[c0:c1]
            bounds[c0:c1] += bound


def _run_identity(echo, number, bits_, seq, configure=None):
    """Runs `seq` (calls of workload `number`) through one plan in the default
    schedule (or as `configure` sets it), checking every call and, at the
    end, each compensator stream's accumulated error.  Returns the largest
    residual as a fraction of its rounding bound."""
    w = WORKLOADS[number]
    P, n = w.P, w.n
    plan = echo.echo_plan(P, n, G, bits_)
    if configure is not None:
        configure(plan)
    x = torch.empty((P, n), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    chk = IdentityCheck(P, n)
    states, drift, bounds = {}, {}, {}
    for k, c in enumerate(seq):
        rank_inputs(number, c, "cuda", out=x)
        if c.state == "none":
            echo.echo_allreduce(plan, list(x), list(out), None)
            y16 = out.view(torch.int16)
            for r in range(1, P):
                assert torch.equal(y16[r], y16[0]), f"call {k}: outputs differ across ranks"
            continue
        comp = states.setdefault(c.state, torch.zeros((P, n), device="cuda"))
        zeros = lambda: torch.zeros(n, dtype=torch.float64, device="cuda")
        d, b = drift.setdefault(c.state, zeros()), bounds.setdefault(c.state, zeros())
        chk.before(x, comp)
        echo.echo_allreduce(plan, list(x), list(out), comp)
        chk.after(out, comp, d, b, f"{w.name} ({bits_}-bit) call {k} ({c.state})")
    assert echo.echo_get_status(plan) == 0
    print(f"{w.name} ({bits_}-bit): {len(seq)} calls, every element; largest residual "
          f"{chk.worst:.3f} of its rounding bound")
    _drift_telescopes(drift, bounds, states)
    return chk.worst


def _drift_telescopes(drift, bounds, states):
    """The accumulated error D_N = sum_k (y_k - sum_p x_pk) of each state's
    calls equals -E_N (E_0 = 0) within the sum of the calls' rounding bounds:
    the per-call identities telescope.  So D_N is bounded by the held errors,
    whatever the number of calls."""
    for name, d in drift.items():
        e = states[name].double().sum(0)
        excess = (d + e).abs() - bounds[name] * (1 + 2.0 ** -30)
        assert float(excess.max()) <= 0.0, f"state {name}: accumulated error is not -E_N"


@pytest.mark.parametrize("number", [1, 2, 4, 5])
def test_every_element_of_every_call(echo, number):
    """p2_n4096 (9 calls), p4_2048x4096 (64), p4_8192x4096 (72) and
    p4_32768x1024 (ten steps of 112 calls, forward and backward states: 1120),
    every element of every call: each workload's whole call sequence."""
    assert _run_identity(echo, number, 4, call_sequence(number)) <= 1.0


SCHEDULES = {
    "tile": None,
    "two-kernels": lambda echo, plan: echo.echo_set_tile_fused(plan, echo.ECHO_TILE_OFF),
    "separate-gather": lambda echo, plan: (echo.echo_set_tile_fused(plan, echo.ECHO_TILE_OFF),
                                           echo.echo_set_fused(plan, False)),
    "persistent": lambda echo, plan: echo.echo_set_persistent(plan, True),
}


@pytest.mark.parametrize("bits_,schedule", [(4, s) for s in SCHEDULES] + [(8, "tile")])
def test_p8_1gib_every_element(echo, bits_, schedule):
    """P = 8 ranks of 1 GiB: the workload's call from zero state, then a second
    call on fresh inputs that carries the first call's held errors, every one
    of the 4 Gi elements checked, in each schedule (the 8-bit variant in the
    default one, the schedule it is timed in)."""
    seq = [call_sequence(3)[0], Call(1, "fwd", "normal_0.02")]
    f = SCHEDULES[schedule]
    configure = None if f is None else (lambda plan: f(echo, plan))
    assert _run_identity(echo, 3, bits_, seq, configure) <= 1.0
    torch.cuda.empty_cache()


def test_drift_bounded_with_compensation_and_growing_without(echo):
    """P = 2, n = 4096 (the two-rank workload's shape and distribution), 1000
    calls on fresh inputs: the RMS of the accumulated error stays within a
    constant of one call's with compensation, and grows like sqrt(N) without."""
    P, n, N = 2, 4096, 1000
    plan = echo.echo_plan(P, n, G, 4)
    x = torch.empty((P, n), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    comp = torch.zeros((P, n), device="cuda")
    rms = lambda t: float(torch.sqrt((t * t).mean()))
    result = {}
    for compensated in (True, False):
        comp.zero_()
        d = torch.zeros(n, dtype=torch.float64, device="cuda")
        d1 = None
        for k in range(N):
            rank_inputs(1, Call(10_000 + k, "fwd", "normal"), "cuda", out=x)
            echo.echo_allreduce(plan, list(x), list(out), comp if compensated else None)
            d += out[0].double() - x.double().sum(0)
            if k == 0:
                d1 = d.clone()
        result[compensated] = (rms(d), rms(d1))
    (dc, dc1), (du, du1) = result[True], result[False]
    assert dc <= 3.0 * dc1
    assert du >= 0.5 * math.sqrt(N) * du1
    assert du > 10 * dc
    print(f"1000 calls: RMS drift {dc:.4f} compensated (one call {dc1:.4f}), "
          f"{du:.4f} uncompensated (one call {du1:.4f})")
