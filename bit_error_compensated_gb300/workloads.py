"""Seeded synthetic inputs shaped like the workloads of the Echo pages.

This module holds none of the all-reduce's arithmetic: it only draws random
bf16 tensors of stated shapes and distributions, and lists each workload's call
sequence.  Both the GPU path and the CPU oracle are fed from it (the same tensor
goes to both sides), so it imports neither.

The pages measure tensor-parallel all-reduce on real models (Llama-3-8B,
Qwen3-0.6B/8B; "Echo: Error-Compensated 4-Bit Tensor-Parallel Communication",
Table 6, Table 7, Fig. 3) and quote a 1 GB message size (abstract).  No model or
dataset is used here; each workload is a stand-in with the activation shape
(tokens x hidden), the per-channel scale spread and the outlier channels that
TP partial sums of such models show, drawn from a fixed seed.

Workloads (one rank's tensor is [tokens, hidden] flattened row-major, so the
channel of element i is i % hidden):

  p2_n4096        P=2, n=4096, i.i.d. N(0,1); one uncompensated call, then
                  8 compensated calls on fresh inputs.
  p4_2048x4096    P=4, 2048 x 4096, N(0,1) x sigma_c with sigma_c ~ LogNormal(0,1)
                  per channel (drawn per call, shared by ranks and tokens) and
                  1% of channels (41 of 4096, drawn per call) x20; 64 compensated
                  calls (32 layers x attention+MLP sites).
  p8_1gib         P=8, 512 Mi elements (1 GiB bf16) per rank, i.i.d. N(0, 0.02^2);
                  one compensated call from zero state; 4-bit and 8-bit codes.
  p4_8192x4096    P=4, 8192 x 4096, Student-t(nu=4) x per-channel LogNormal(0,0.5);
                  72 compensated calls (36 layers x 2 sites).
  p4_32768x1024   P=4, (8 x 4096) x 1024; per step 56 forward sites drawn as
                  N(0,1) x per-channel LogNormal(0,1) on one compensator state,
                  then 56 backward sites drawn as N(0, 1e-3^2) on a second state;
                  10 steps, both states carried (1120 calls).

The seed of call k of workload c is 1000*c + k, with c the workload's number.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    number: int
    name: str
    P: int
    tokens: int
    hidden: int
    bits: tuple          # code widths the workload runs with
    description: str

    @property
    def n(self) -> int:
        return self.tokens * self.hidden


WORKLOADS = {
    1: Workload(1, "p2_n4096", 2, 1, 4096, (4,),
                "P=2, n=4096, iid N(0,1); 1 uncompensated + 8 compensated calls"),
    2: Workload(2, "p4_2048x4096", 4, 2048, 4096, (4,),
                "P=4, 2048x4096, N(0,1) x LogNormal(0,1) channels, 1% x20 outliers; 64 calls"),
    3: Workload(3, "p8_1gib", 8, 131072, 4096, (4, 8),
                "P=8, 512Mi elements per rank, iid N(0,0.02^2); 1 call, 4-bit and 8-bit"),
    4: Workload(4, "p4_8192x4096", 4, 8192, 4096, (4,),
                "P=4, 8192x4096, Student-t(4) x LogNormal(0,0.5) channels; 72 calls"),
    5: Workload(5, "p4_32768x1024", 4, 32768, 1024, (4,),
                "P=4, 32768x1024, 10 steps x (56 fwd N(0,1)xLogNormal(0,1) + 56 bwd N(0,1e-6))"),
}


@dataclass(frozen=True)
class Call:
    index: int        # position in the workload's sequence (also seeds the inputs)
    state: str        # "none" (uncompensated), "fwd" or "bwd": which compensator state
    dist: str         # distribution family drawn for this call


def call_sequence(number: int, steps: int | None = None) -> list:
    """The ordered calls of a workload (see the module docstring)."""
    if number == 1:
        return [Call(0, "none", "normal")] + [Call(k, "fwd", "normal") for k in range(1, 9)]
    if number == 2:
        return [Call(k, "fwd", "lognormal_outliers") for k in range(64)]
    if number == 3:
        return [Call(0, "fwd", "normal_0.02")]
    if number == 4:
        return [Call(k, "fwd", "student_t") for k in range(72)]
    if number == 5:
        seq, k = [], 0
        for _ in range(10 if steps is None else steps):
            for _ in range(56):
                seq.append(Call(k, "fwd", "lognormal"))
                k += 1
            for _ in range(56):
                seq.append(Call(k, "bwd", "normal_1e-3"))
                k += 1
        return seq
    raise KeyError(number)


def seed_of(number: int, call_index: int) -> int:
    return 1000 * number + call_index


def _channel_scales(gen, hidden, sigma, device):
    return torch.exp(sigma * torch.randn(hidden, generator=gen, device=device))


def rank_inputs(number: int, call: Call, device="cpu", P: int | None = None,
                tokens: int | None = None, hidden: int | None = None,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """Draw one call's inputs: a [P, tokens*hidden] bf16 tensor on ``device``.

    P, tokens and hidden default to the workload's own; overriding them gives a
    smaller tensor with the same distribution (used by the fast tests).  ``out``
    (a [P, n] bf16 tensor) is filled in place when given.
    """
    w = WORKLOADS[number]
    P = w.P if P is None else P
    tokens = w.tokens if tokens is None else tokens
    hidden = w.hidden if hidden is None else hidden
    n = tokens * hidden
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed_of(number, call.index))
    if out is None:
        out = torch.empty((P, n), dtype=torch.bfloat16, device=dev)
    assert out.shape == (P, n) and out.dtype == torch.bfloat16

    scales = None
    if call.dist == "lognormal_outliers":
        scales = _channel_scales(gen, hidden, 1.0, dev)
        n_out = max(1, round(0.01 * hidden))
        idx = torch.randperm(hidden, generator=gen, device=dev)[:n_out]
        scales[idx] *= 20.0
    elif call.dist == "lognormal":
        scales = _channel_scales(gen, hidden, 1.0, dev)
    elif call.dist == "student_t":
        scales = _channel_scales(gen, hidden, 0.5, dev)

    for p in range(P):  # one rank at a time bounds the fp32 temporaries
        z = torch.randn((tokens, hidden), generator=gen, device=dev)
        if call.dist == "normal_0.02":
            z *= 0.02
        elif call.dist == "normal_1e-3":
            z *= 1e-3
        elif call.dist == "student_t":
            # t with 4 degrees of freedom: Z / sqrt(V / 4), V a chi-square(4)
            # drawn as the sum of four squared standard normals.
            v = torch.zeros_like(z)
            for _ in range(4):
                v += torch.randn((tokens, hidden), generator=gen, device=dev) ** 2
            z /= torch.sqrt(v / 4.0)
        if scales is not None:
            z *= scales
        out[p].copy_(z.reshape(-1))
        del z
    return out
