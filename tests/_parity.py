"""Helpers for comparing the CUDA path (through the C ABI) with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Outputs and codes must match bit for bit (both sides take every step in the
# same IEEE fp32 order); the compensator state is held to 1e-6 relative to the
# fp32 value, and in practice matches bit for bit too.
STATE_RTOL = 1e-6


# torch dtype of a compensator state in each format (0 fp32, 1 bf16, 2 fp16)
STATE_DTYPES = {0: torch.float32, 1: torch.bfloat16, 2: torch.float16}


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def unpack_codes(raw: np.ndarray, bits_: int) -> np.ndarray:
    """Packed code bytes -> one code per element (the wire format of echo.h)."""
    raw = np.asarray(raw, np.uint8)
    if bits_ == 8:
        return raw.copy()
    out = np.empty(raw.size * 2, np.uint8)
    out[0::2] = raw & 0xF
    out[1::2] = raw >> 4
    return out


def wire_to_canonical(wire: bytes, lay: dict, P: int, n: int, bits_: int) -> dict:
    """Receive slots of the GPU plan -> the oracle's canonical layout:
    q1 [P, n] (own-segment entries 0), m1 [P, P, Gs], q2 [n], m2 [P, Gs]."""
    buf = np.frombuffer(wire, np.uint8)
    Gs, Gs_pad, CB = lay["Gs"], lay["Gs_pad"], lay["code_bytes"]
    m = n // P
    q1 = np.zeros((P, n), np.uint8)
    m1 = np.zeros((P, P, Gs), np.uint32)
    if P > 1:
        c1 = buf[lay["codes1"]:lay["codes1"] + P * (P - 1) * Gs * CB].reshape(P, P - 1, Gs * CB)
        mt1 = buf[lay["meta1"]:lay["meta1"] + P * (P - 1) * Gs_pad * 4].view(np.uint32)
        mt1 = mt1.reshape(P, P - 1, Gs_pad)
        for o in range(P):
            for js in range(P - 1):
                p = js if js < o else js + 1
                q1[p, o * m:(o + 1) * m] = unpack_codes(c1[o, js], bits_)
                m1[p, o] = mt1[o, js, :Gs]
    c2 = buf[lay["codes2"]:lay["codes2"] + P * Gs * CB]
    q2 = unpack_codes(c2, bits_)
    m2 = buf[lay["meta2"]:lay["meta2"] + P * Gs_pad * 4].view(np.uint32).reshape(P, Gs_pad)[:, :Gs]
    return dict(q1=q1, m1=m1, q2=q2, m2=m2.copy())


def assert_state_close(got: np.ndarray, want: np.ndarray, what: str = "state"):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    if np.array_equal(got.view(np.uint32), want.view(np.uint32)):
        return
    denom = np.maximum(np.abs(want.astype(np.float64)), np.finfo(np.float32).tiny)
    rel = np.abs(got.astype(np.float64) - want) / denom
    # values that are both (signed) zero compare equal
    rel[(got == 0) & (want == 0)] = 0
    assert rel.max() <= STATE_RTOL, f"{what}: max rel err {rel.max():.3g} at {np.argmax(rel)}"


def assert_wire_equal(gpu: dict, ref: dict, P: int):
    assert np.array_equal(gpu["q2"], ref["q2"]), "gather codes differ"
    assert np.array_equal(gpu["m2"], ref["m2"]), "gather meta differ"
    if P > 1:
        assert np.array_equal(gpu["q1"], ref["q1"]), "push codes differ"
        assert np.array_equal(gpu["m1"], ref["m1"]), "push meta differ"


def group_element_index(groups: np.ndarray, g: int = 128) -> np.ndarray:
    """Element indices (within a rank tensor) of the given group indices."""
    return (np.asarray(groups, np.int64)[:, None] * g + np.arange(g)[None, :]).ravel()


def sample_groups(P: int, Gs: int, count: int, seed: int) -> np.ndarray:
    """A fixed, seed-chosen sample of group positions (global group index
    o*Gs + j), always including the first and last group of every segment."""
    rng = np.random.default_rng(seed)
    total = P * Gs
    base = set()
    for o in range(P):
        base.update({o * Gs, o * Gs + Gs - 1})
    extra = rng.choice(total, size=min(count, total), replace=False)
    return np.array(sorted(base.union(int(v) for v in extra)), np.int64)


class SampledOracle:
    """Runs the oracle on a fixed set of group positions, carrying each
    position's compensator state from call to call (positions are independent,
    so this is exactly the oracle's whole call restricted to them)."""

    def __init__(self, P: int, Gs: int, groups: np.ndarray, bits_: int, g: int = 128,
                 mode: int = 0, state_fmt: int = 0, decay: float = 1.0):
        self.P, self.Gs, self.groups, self.bits, self.g = P, Gs, groups, bits_, g
        self.mode, self.state_fmt, self.decay = mode, state_fmt, decay
        self.owners = (groups // Gs).astype(np.int32)
        self.idx = group_element_index(groups, g)
        self.idx_t = None
        self.states = {}

    def gather(self, t: torch.Tensor) -> torch.Tensor:
        """t [P, n] on the device -> the sampled elements, [P, npos*g] on host."""
        if self.idx_t is None or self.idx_t.device != t.device:
            self.idx_t = torch.from_numpy(self.idx).to(t.device)
        return t.index_select(1, self.idx_t).cpu()

    def call(self, x_sampled: np.ndarray, state: str | None, want_wire: bool = False):
        """x_sampled [P, npos*g] bf16 bits.  state: None (uncompensated) or a key."""
        npos = self.groups.size
        x = x_sampled.reshape(self.P, npos, self.g).transpose(1, 0, 2).copy()
        e = None
        if state is not None:
            e = self.states.setdefault(state, np.zeros((npos, self.P, self.g), np.float32))
        r = oracle.group_positions(self.P, self.owners, self.bits, x, e, want_wire=want_wire,
                                   mode=self.mode, state_fmt=self.state_fmt, decay=self.decay)
        r["y_rows"] = r["y"].reshape(-1)          # [npos*g], same for every rank
        return r

    def state_rows(self, state: str) -> np.ndarray:
        """The carried state as [P, npos*g] (the layout of gather())."""
        e = self.states[state]
        return e.transpose(1, 0, 2).reshape(self.P, -1)


def sampled_wire(wire: bytes, lay: dict, P: int, groups: np.ndarray, bits_: int) -> dict:
    """The receive slots of the sampled group positions, in the layout of
    oracle.group_positions: q1 [npos, P, g] (own rows 0), m1 [npos, P] (own 0),
    q2 [npos, g], m2 [npos]."""
    buf = np.frombuffer(wire, np.uint8)
    Gs, Gs_pad, CB = lay["Gs"], lay["Gs_pad"], lay["code_bytes"]
    g = CB * 8 // bits_
    npos = groups.size
    q1 = np.zeros((npos, P, g), np.uint8)
    m1 = np.zeros((npos, P), np.uint32)
    q2 = np.zeros((npos, g), np.uint8)
    m2 = np.zeros(npos, np.uint32)
    meta1 = buf[lay["meta1"]:lay["meta1"] + P * max(P - 1, 0) * Gs_pad * 4].view(np.uint32)
    meta2 = buf[lay["meta2"]:lay["meta2"] + P * Gs_pad * 4].view(np.uint32)
    for k, grp in enumerate(groups):
        o, j = int(grp) // Gs, int(grp) % Gs
        c = lay["codes2"] + int(grp) * CB
        q2[k] = unpack_codes(buf[c:c + CB], bits_)
        m2[k] = meta2[o * Gs_pad + j]
        for p in range(P):
            if p == o:
                continue
            slot = o * (P - 1) + (p if p < o else p - 1)
            c = lay["codes1"] + (slot * Gs + j) * CB
            q1[k, p] = unpack_codes(buf[c:c + CB], bits_)
            m1[k, p] = meta1[slot * Gs_pad + j]
    return dict(q1=q1, m1=m1, q2=q2, m2=m2)
