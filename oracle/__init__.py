"""Test infrastructure only: the CPU oracle for the Echo emulated all-reduce.

A plain, slow, single-threaded restatement of the per-call arithmetic of Echo
("Echo: Error-Compensated 4-Bit Tensor-Parallel Communication for LLM Training
and Inference", arXiv 2610.14277, Fig. 2(a)), in C++ (``echo_oracle.cpp``),
wrapped here with ctypes and numpy.  Only the test suite, the smoke check and the
bench's CPU-baseline leg import this package; the GPU library never does, and
this package never imports the GPU library.

Arrays cross the boundary as numpy arrays: bf16 values as their uint16 bit
patterns, the compensator state as float32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_DIR = Path(__file__).resolve().parent
_SRC = _DIR / "echo_oracle.cpp"
_LIB = _DIR / "liboracle.so"


def build(force: bool = False) -> Path:
    """Compile the oracle with plain IEEE fp32 (no fused multiply-add)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        subprocess.check_call([
            "g++", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17",
            "-fPIC", "-shared", "-o", str(tmp), str(_SRC),
        ])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB))
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_f16_ru.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_f16_ru.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_bf16_rn.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16_rn.restype = ctypes.c_uint16
        for fn in ("oracle_f32_to_f16_ru_n", "oracle_f16_to_f32_n", "oracle_f32_to_bf16_rn_n",
                   "oracle_f32_to_f16_rd_n", "oracle_f32_to_f16_rn_n"):
            getattr(lib, fn).argtypes = [P, i64, P]
            getattr(lib, fn).restype = None
        lib.oracle_quantize_group.argtypes = [P, i32, i32, P, P, P, P]
        lib.oracle_quantize_group.restype = i32
        lib.oracle_dequantize_group.argtypes = [P, i32, ctypes.c_uint16, ctypes.c_uint16, P]
        lib.oracle_dequantize_group.restype = None
        lib.oracle_pack_codes.argtypes = [P, i64, i32, P]
        lib.oracle_pack_codes.restype = None
        lib.oracle_group_position.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_group_position.restype = i32
        lib.oracle_group_positions.argtypes = [i32, i64, P, i32, i32, P, P, P, P, P, P, P, P]
        lib.oracle_group_positions.restype = i64
        lib.oracle_quantize_group_mode.argtypes = [P, i32, i32, i32, P, P, P, P]
        lib.oracle_quantize_group_mode.restype = i32
        lib.oracle_dequantize_group_mode.argtypes = [P, i32, i32, ctypes.c_uint16, ctypes.c_uint16, P]
        lib.oracle_dequantize_group_mode.restype = None
        lib.oracle_group_positions_mode.argtypes = [i32, i64, P, i32, i32, i32, P, P, P, P, P, P, P, P]
        lib.oracle_group_positions_mode.restype = i64
        lib.oracle_allreduce_mode.argtypes = [i32, i64, i32, i32, i32, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_allreduce_mode.restype = i64
        lib.oracle_group_positions_ex.argtypes = [i32, i64, P, i32, i32, i32, i32, ctypes.c_float,
                                                  P, P, P, P, P, P, P, P]
        lib.oracle_group_positions_ex.restype = i64
        lib.oracle_allreduce_ex.argtypes = [i32, i64, i32, i32, i32, i32, ctypes.c_float,
                                            P, P, P, P, P, P, P, P, P, P]
        lib.oracle_allreduce_ex.restype = i64
        lib.oracle_allreduce.argtypes = [i32, i64, i32, i32, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_allreduce.restype = i64
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- formats ----

def f32_to_f16_ru(x: np.ndarray) -> np.ndarray:
    """binary32 -> binary16 bits, rounding toward +infinity (element-wise)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.zeros(x.size, dtype=np.uint16)
    _load().oracle_f32_to_f16_ru_n(_ptr(x), x.size, _ptr(out))
    return out


def f32_to_f16_rn(x: np.ndarray) -> np.ndarray:
    """float32 -> binary16 bits, round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_f32_to_f16_rn_n(_ptr(x), x.size, _ptr(out))
    return out


def f32_to_f16_rd(x: np.ndarray) -> np.ndarray:
    """binary32 -> binary16 bits, rounding toward -infinity (element-wise)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.zeros(x.size, dtype=np.uint16)
    _load().oracle_f32_to_f16_rd_n(_ptr(x), x.size, _ptr(out))
    return out


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    """binary16 bits -> binary32 (exact)."""
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.zeros(h.size, dtype=np.float32)
    _load().oracle_f16_to_f32_n(_ptr(h), h.size, _ptr(out))
    return out


def f32_to_bf16_rn(x: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bits, round to nearest even (element-wise)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.zeros(x.size, dtype=np.uint16)
    _load().oracle_f32_to_bf16_rn_n(_ptr(x), x.size, _ptr(out))
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact: a bf16 bit pattern is the high half of the binary32 pattern."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# -------------------------------------------------------------- quantizer ----

# Quantizer variants: the method's zero-aware asymmetric quantizer and the two
# ablations of Table 8 ("naive zero-point", "symmetric grid").
ZERO_AWARE, NAIVE_ZERO_POINT, SYMMETRIC = 0, 1, 2
# Compensator state storage (the value kept for each revealed error).
STATE_F32, STATE_BF16, STATE_F16 = 0, 1, 2

def quantize_group(v: np.ndarray, bits: int, mode: int = ZERO_AWARE):
    """Q_b on one group.  Returns (codes uint8, s_bits, z_bits, flagged, ties);
    for the naive zero-point mode z_bits is the fp16 offset m.  ``ties`` counts
    the exact rounding ties met: every rint whose fp32 argument lies exactly on
    a half-integer (a code's v/s -- (v - m)/s for the naive zero point -- and
    the zero-aware zero point's -lo/s), negative or positive, before any clamp."""
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float32)
    q = np.zeros(v.size, dtype=np.uint8)
    sb = ctypes.c_uint16()
    zb = ctypes.c_uint16()
    ties = ctypes.c_int64(0)
    if mode == ZERO_AWARE:
        bad = lib.oracle_quantize_group(_ptr(v), v.size, bits, _ptr(q), ctypes.byref(sb),
                                        ctypes.byref(zb), ctypes.byref(ties))
    else:
        bad = lib.oracle_quantize_group_mode(_ptr(v), v.size, bits, mode, _ptr(q), ctypes.byref(sb),
                                             ctypes.byref(zb), ctypes.byref(ties))
    return q, sb.value, zb.value, bad, ties.value


def dequantize_group(q: np.ndarray, s_bits: int, z_bits: int, mode: int = ZERO_AWARE) -> np.ndarray:
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.zeros(q.size, dtype=np.float32)
    if mode == ZERO_AWARE:
        lib.oracle_dequantize_group(_ptr(q), q.size, s_bits, z_bits, _ptr(out))
    else:
        lib.oracle_dequantize_group_mode(_ptr(q), q.size, mode, s_bits, z_bits, _ptr(out))
    return out


def pack_codes(q: np.ndarray, bits: int) -> np.ndarray:
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint8).ravel()
    out = np.zeros(q.size if bits == 8 else (q.size + 1) // 2, dtype=np.uint8)
    lib.oracle_pack_codes(_ptr(q), q.size, bits, _ptr(out))
    return out


# ------------------------------------------------------------------ calls ----

def group_position(P: int, owner: int, bits: int, x: np.ndarray, e: np.ndarray | None):
    """One group position: x [P, len] bf16 bits; e [P, len] float32 (updated in
    place) or None.  Returns a dict of y, q1, m1, q2, m2, acc, nq, flagged, ties."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert x.ndim == 2 and x.shape[0] == P
    ln = x.shape[1]
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.shape == x.shape
    r = dict(y=np.zeros(ln, np.uint16), q1=np.zeros((P, ln), np.uint8),
             m1=np.zeros(P, np.uint32), q2=np.zeros(ln, np.uint8), m2=np.zeros(1, np.uint32),
             acc=np.zeros(ln, np.float32), nq=np.zeros((P, ln), np.uint8))
    ties = ctypes.c_int64(0)
    r["flagged"] = lib.oracle_group_position(
        P, owner, ln, bits, _ptr(x), _ptr(e), _ptr(r["y"]), _ptr(r["q1"]), _ptr(r["m1"]),
        _ptr(r["q2"]), _ptr(r["m2"]), _ptr(r["acc"]), _ptr(r["nq"]), ctypes.byref(ties))
    r["ties"] = ties.value
    return r


def _state_fmt(bf16_state: bool, state_fmt: int | None) -> int:
    fmt = (STATE_BF16 if bf16_state else STATE_F32) if state_fmt is None else state_fmt
    if fmt not in (STATE_F32, STATE_BF16, STATE_F16):
        raise ValueError(f"state format {fmt}")
    return fmt


def group_positions(P: int, owners: np.ndarray, bits: int, x: np.ndarray,
                    e: np.ndarray | None, want_wire: bool = False, mode: int = ZERO_AWARE,
                    bf16_state: bool = False, decay: float = 1.0, state_fmt: int | None = None):
    """Many independent group positions at once.

    owners [npos] int; x [npos, P, len] bf16 bits; e [npos, P, len] float32
    (updated in place) or None.  Returns a dict with y [npos, len] and, on
    request, q1 [npos, P, len], m1 [npos, P], q2 [npos, len], m2 [npos]; plus
    ``flagged`` and ``ties``."""
    lib = _load()
    owners = np.ascontiguousarray(owners, dtype=np.int32)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    npos, P_, ln = x.shape
    assert P_ == P and owners.shape == (npos,)
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.shape == x.shape
    r = dict(y=np.zeros((npos, ln), np.uint16))
    if want_wire:
        r.update(q1=np.zeros((npos, P, ln), np.uint8), m1=np.zeros((npos, P), np.uint32),
                 q2=np.zeros((npos, ln), np.uint8), m2=np.zeros(npos, np.uint32))
    ties = ctypes.c_int64(0)
    bad = lib.oracle_group_positions_ex(P, npos, _ptr(owners), ln, bits, mode,
                                        _state_fmt(bf16_state, state_fmt),
                                        decay, _ptr(x), _ptr(e), _ptr(r["y"]), _ptr(r.get("q1")),
                                        _ptr(r.get("m1")), _ptr(r.get("q2")), _ptr(r.get("m2")),
                                        ctypes.byref(ties))
    if bad < 0:
        raise ValueError("oracle_group_positions rejected its arguments")
    r["flagged"] = int(bad)
    r["ties"] = ties.value
    return r


def allreduce(x: np.ndarray, g: int, bits: int, e: np.ndarray | None = None,
              want_wire: bool = False, want_acc: bool = False, want_nq: bool = False,
              mode: int = ZERO_AWARE, bf16_state: bool = False, decay: float = 1.0,
              state_fmt: int | None = None):
    """One emulated all-reduce call.

    x: [P, n] uint16 bf16 bits.  e: [P, n] float32 compensator state, updated IN
    PLACE, or None for an uncompensated call.  state_fmt (STATE_F32, STATE_BF16,
    STATE_F16; bf16_state=True is STATE_BF16) makes the state keep values
    rounded to that type (still in the float32 array); decay scales each
    revealed error before it is kept.  Returns a dict with ``out``
    ([P, n] bf16 bits), ``flagged``, ``ties`` and, on request, the wire codes in
    the oracle's canonical layout (q1 [P, n], m1 [P, P, Gs], q2 [n], m2 [P, Gs]),
    the owner sums ``acc`` [n] and the quantization counts ``nq`` [P, n].
    """
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    P, n = x.shape
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.shape == (P, n)
    m = n // P
    Gs = -(-m // g)
    r = dict(out=np.zeros((P, n), np.uint16))
    if want_wire:
        r.update(q1=np.zeros((P, n), np.uint8), m1=np.zeros((P, P, Gs), np.uint32),
                 q2=np.zeros(n, np.uint8), m2=np.zeros((P, Gs), np.uint32))
    if want_acc:
        r["acc"] = np.zeros(n, np.float32)
    if want_nq:
        r["nq"] = np.zeros((P, n), np.uint8)
    ties = ctypes.c_int64(0)
    bad = lib.oracle_allreduce_ex(P, n, g, bits, mode, _state_fmt(bf16_state, state_fmt), decay, _ptr(x),
                                  _ptr(r["out"]), _ptr(e),
                                    _ptr(r.get("q1")), _ptr(r.get("m1")), _ptr(r.get("q2")),
                                    _ptr(r.get("m2")), _ptr(r.get("acc")), _ptr(r.get("nq")),
                                    ctypes.byref(ties))
    if bad < 0:
        raise ValueError(f"oracle_allreduce rejected P={P} n={n} g={g} bits={bits} mode={mode}")
    r["flagged"] = int(bad)
    r["ties"] = ties.value
    return r
