"""ctypes binding of libecho.so (include/echo.h), with the same call names.

Argument marshalling only: tensors become device pointers, torch streams become
cudaStream_t handles, status codes become exceptions.  Every step of the
all-reduce runs in the library's CUDA kernels; there is no fallback.  Importing
this module raises if the library has not been built
(``python -m bit_error_compensated_gb300.build``).
"""
from __future__ import annotations

import ctypes
from pathlib import Path

_LIB_PATH = Path(__file__).resolve().parent / "lib" / "libecho.so"
if not _LIB_PATH.exists():
    raise ImportError(f"{_LIB_PATH} is missing: build it with "
                      "`python -m bit_error_compensated_gb300.build` (needs nvcc)")
_lib = ctypes.CDLL(str(_LIB_PATH))

ECHO_OK = 0
ECHO_ERR_ARG = 1
ECHO_ERR_SHAPE = 2
ECHO_ERR_UNSUPPORTED = 3
ECHO_ERR_ALIGN = 4
ECHO_ERR_CUDA = 5
ECHO_ERR_OVERFLOW = 6
ECHO_ERR_TIMEOUT = 7
ECHO_ERR_TOO_LARGE = 8
ECHO_NOALLOC_SCRATCH_BYTES = 32 << 20
ECHO_MAX_RANKS = 16
ECHO_QUANT_ZERO_AWARE = 0
ECHO_QUANT_NAIVE_ZERO_POINT = 1
ECHO_QUANT_SYMMETRIC = 2
ECHO_TILE_OFF = 0
ECHO_TILE_AUTO = 1
ECHO_TILE_RANK_LOOP = 2
ECHO_TILE_RANK_PARALLEL = 3
ECHO_STATE_F32 = 0
ECHO_STATE_BF16 = 1
ECHO_STATE_F16 = 2
COMP_DEFAULT = ctypes.c_void_p(-1 & (2 ** 64 - 1))   # ECHO_COMP_DEFAULT

_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "echo_plan": (_i32, [_i32, _i64, _i32, _i32, ctypes.POINTER(_vp)]),
    "echo_allreduce": (_i32, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, _vp]),
    "echo_reset_comp": (_i32, [_vp]),
    "echo_reset_comp_async": (_i32, [_vp, _vp, _vp]),
    "echo_comp_bytes": (_sz, [_vp]),
    "echo_wire_bytes": (_sz, [_vp]),
    "echo_wire_layout": (_i32, [_vp, ctypes.POINTER(_i64)]),
    "echo_get_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32)]),
    "echo_debug_wire": (_i32, [_vp, _vp, _sz, _vp]),
    "echo_set_fused": (_i32, [_vp, _i32]),
    "echo_set_timing": (_i32, [_vp, ctypes.POINTER(_vp), _i32]),
    "echo_set_quantizer": (_i32, [_vp, _i32]),
    "echo_set_state": (_i32, [_vp, _i32, ctypes.c_float]),
    "echo_set_persistent": (_i32, [_vp, _i32]),
    "echo_set_tile_fused": (_i32, [_vp, _i32]),
    "echo_debug_hold_push": (_i32, [_vp, _i64]),
    "echo_debug_set_grid": (_i32, [_vp, _i32]),
    "echo_debug_check_guards": (_i32, [_vp, ctypes.POINTER(_i32)]),
    "echo_allreduce_noalloc": (_i32, [_i32, _i64, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                      _vp, _vp]),
    "echo_plan_destroy": (None, [_vp]),
    "echo_strerror": (ctypes.c_char_p, [_i32]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


class EchoError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {_lib.echo_strerror(status).decode()} (status {status})")


def _check(status: int, call: str):
    if status != ECHO_OK:
        raise EchoError(status, call)


def _ptr(x) -> int | None:
    """A device pointer from a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, ctypes.c_void_p):
        return x.value
    return x.data_ptr()


def _tensor_ptrs(*args) -> list:
    """_ptr over (buffer, name, dtypes, min_numel) tuples, with the checks a
    torch tensor allows: the dtype, contiguous, large enough -- for every
    buffer first -- then on a CUDA device.  Raw addresses pass unchecked."""
    import torch
    tensors = [a for a in args if isinstance(a[0], torch.Tensor)]
    for t, what, dtypes, min_numel in tensors:
        if t.dtype not in dtypes:
            raise ValueError(f"{what}: dtype {t.dtype}, expected {' or '.join(map(str, dtypes))}")
        if not t.is_contiguous():
            raise ValueError(f"{what}: tensor must be contiguous")
        if t.numel() < min_numel:
            raise ValueError(f"{what}: {t.numel()} elements, at least {min_numel} needed")
    for t, what, _, _ in tensors:
        if not t.is_cuda:
            raise ValueError(f"{what}: tensor must be on a CUDA device")
    return [_ptr(a[0]) for a in args]


def _buffers(P: int, n: int, ins, outs, comp_state, state_fmt: int):
    """Checked pointers of one call's P inputs, P outputs and state."""
    if len(ins) != P or len(outs) != P:
        raise ValueError(f"expected {P} input and {P} output buffers")
    bf = _bf16()
    args = ([(t, f"in[{p}]", bf, n) for p, t in enumerate(ins)]
            + [(t, f"out[{p}]", bf, n) for p, t in enumerate(outs)]
            + [(None if comp_state is COMP_DEFAULT else comp_state, "comp_state",
                _state_dtypes(state_fmt), P * n)])
    ptrs = _tensor_ptrs(*args)
    comp = COMP_DEFAULT if comp_state is COMP_DEFAULT else ptrs[2 * P]
    return (_vp * P)(*ptrs[:P]), (_vp * P)(*ptrs[P:2 * P]), comp


def _bf16():
    import torch
    return (torch.bfloat16,)


def _state_dtypes(fmt: int):
    import torch
    return ((torch.float32,), (torch.bfloat16,), (torch.float16,))[fmt]


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owning handle of an echo_plan_t; frees the plan when collected."""

    def __init__(self, handle: int, P: int, n: int, g: int, bits: int):
        self.handle = handle
        self.P, self.n, self.g, self.bits = P, n, g, bits
        self.state_fmt = ECHO_STATE_F32          # kept in step with echo_set_state

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            _lib.echo_plan_destroy(h)

    @property
    def _as_parameter_(self):
        return ctypes.c_void_p(self.handle)


def echo_plan(P: int, n: int, g: int = 128, bits: int = 4) -> Plan:
    h = _vp()
    _check(_lib.echo_plan(P, n, g, bits, ctypes.byref(h)), "echo_plan")
    return Plan(h.value, P, n, g, bits)


def echo_allreduce(plan: Plan, ins, outs, comp_state=None, stream=None) -> None:
    """ins/outs: sequences of P device tensors (or int addresses); comp_state:
    None (uncompensated), COMP_DEFAULT (the plan's own state) or a device
    buffer of echo_comp_bytes(plan) bytes."""
    arr_in, arr_out, comp = _buffers(plan.P, plan.n, ins, outs, comp_state, plan.state_fmt)
    _check(_lib.echo_allreduce(plan, arr_in, arr_out, comp, _stream(stream)), "echo_allreduce")


class PreparedCall:
    """echo_allreduce with its buffers checked and marshalled once, for a loop
    that repeats one call on the same buffers (an all-reduce site of a model,
    a benchmark): calling it issues only the C call, without re-checking the
    2P + 1 buffers (about 1 us a buffer in Python), which is what dominates the
    cost of a call on a small message.  It keeps references to the buffers so
    that they stay allocated; their addresses are taken once, so a buffer must
    not be resized or re-pointed while the prepared call is in use.  Calling it
    after the plan's state format changed, or after the plan was destroyed,
    raises ValueError."""

    __slots__ = ("plan", "_keep", "_fmt", "_args")

    def __init__(self, plan: Plan, ins, outs, comp_state=None):
        arr_in, arr_out, comp = _buffers(plan.P, plan.n, ins, outs, comp_state, plan.state_fmt)
        self.plan = plan
        self._keep = (tuple(ins), tuple(outs), comp_state)
        self._fmt = plan.state_fmt
        self._args = (_vp(plan.handle), arr_in, arr_out, comp)

    def __call__(self, stream=None) -> None:
        if self.plan.handle is None or self.plan.handle != self._args[0].value:
            raise ValueError("prepared call: its plan was destroyed")
        if self.plan.state_fmt != self._fmt:
            raise ValueError("prepared call: the plan's state format changed; prepare it again")
        _check(_lib.echo_allreduce(*self._args, _stream(stream)), "echo_allreduce")


def prepare_allreduce(plan: Plan, ins, outs, comp_state=None) -> PreparedCall:
    """A PreparedCall of echo_allreduce(plan, ins, outs, comp_state)."""
    return PreparedCall(plan, ins, outs, comp_state)


def echo_reset_comp(plan: Plan) -> None:
    _check(_lib.echo_reset_comp(plan), "echo_reset_comp")


def echo_reset_comp_async(plan: Plan, comp_state=COMP_DEFAULT, stream=None) -> None:
    comp = COMP_DEFAULT if comp_state is COMP_DEFAULT else _tensor_ptrs(
        (comp_state, "comp_state", _state_dtypes(plan.state_fmt), plan.P * plan.n))[0]
    _check(_lib.echo_reset_comp_async(plan, comp, _stream(stream)), "echo_reset_comp_async")


def echo_comp_bytes(plan: Plan) -> int:
    return int(_lib.echo_comp_bytes(plan))


def echo_wire_bytes(plan: Plan) -> int:
    return int(_lib.echo_wire_bytes(plan))


def echo_wire_layout(plan: Plan) -> dict:
    d = (_i64 * 8)()
    _check(_lib.echo_wire_layout(plan, d), "echo_wire_layout")
    keys = ("codes1", "meta1", "codes2", "meta2", "Gs", "Gs_pad", "code_bytes", "total")
    return dict(zip(keys, [int(v) for v in d]))


def echo_get_status(plan: Plan, stream=None) -> int:
    st = _i32(0)
    _check(_lib.echo_get_status(plan, _stream(stream), ctypes.byref(st)), "echo_get_status")
    return st.value


def echo_debug_wire(plan: Plan, stream=None) -> bytes:
    nbytes = echo_wire_bytes(plan)
    buf = (ctypes.c_uint8 * max(nbytes, 1))()
    _check(_lib.echo_debug_wire(plan, buf, nbytes, _stream(stream)), "echo_debug_wire")
    return bytes(buf)[:nbytes]


def echo_set_fused(plan: Plan, fused: bool) -> None:
    _check(_lib.echo_set_fused(plan, 1 if fused else 0), "echo_set_fused")


def echo_set_quantizer(plan: Plan, mode: int) -> None:
    _check(_lib.echo_set_quantizer(plan, mode), "echo_set_quantizer")


def echo_set_state(plan: Plan, fmt: int = ECHO_STATE_F32, decay: float = 1.0) -> None:
    _check(_lib.echo_set_state(plan, fmt, decay), "echo_set_state")
    plan.state_fmt = fmt


def echo_set_tile_fused(plan: Plan, on: int) -> None:
    """on: ECHO_TILE_OFF/AUTO/RANK_LOOP/RANK_PARALLEL; False and True mean OFF and AUTO."""
    _check(_lib.echo_set_tile_fused(plan, int(on)), "echo_set_tile_fused")


def echo_set_persistent(plan: Plan, on: bool) -> None:
    _check(_lib.echo_set_persistent(plan, 1 if on else 0), "echo_set_persistent")


def echo_debug_hold_push(plan: Plan, item: int) -> None:
    _check(_lib.echo_debug_hold_push(plan, item), "echo_debug_hold_push")


def echo_debug_set_grid(plan: Plan, blocks: int) -> None:
    _check(_lib.echo_debug_set_grid(plan, blocks), "echo_debug_set_grid")


def echo_debug_check_guards(plan: Plan) -> bool:
    intact = ctypes.c_int(0)
    _check(_lib.echo_debug_check_guards(plan, ctypes.byref(intact)), "echo_debug_check_guards")
    return bool(intact.value)


def echo_set_timing(plan: Plan, events) -> None:
    """events: four torch.cuda.Event (enable_timing=True), or None to disable."""
    if not events:
        _check(_lib.echo_set_timing(plan, None, 0), "echo_set_timing")
        return
    arr = (_vp * 4)(*[ev.cuda_event for ev in events])
    _check(_lib.echo_set_timing(plan, arr, 4), "echo_set_timing")


def echo_allreduce_noalloc(P: int, n: int, bits: int, ins, outs, comp_state=None,
                           stream=None) -> None:
    """The no-allocation call (see include/echo.h): no plan, receive slots in
    the library's fixed device array; comp_state is None or a caller buffer."""
    arr_in, arr_out, comp = _buffers(P, n, ins, outs, comp_state, ECHO_STATE_F32)
    _check(_lib.echo_allreduce_noalloc(P, n, bits, arr_in, arr_out, comp,
                                       _stream(stream)), "echo_allreduce_noalloc")


def echo_plan_destroy(plan: Plan) -> None:
    h, plan.handle = plan.handle, None
    if h:
        _lib.echo_plan_destroy(h)


def echo_strerror(status: int) -> str:
    return _lib.echo_strerror(status).decode()


def library_path() -> str:
    return str(_LIB_PATH)
