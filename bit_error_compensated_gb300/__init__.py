"""Echo emulated 4-bit error-compensated all-reduce, native to one GB300 (sm_103a).

The compute path is the C-ABI library ``libecho.so`` (hand-written CUDA kernels);
``bit_error_compensated_gb300.echo`` is its thin ctypes binding, loaded on first
use and failing loudly when the library has not been built.  ``workloads`` holds
the seeded synthetic input generators.
"""
_BINDING_NAMES = (
    "echo_plan", "echo_allreduce", "echo_reset_comp", "echo_reset_comp_async",
    "echo_comp_bytes", "echo_wire_bytes", "echo_wire_layout", "echo_get_status",
    "echo_debug_wire", "echo_plan_destroy", "echo_strerror", "echo_set_fused",
    "echo_set_timing", "echo_set_quantizer", "echo_allreduce_noalloc", "Plan", "EchoError",
    "COMP_DEFAULT",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import echo
        return getattr(echo, name)
    raise AttributeError(name)
