"""The C-ABI library builds, loads, and exports every entry point include/echo.h
declares; host-side argument checks that need no GPU."""
import ctypes
import re
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADERS = sorted((ROOT / "include").glob("*.h"))


def _declared():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(echo_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from bit_error_compensated_gb300.build import build_library
    return ctypes.CDLL(str(build_library()))


def test_headers_declare_the_three_named_calls():
    d = _declared()
    assert {"echo_plan", "echo_allreduce", "echo_reset_comp"} <= d
    assert len(d) >= 12


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_wraps_every_declared_call(lib):
    from bit_error_compensated_gb300 import echo
    assert set(echo.EXPORTED) == _declared()
    assert echo.library_path().endswith("libecho.so")


def test_host_argument_checks_without_gpu(lib):
    from bit_error_compensated_gb300 import echo
    h = ctypes.c_void_p()
    lib.echo_plan.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                              ctypes.POINTER(ctypes.c_void_p)]
    # argument errors are reported before any CUDA call
    assert lib.echo_plan(0, 128, 128, 4, ctypes.byref(h)) == echo.ECHO_ERR_ARG
    assert lib.echo_plan(17, 17 * 128, 128, 4, ctypes.byref(h)) == echo.ECHO_ERR_ARG
    assert lib.echo_plan(2, 256, 0, 4, ctypes.byref(h)) == echo.ECHO_ERR_ARG
    assert lib.echo_plan(2, 256, 128, 5, ctypes.byref(h)) == echo.ECHO_ERR_UNSUPPORTED
    assert lib.echo_plan(2, 256, 32, 4, ctypes.byref(h)) == echo.ECHO_ERR_UNSUPPORTED
    assert lib.echo_plan(2, 1024, 512, 4, ctypes.byref(h)) == echo.ECHO_ERR_UNSUPPORTED
    assert lib.echo_plan(2, 300, 128, 4, ctypes.byref(h)) == echo.ECHO_ERR_SHAPE
    assert lib.echo_plan(2, -256, 128, 4, ctypes.byref(h)) == echo.ECHO_ERR_SHAPE
    assert lib.echo_plan(2, 256, 128, 4, None) == echo.ECHO_ERR_ARG
    assert h.value is None
    assert lib.echo_allreduce(None, None, None, None, None) == echo.ECHO_ERR_ARG
    assert lib.echo_reset_comp(None) == echo.ECHO_ERR_ARG
    lib.echo_comp_bytes.restype = ctypes.c_size_t
    assert lib.echo_comp_bytes(None) == 0
    lib.echo_plan_destroy(None)
    for code, word in [(0, "ok"), (2, "multiple"), (4, "aligned"), (7, "wait")]:
        assert word in echo.echo_strerror(code)


def test_comp_default_sentinel_matches_header():
    from bit_error_compensated_gb300 import echo
    text = (ROOT / "include" / "echo.h").read_text()
    assert "#define ECHO_COMP_DEFAULT ((void*)(intptr_t)-1)" in text
    assert echo.COMP_DEFAULT.value == 2 ** 64 - 1
    for name in ("ECHO_OK", "ECHO_ERR_ARG", "ECHO_ERR_SHAPE", "ECHO_ERR_UNSUPPORTED",
                 "ECHO_ERR_ALIGN", "ECHO_ERR_CUDA", "ECHO_ERR_OVERFLOW", "ECHO_ERR_TIMEOUT",
                 "ECHO_ERR_TOO_LARGE", "ECHO_MAX_RANKS", "ECHO_QUANT_ZERO_AWARE",
                 "ECHO_QUANT_NAIVE_ZERO_POINT", "ECHO_QUANT_SYMMETRIC", "ECHO_STATE_F32",
                 "ECHO_STATE_BF16", "ECHO_STATE_F16"):
        m = re.search(rf"#define {name}\s+(\d+)", text)
        assert m and int(m.group(1)) == getattr(echo, name), name


def test_binding_checks_tensors_before_the_call(lib):
    """The binding turns a tensor into a pointer only when the pointer means
    what the C call assumes: the dtype of the buffer's role, contiguous, at
    least n (state: P*n) elements, on a CUDA device.  A stand-in plan with a
    null handle shows the checks come before any call into the library."""
    import torch
    from bit_error_compensated_gb300 import echo
    P, n = 2, 256
    plan = echo.Plan(0, P, n, 128, 4)
    good = [torch.zeros(n, dtype=torch.bfloat16) for _ in range(P)]

    def rejects(word, ins=good, outs=good, comp=None, noalloc=False):
        with pytest.raises(ValueError, match=word):
            if noalloc:
                echo.echo_allreduce_noalloc(P, n, 4, ins, outs, comp)
            else:
                echo.echo_allreduce(plan, ins, outs, comp)

    rejects("dtype", ins=[torch.zeros(n), good[1]])
    rejects("contiguous", outs=[good[0], torch.zeros(2 * n, dtype=torch.bfloat16)[::2]])
    rejects("at least 256", ins=[good[0], torch.zeros(n - 1, dtype=torch.bfloat16)])
    rejects("CUDA device")                                  # right in every other way
    rejects("expected 2", ins=good[:1])
    rejects("dtype", comp=torch.zeros(P * n, dtype=torch.bfloat16))   # plan holds fp32
    rejects("at least 512", comp=torch.zeros(P * n - 1))
    rejects("dtype", comp=torch.zeros(P * n, dtype=torch.float16), noalloc=True)
    plan.state_fmt = echo.ECHO_STATE_F16                   # as echo_set_state records it
    rejects("dtype", comp=torch.zeros(P * n))
    rejects("CUDA device", comp=torch.zeros(P * n, dtype=torch.float16))
    with pytest.raises(ValueError, match="dtype"):
        echo.echo_reset_comp_async(plan, torch.zeros(P * n))


def test_binding_passes_raw_addresses_and_the_default_state_through(lib, monkeypatch):
    """Integer addresses are the caller's responsibility and reach the C call
    unchanged, as does the ECHO_COMP_DEFAULT sentinel; a stand-in for the C
    entry point records what it was given (no GPU call is made)."""
    from bit_error_compensated_gb300 import echo
    P, n = 2, 256
    plan = echo.Plan(0, P, n, 128, 4)
    seen = {}

    class FakeLib:
        def echo_allreduce(self, plan_, ins, outs, comp, stream):
            seen.update(ins=[ins[i] for i in range(P)], outs=[outs[i] for i in range(P)],
                        comp=comp)
            return 0

    monkeypatch.setattr(echo, "_lib", FakeLib())
    echo.echo_allreduce(plan, [4096, 8192], [12288, 16384], echo.COMP_DEFAULT, stream=0)
    assert seen["ins"] == [4096, 8192] and seen["outs"] == [12288, 16384]
    assert seen["comp"] is echo.COMP_DEFAULT
    echo.echo_allreduce(plan, [4096, 8192], [12288, 16384], 1 << 20, stream=0)
    assert seen["comp"] == 1 << 20
    echo.echo_allreduce(plan, [4096, 8192], [12288, 16384], None, stream=0)
    assert seen["comp"] is None


def test_noalloc_rejects_huge_n_before_any_layout_arithmetic(lib):
    """n so large that the receive-slot sums would wrap around 2^64 must come
    back as ECHO_ERR_TOO_LARGE from the host checks (no CUDA call is made)."""
    from bit_error_compensated_gb300 import echo
    fn = lib.echo_allreduce_noalloc
    fn.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    P = 16
    ptrs = (ctypes.c_void_p * P)(*[0x100000 * (p + 1) for p in range(P)])
    limit = (32 << 20) * 8
    for bits_ in (4, 8):
        for n in (1 << 61, (1 << 62) + P * 128 * 7, (limit // bits_ // (P * 128) + 1) * P * 128):
            assert n % (P * 128) == 0
            assert fn(P, n, bits_, ptrs, ptrs, None, None) == echo.ECHO_ERR_TOO_LARGE


def test_prepared_call_checks_once_and_passes_the_same_arguments(lib, monkeypatch):
    """A prepared call checks its buffers when it is made (the same checks as
    echo_allreduce) and then hands the C call the same pointers every time;
    it refuses to run after the plan's state format changed or the plan is
    gone.  A stand-in for the C entry point records the calls."""
    import torch
    from bit_error_compensated_gb300 import echo
    P, n = 2, 256
    plan = echo.Plan(0x1000, P, n, 128, 4)
    seen = []

    class FakeLib:
        def echo_allreduce(self, plan_, ins, outs, comp, stream):
            seen.append((plan_.value, [ins[i] for i in range(P)], [outs[i] for i in range(P)],
                         comp, stream))
            return 0

        def echo_plan_destroy(self, h):
            pass

        def echo_strerror(self, status):
            return b"x"

    with pytest.raises(ValueError, match="dtype"):
        echo.prepare_allreduce(plan, [torch.zeros(n), torch.zeros(n)], [4096, 8192])
    monkeypatch.setattr(echo, "_lib", FakeLib())
    call = echo.prepare_allreduce(plan, [4096, 8192], [12288, 16384], echo.COMP_DEFAULT)
    call(stream=7)
    call(stream=7)
    assert seen[0] == seen[1] == (0x1000, [4096, 8192], [12288, 16384], echo.COMP_DEFAULT, 7)
    plan.state_fmt = echo.ECHO_STATE_BF16
    with pytest.raises(ValueError, match="state format"):
        call(stream=7)
    plan.state_fmt = echo.ECHO_STATE_F32
    echo.echo_plan_destroy(plan)
    with pytest.raises(ValueError, match="destroyed"):
        call(stream=7)
    assert len(seen) == 2


C_CALLER = r"""
#include <stdio.h>
#include "echo.h"
int main(void) {
  echo_plan_t plan = 0;
  /* rejected before any device work, so this runs without a GPU */
  int rc = echo_plan(0, 0, 128, 4, &plan);
  if (rc != ECHO_ERR_ARG || plan != 0) return 1;
  rc = echo_plan(4, 4 * 128 + 1, 128, 4, &plan);
  if (rc != ECHO_ERR_SHAPE) return 2;
  if (echo_set_tile_fused(0, ECHO_TILE_AUTO) != ECHO_ERR_ARG) return 3;
  printf("%s\n", echo_strerror(ECHO_ERR_ARG));
  return 0;
}
"""


def test_header_compiles_as_c_and_a_c_program_links(tmp_path):
    """include/echo.h is a plain C interface: a C11 program including it builds
    with every warning as an error, links against libecho.so and calls it."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from bit_error_compensated_gb300.build import build_library
    lib = build_library()
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", str(ROOT / "include"), str(src), "-o", str(exe),
                    "-L", str(lib.parent), "-lecho", f"-Wl,-rpath,{lib.parent}"],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.strip() == "invalid argument"

