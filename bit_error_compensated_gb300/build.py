"""Build libecho.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit is compiled in parallel to an object file, then
linked into ``bit_error_compensated_gb300/lib/libecho.so``.  No fast-math: the
kernels rely on IEEE fp32 division and explicit round-to-nearest intrinsics.

    python -m bit_error_compensated_gb300.build [--ptxas-verbose]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
LIBDIR = PKG / "lib"
LIB = LIBDIR / "libecho.so"
# (source, group size it is compiled for, or None).  Every kernel source is
# compiled once per supported group size; the objects compile in parallel.
GROUPS = (64, 128, 256)
SOURCES = [("echo_api.cu", None), ("echo_noalloc.cu", None)] + [
    (src, g) for src in ("k_push.cu", "k_reduce.cu", "k_gather.cu", "k_call.cu", "k_tile.cu")
    for g in GROUPS]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libecho.so")


def _flags(ptxas_verbose: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I", str(ROOT / "include"), "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    # tuning overrides, e.g. ECHO_NVCC_FLAGS="-DECHO_REDUCE_TILE=16"
    f += os.environ.get("ECHO_NVCC_FLAGS", "").split()
    return f


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = [CSRC / s for s, _ in SOURCES] + list(CSRC.glob("*.h")) + list(CSRC.glob("*.cuh"))
    deps.append(ROOT / "include" / "echo.h")
    return any(d.stat().st_mtime > t for d in deps)


def build_library(force: bool = False, ptxas_verbose: bool = False) -> Path:
    if not (force or ptxas_verbose or _stale()):
        return LIB
    cc = nvcc()
    objdir = ROOT / "_build" / "echo"
    objdir.mkdir(parents=True, exist_ok=True)
    LIBDIR.mkdir(exist_ok=True)
    procs = []
    for src, g in SOURCES:
        stem = Path(src).stem + ("" if g is None else f"_g{g}")
        obj = objdir / (stem + ".o")
        defs = [] if g is None else [f"-DECHO_G={g}"]
        cmd = [cc, *_flags(ptxas_verbose), *defs, "-c", str(CSRC / src), "-o", str(obj)]
        procs.append((stem, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, obj, pr in procs:
        out, _ = pr.communicate()
        if out.strip():
            sys.stderr.write(f"--- {src}\n{out}")
        if pr.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    tmp = LIB.with_suffix(f".so.tmp{os.getpid()}")
    subprocess.check_call([cc, *ARCH, "-shared", "-o", str(tmp), *[str(o) for _, o, _ in procs],
                           "-lcudart"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build_library(force=True, ptxas_verbose="--ptxas-verbose" in sys.argv)
    print(LIB)
