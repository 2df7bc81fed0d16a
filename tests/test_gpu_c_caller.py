"""A C program as the library's only user on the GPU: no Python, no torch in
its process.  It allocates its buffers with cudaMalloc, fills the P ranks'
bf16 inputs from a seeded generator of its own, runs one uncompensated and two
compensated echo_allreduce calls on its own state buffer through the C ABI of
include/echo.h, and writes every call's inputs and outputs and the final state
to a file, which is then checked here against the oracle: outputs bit for
bit, state within STATE_RTOL."""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

import oracle
from _parity import assert_state_close

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent
CUDA = Path("/usr/local/cuda")
P, G, GS, CALLS = 4, 128, 50, 3
N = P * G * GS

C_PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "echo.h"

#define P %(P)d
#define N %(N)d
#define CALLS %(CALLS)d

static uint64_t rng = 0x9E3779B97F4A7C15ull;
static uint32_t next32(void) {            /* xorshift64* */
  rng ^= rng >> 12; rng ^= rng << 25; rng ^= rng >> 27;
  return (uint32_t)((rng * 0x2545F4914F6CDD1Dull) >> 32);
}

#define CHECK(x) do { int rc_ = (x); if (rc_) { fprintf(stderr, "%%s: %%d (%%s)\n", #x, rc_, \
    echo_strerror(rc_)); return 1; } } while (0)
#define CUDA_OK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { fprintf(stderr, \
    "%%s: %%s\n", #x, cudaGetErrorString(e_)); return 1; } } while (0)

int main(int argc, char** argv) {
  if (argc != 2) return 2;
  FILE* f = fopen(argv[1], "wb");
  if (!f) return 2;
  static uint16_t host[P][N];
  static float state[P][N];
  void* in[P];
  void* out[P];
  void* comp = NULL;
  for (int p = 0; p < P; ++p) {
    CUDA_OK(cudaMalloc(&in[p], N * sizeof(uint16_t)));
    CUDA_OK(cudaMalloc(&out[p], N * sizeof(uint16_t)));
  }
  CUDA_OK(cudaMalloc(&comp, (size_t)P * N * sizeof(float)));
  CUDA_OK(cudaMemset(comp, 0, (size_t)P * N * sizeof(float)));
  echo_plan_t plan = NULL;
  CHECK(echo_plan(P, N, 128, 4, &plan));
  for (int k = 0; k < CALLS; ++k) {
    for (int p = 0; p < P; ++p) {
      for (int i = 0; i < N; ++i) {
        /* a bf16 with a random sign, an exponent in [2^-6, 2^5) and mantissa */
        uint32_t r = next32();
        host[p][i] = (uint16_t)((r & 0x807Fu) | ((121u + (r >> 8) %% 11u) << 7));
      }
      CUDA_OK(cudaMemcpy(in[p], host[p], N * sizeof(uint16_t), cudaMemcpyHostToDevice));
    }
    fwrite(host, sizeof(uint16_t), (size_t)P * N, f);
    CHECK(echo_allreduce(plan, (const void* const*)in, out, k == 0 ? NULL : comp, NULL));
    CUDA_OK(cudaDeviceSynchronize());
    for (int p = 0; p < P; ++p)
      CUDA_OK(cudaMemcpy(host[p], out[p], N * sizeof(uint16_t), cudaMemcpyDeviceToHost));
    fwrite(host, sizeof(uint16_t), (size_t)P * N, f);
  }
  int status = -1;
  CHECK(echo_get_status(plan, NULL, &status));
  CUDA_OK(cudaMemcpy(state, comp, (size_t)P * N * sizeof(float), cudaMemcpyDeviceToHost));
  fwrite(state, sizeof(float), (size_t)P * N, f);
  fclose(f);
  echo_plan_destroy(plan);
  for (int p = 0; p < P; ++p) {
    cudaFree(in[p]);
    cudaFree(out[p]);
  }
  cudaFree(comp);
  printf("status %%d\n", status);
  return 0;
}
""" % dict(P=P, N=N, CALLS=CALLS)


def test_a_c_program_runs_the_call_through_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from bit_error_compensated_gb300.build import build_library
    lib = build_library()
    src = tmp_path / "caller.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "caller"
    subprocess.run([cc, "-std=c11", "-O2", "-Wall", "-Werror", "-I", str(ROOT / "include"),
                    "-I", str(CUDA / "include"), str(src), "-o", str(exe),
                    "-L", str(lib.parent), "-lecho", f"-Wl,-rpath,{lib.parent}",
                    "-L", str(CUDA / "lib64"), "-lcudart", f"-Wl,-rpath,{CUDA / 'lib64'}"],
                   check=True, capture_output=True, text=True)
    data = tmp_path / "calls.bin"
    run = subprocess.run([str(exe), str(data)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.stdout, run.stderr)
    assert run.stdout.strip() == "status 0"
    raw = np.fromfile(data, np.uint8)
    per_call = 2 * P * N * 2
    assert raw.size == CALLS * per_call + P * N * 4
    e = np.zeros((P, N), np.float32)
    for k in range(CALLS):
        blob = raw[k * per_call:(k + 1) * per_call].view(np.uint16)
        x, y = blob[:P * N].reshape(P, N), blob[P * N:].reshape(P, N)
        ref = oracle.allreduce(x, G, 4, e=None if k == 0 else e)
        assert np.array_equal(y, ref["out"]), f"outputs differ from the oracle at call {k}"
    state = raw[CALLS * per_call:].view(np.float32).reshape(P, N)
    assert_state_close(state, e, "state after the last call")
