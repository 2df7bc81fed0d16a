// echo_noalloc.cu -- echo_allreduce_noalloc: the emulated all-reduce for
// callers that must not allocate device memory (contract in include/echo.h).
//
// The receive slots that the push kernel writes and the reduce kernel reads
// (and writes its gather codes to) live in a file-scope __device__ array instead of a plan's
// cudaMalloc'd workspace.  Host code never passes the array's name to a kernel
// (on the host it is only a stand-in symbol): the device address is looked up
// once per device with cudaGetSymbolAddress and passed as a plain pointer.
// The kernels and their launchers are the ones echo_allreduce uses.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "echo_internal.h"

namespace {

// Status word (first 256 bytes) followed by the receive slots.
static __device__ __align__(256) uint8_t g_noalloc_scratch[ECHO_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
uint8_t* g_scratch_addr[kMaxDevices] = {nullptr};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool overlap(uintptr_t a, uintptr_t b, size_t bytes) { return a < b + bytes && b < a + bytes; }

// Device address of the scratch array on the current device, looked up (and
// the kernels' attributes set) on the first call there.
int scratch_for_current_device(uint8_t** base) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return echo::note_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return ECHO_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return echo::note_cuda_error(e);
    e = echo::prepare_kernels();
    if (e != cudaSuccess) return echo::note_cuda_error(e);
    g_scratch_addr[dev] = static_cast<uint8_t*>(p);
  }
  *base = g_scratch_addr[dev];
  return ECHO_OK;
}

}  // namespace

extern "C" int echo_allreduce_noalloc(int P, int64_t n, int bits, const void* const* in,
                                      void* const* out, void* comp_state, void* stream) {
  if (in == nullptr || out == nullptr) return ECHO_ERR_ARG;
  if (P < 1 || P > ECHO_MAX_RANKS) return ECHO_ERR_ARG;
  if (bits != 4 && bits != 8) return ECHO_ERR_UNSUPPORTED;
  if (n < 0 || n % ((int64_t)P * echo::kGroup) != 0) return ECHO_ERR_SHAPE;
  if (comp_state == ECHO_COMP_DEFAULT) return ECHO_ERR_ARG;
  // Every element needs at least b/8 bytes of gather codes in the array, so a
  // larger n can never fit; rejecting it first also keeps the layout sums
  // below far from any overflow.
  if (n > (int64_t)(ECHO_NOALLOC_SCRATCH_BYTES * 8 / bits)) return ECHO_ERR_TOO_LARGE;

  // Receive-slot layout, the same as a plan's (see echo_wire_layout).
  const int64_t Gs = n / P / echo::kGroup;
  const int64_t Gs_pad = (Gs + 3) / 4 * 4;
  const int64_t CB = (int64_t)echo::kGroup * bits / 8;
  const size_t off_codes1 = 256;                              // after the status word
  const size_t off_meta1 = round256(off_codes1 + (size_t)P * (P - 1) * Gs * CB);
  const size_t off_codes2 = round256(off_meta1 + (size_t)P * (P - 1) * Gs_pad * 4);
  const size_t off_meta2 = round256(off_codes2 + (size_t)P * Gs * CB);
  const size_t total = round256(off_meta2 + (size_t)P * Gs_pad * 4);
  if (total > ECHO_NOALLOC_SCRATCH_BYTES) return ECHO_ERR_TOO_LARGE;

  const size_t bytes = (size_t)n * 2;
  const size_t comp_bytes = (size_t)P * n * sizeof(float);
  for (int p = 0; p < P; ++p) {
    if (in[p] == nullptr || out[p] == nullptr) return ECHO_ERR_ARG;
    if (!aligned16(in[p]) || !aligned16(out[p])) return ECHO_ERR_ALIGN;
  }
  if (comp_state != nullptr && ((uintptr_t)comp_state & 31u) != 0) return ECHO_ERR_ALIGN;
  for (int p = 0; p < P; ++p) {            // same aliasing rules as echo_allreduce
    const uintptr_t op = (uintptr_t)out[p];
    for (int q = 0; q < P; ++q) {
      const uintptr_t iq = (uintptr_t)in[q];
      if (op == iq && p == q) continue;
      if (overlap(op, iq, bytes)) return ECHO_ERR_ARG;
      if (q != p && overlap(op, (uintptr_t)out[q], bytes)) return ECHO_ERR_ARG;
    }
    if (comp_state != nullptr && comp_bytes > 0) {
      const uintptr_t c = (uintptr_t)comp_state;
      if (c < op + bytes && op < c + comp_bytes) return ECHO_ERR_ARG;
      if (c < (uintptr_t)in[p] + bytes && (uintptr_t)in[p] < c + comp_bytes) return ECHO_ERR_ARG;
    }
  }

  uint8_t* base = nullptr;
  int rc = scratch_for_current_device(&base);
  if (rc != ECHO_OK) return rc;
  if (n == 0) return ECHO_OK;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  echo::CallArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int p = 0; p < P; ++p) {
    a.in[p] = static_cast<const __nv_bfloat16*>(in[p]);
    a.out[p] = static_cast<__nv_bfloat16*>(out[p]);
  }
  a.comp = static_cast<float*>(comp_state);
  a.status = reinterpret_cast<int*>(base);
  a.codes1 = base + off_codes1;
  a.meta1 = reinterpret_cast<uint32_t*>(base + off_meta1);
  a.codes2 = base + off_codes2;
  a.meta2 = reinterpret_cast<uint32_t*>(base + off_meta2);
  a.n = n;
  a.Gs = Gs;
  a.Gs_pad = Gs_pad;
  a.P = P;
  a.state_fmt = 0;             // fp32 state, plain error feedback
  a.decay = 1.0f;

  // The kernels only OR flags into the status word; it is the one part of the
  // array that must start at zero.  The receive slots are fully rewritten by
  // every call before they are read.
  cudaError_t e = cudaMemsetAsync(a.status, 0, sizeof(int), s);
  if (e == cudaSuccess && P > 1) e = echo::launch_push(a, echo::kGroup, bits, s, true);
  // The reduce kernel writes the P outputs itself (the fused gather).
  if (e == cudaSuccess) e = echo::launch_reduce(a, echo::kGroup, bits, true, s, true);
  if (e != cudaSuccess) return echo::note_cuda_error(e);
  return ECHO_OK;
}
