// echo_internal.h -- types shared by the host side of libecho.so and its
// kernels.  Not part of the public ABI (include/echo.h is).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/echo.h"

namespace echo {

// Elements per quantization group the GPU supports: 64, 128 (the method's
// default) and 256.  Each kernel source is compiled once per group size, with
// ECHO_G set to it.
constexpr int kGroup = 128;
constexpr bool group_supported(int g) { return g == 64 || g == 128 || g == 256; }
// Elements per reduce tile (one thread block of the reduce kernel works on one
// tile at a time): kReduceTileElems / g groups, a multiple of 4 for every
// supported g, so that every tile's meta words form a 16-byte-aligned copy.
// Warps per reduce block: each takes 512 elements of a tile per pass.
#ifndef ECHO_REDUCE_TILE
#define ECHO_REDUCE_TILE 8    // in groups of 128
#endif
#ifndef ECHO_REDUCE_WARPS
#define ECHO_REDUCE_WARPS 2
#endif
constexpr int kReduceTileElems = ECHO_REDUCE_TILE * 128;
constexpr int kReduceWarps = ECHO_REDUCE_WARPS;
static_assert(kReduceTileElems % (4 * 256) == 0, "reduce tile: a multiple of 4 groups of 256");
// Ranks the rank-parallel form of the tile kernel takes (a warp group of
// kReduceWarps warps per rank, at most 1024 threads a block); above it the
// rank loop runs.
constexpr int kTileRpMaxP = 1024 / (32 * kReduceWarps) < ECHO_MAX_RANKS
                                ? 1024 / (32 * kReduceWarps) : ECHO_MAX_RANKS;
// Elements per tile of the persistent kernel: one 512-element unit per warp.
constexpr int kCallTileElems = 4096;
// Threads per block of the push, gather and persistent kernels (the reduce
// kernel's blocks have kReduceWarps warps).
constexpr int kThreads = 256;
// Blocks of 256 threads per SM the register allocation of the unfused reduce
// kernel and the persistent kernel must allow (the reduce kernel scales it to
// its block size; the fused one has its own, higher bound).  3 leaves them up
// to 80 registers a thread, which they use without spilling.
#ifndef ECHO_REDUCE_MIN_BLOCKS
#define ECHO_REDUCE_MIN_BLOCKS 3
#endif

// A launch parameter computed once per device (and key) by the first call:
// threads that race on the first call compute the same value, and the reads
// and writes are atomic.  0 means not yet computed.
struct CachedInt {
  std::atomic<int> v{0};
  int get() const { return v.load(std::memory_order_relaxed); }
  void set(int x) { v.store(x, std::memory_order_relaxed); }
};

// Status-word bits written by the kernels (read by echo_get_status).
constexpr int kStatusOverflow = 1;
constexpr int kStatusTimeout = 2;

// Everything a kernel needs about one call, passed by value.
struct CallArgs {
  const __nv_bfloat16* in[ECHO_MAX_RANKS];   // rank p's input, n elements
  __nv_bfloat16* out[ECHO_MAX_RANKS];        // rank p's output, n elements
  float* comp;         // [P][n] compensator state, or nullptr (uncompensated)
  uint8_t* codes1;     // push codes  [P owners][P-1 senders][Gs][CB]
  uint32_t* meta1;     // push meta   [P owners][P-1 senders][Gs_pad]
  uint8_t* codes2;     // gather codes [P owners][Gs][CB]
  uint32_t* meta2;     // gather meta  [P owners][Gs_pad]
  int* status;         // device status word
  int64_t n;           // elements per rank
  int64_t Gs;          // groups per owner segment (m / g)
  int64_t Gs_pad;      // Gs rounded up to a multiple of 4
  int P;
  int mode;            // quantizer: 0 zero-aware (the method), 1 naive zero point, 2 symmetric
  int state_fmt;       // format of the state at comp: 0 fp32, 1 bf16, 2 fp16
  float decay;         // the kept error is decay * (revealed error); 1 = plain feedback
  int grid_cap;        // debug: at most this many blocks along each kernel's grid (0: none)
};

// The schedule of the single persistent kernel of a call (k_call.cu).
struct CallSched {
  int64_t tiles;          // reduce tiles per owner segment
  int64_t round;          // tickets per round (set by the launcher)
  int64_t lag;            // D: round r reduces tile r - D, gathers tile r - 2D (launcher)
  int64_t total;          // tickets of the call (launcher)
  int64_t hold;           // test hook: this push ticket never reports completion; -1 none
  uint32_t* push_done;    // [P][tiles] pushes of the tile finished in this call
  uint32_t* reduce_done;  // [P][tiles] the tile's reduce finished in this call
  uint32_t* ctrl;         // [0] ticket counter, [1] blocks finished, [2] abort
};
// 32-bit words of a plan's schedule area.
inline int64_t sched_words(int P, int64_t tiles) { return 2 * (int64_t)P * tiles + 4; }

// Launchers for group size G, defined in the translation unit compiled with
// ECHO_G = G.  They return the launch error.
template <int G> cudaError_t launch_push_g(const CallArgs& a, int bits, cudaStream_t s, bool pdl);
template <int G>
cudaError_t launch_reduce_g(const CallArgs& a, int bits, bool fused, cudaStream_t s, bool pdl);
template <int G> cudaError_t launch_gather_g(const CallArgs& a, int bits, cudaStream_t s, bool pdl);
// One-time per-device set-up of the reduce kernels' attributes (dynamic
// shared memory) for group size G.
template <int G> cudaError_t prepare_reduce_g();

template <int G>
cudaError_t launch_call_g(const CallArgs& a, const CallSched& sch, int bits, bool fused,
                          cudaStream_t s);
template <int G>
cudaError_t launch_tile_g(const CallArgs& a, int bits, bool rank_parallel, cudaStream_t s, bool pdl);
// One-time per-device set-up of the rank-parallel tile kernels' attributes.
template <int G> cudaError_t prepare_tile_g();

// Dispatch on the group size g (defined in echo_api.cu, which sees only the
// declarations above, so each kernel source instantiates its own g alone).
cudaError_t launch_push(const CallArgs& a, int g, int bits, cudaStream_t s, bool pdl);
cudaError_t launch_reduce(const CallArgs& a, int g, int bits, bool fused, cudaStream_t s, bool pdl);
cudaError_t launch_gather(const CallArgs& a, int g, int bits, cudaStream_t s, bool pdl);
cudaError_t launch_call(const CallArgs& a, const CallSched& sch, int g, int bits, bool fused,
                        cudaStream_t s);
cudaError_t launch_tile(const CallArgs& a, int g, int bits, bool rank_parallel, cudaStream_t s,
                        bool pdl);
// Attributes of every reduce and rank-parallel tile kernel, all group sizes.
cudaError_t prepare_kernels();
// Records `e` as the error echo_strerror(ECHO_ERR_CUDA) reports in this thread
// and returns ECHO_ERR_CUDA.
int note_cuda_error(cudaError_t e);

}  // namespace echo
