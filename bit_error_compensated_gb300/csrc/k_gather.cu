// k_gather.cu -- the gather of the quantized P2P all-reduce ("Echo: Error-
// Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)): every rank,
// the owner included, decodes the same gather codes of every segment, so all
// P outputs hold identical bits.  With the ranks in one GPU's memory, the
// all-gather is one read of each segment's codes and P writes of the decoded
// bf16 values.
//
// One warp per group, 4 elements per lane: a warp reads 64 B (4-bit) or 128 B
// (8-bit) of codes plus one meta word and writes P x 256 B of bf16 with
// streaming stores.  U groups per warp are read before any is written, to keep
// several code reads in flight.  Write-bound: P * 2 bytes out per element.
#include "echo_internal.h"
#include "quant.cuh"

namespace echo {
namespace {

template <int BITS, int U>
__global__ void __launch_bounds__(kThreads)
gather_kernel(const CallArgs a) {
  constexpr int CB = 16 * BITS;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarp = ((int64_t)gridDim.x * kThreads) >> 5;
  const int P = a.P;
  const int64_t W = (int64_t)P * a.Gs;    // groups of one rank tensor

  for (int64_t base = warp; base < W; base += nwarp * U) {
    uint32_t word[U], meta[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t w = base + (int64_t)u * nwarp;
      if (w < W) {
        const int64_t o = w / a.Gs;
        const int64_t j = w - o * a.Gs;
        meta[u] = a.meta2[o * a.Gs_pad + j];
        if (BITS == 4) {
          word[u] = reinterpret_cast<const uint16_t*>(a.codes2 + w * CB)[lane];
        } else {
          word[u] = reinterpret_cast<const uint32_t*>(a.codes2 + w * CB)[lane];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t w = base + (int64_t)u * nwarp;
      if (w >= W) break;                      // warp-uniform
      float s;
      int z;
      unpack_meta(meta[u], s, z);
      int q[4];
      unpack4<BITS>(word[u], q);
      float deq[4], yb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) deq[k] = decode(q[k], z, s);
      const uint2 y = f32x4_to_bf16(deq, yb);
      const int64_t elem = w * kGroup + 4 * lane;
      for (int r = 0; r < P; ++r) __stcs(reinterpret_cast<uint2*>(a.out[r] + elem), y);
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kGatherUnroll = 4;

template <int BITS>
cudaError_t launch_t(const CallArgs& a, cudaStream_t s, bool pdl) {
  static int grid_cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int& grid = grid_cache[dev & 63];
  if (grid == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_kernel<BITS, kGatherUnroll>,
                                                  kThreads, 0);
    grid = sms * (per_sm > 0 ? per_sm : 1);
  }
  const int64_t W = (int64_t)a.P * a.Gs;
  const int64_t warps_needed = (W + kGatherUnroll - 1) / kGatherUnroll;
  const int64_t blocks_needed = (warps_needed + (kThreads / 32) - 1) / (kThreads / 32);
  const int blocks = (int)(blocks_needed < grid ? blocks_needed : grid);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gather_kernel<BITS, kGatherUnroll>, a);
}

}  // namespace

cudaError_t launch_gather(const CallArgs& a, int bits, cudaStream_t s, bool pdl) {
  return bits == 4 ? launch_t<4>(a, s, pdl) : launch_t<8>(a, s, pdl);
}

}  // namespace echo
