// k_push.cu -- the push of the quantized P2P all-reduce ("Echo: Error-
// Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)): every rank
// quantizes each segment it does not own and sends the codes to the owner.
// With the ranks emulated in one GPU's memory, "sending" is writing the codes
// and the per-group meta word into the owner's receive slot for that sender.
//
// The compensator's entry pass is fused in: the rank's held error for the
// element is added before quantizing, and the error this quantization reveals,
// v - deq(q), replaces it (the update changes nothing this call computes).
//
// Work unit: one group of 128 elements of one rank's non-owned segment, one
// warp per group, 4 consecutive elements per lane, so each warp-wide access is
// contiguous: 256 B of bf16 input, 512 B of fp32 state, 64 B (4-bit) or 128 B
// (8-bit) of codes.  U groups per warp are loaded before any is processed to
// keep enough bytes in flight for HBM.  HBM-bound: per group the kernel reads
// 256 B + 512 B and writes 512 B + codes + 4 B of meta.
#include "echo_internal.h"
#include "quant.cuh"

namespace echo {
namespace {

template <int BITS, bool COMP, int U>
__global__ void __launch_bounds__(kThreads)
push_kernel(const CallArgs a) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr int CB = 16 * BITS;                 // code bytes per group
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarp = ((int64_t)gridDim.x * kThreads) >> 5;
  const int P = a.P;
  const int64_t Gs = a.Gs;
  const int64_t per_rank = (int64_t)(P - 1) * Gs;  // non-owned groups of a rank
  const int64_t W = (int64_t)P * per_rank;

  for (int64_t base = warp; base < W; base += nwarp * U) {
    float v[U][4];
    int64_t elem[U];      // first element of the group within the rank's tensor
    int64_t dst[U];       // group index in the push-code array
    int64_t midx[U];      // index in the push-meta array
    int prank[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t w = base + (int64_t)u * nwarp;
      prank[u] = -1;
      if (w < W) {
        const int p = (int)(w / per_rank);
        const int64_t r = w - (int64_t)p * per_rank;
        const int oi = (int)(r / Gs);
        const int64_t j = r - (int64_t)oi * Gs;
        const int o = oi + (oi >= p ? 1 : 0);         // owner of the segment
        const int slot = o * (P - 1) + (p < o ? p : p - 1);
        prank[u] = p;
        elem[u] = ((int64_t)o * Gs + j) * kGroup + 4 * lane;
        dst[u] = (int64_t)slot * Gs + j;
        midx[u] = (int64_t)slot * a.Gs_pad + j;
        const uint2 xr = __ldcs(reinterpret_cast<const uint2*>(a.in[p] + elem[u]));
        bf16x4_to_f32(xr, v[u]);
        if (COMP) {
          const float4 e = __ldcs(reinterpret_cast<const float4*>(a.comp + (int64_t)p * a.n + elem[u]));
          v[u][0] = __fadd_rn(v[u][0], e.x);
          v[u][1] = __fadd_rn(v[u][1], e.y);
          v[u][2] = __fadd_rn(v[u][2], e.z);
          v[u][3] = __fadd_rn(v[u][3], e.w);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (prank[u] < 0) break;                       // warp-uniform
      float lo, hi;
      warp_range(v[u], lo, hi);
      const GroupGrid gg = make_grid(lo, hi, L);
      int q[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) q[k] = encode(v[u][k], gg, L);
      const uint32_t word = pack4<BITS>(q);
      if (BITS == 4) {
        reinterpret_cast<uint16_t*>(a.codes1 + dst[u] * CB)[lane] = (uint16_t)word;
      } else {
        reinterpret_cast<uint32_t*>(a.codes1 + dst[u] * CB)[lane] = word;
      }
      if (lane == 0) a.meta1[midx[u]] = gg.meta;
      if (COMP) {
        float4 en;
        en.x = __fsub_rn(v[u][0], decode(q[0], gg.z, gg.s));
        en.y = __fsub_rn(v[u][1], decode(q[1], gg.z, gg.s));
        en.z = __fsub_rn(v[u][2], decode(q[2], gg.z, gg.s));
        en.w = __fsub_rn(v[u][3], decode(q[3], gg.z, gg.s));
        *reinterpret_cast<float4*>(a.comp + (int64_t)prank[u] * a.n + elem[u]) = en;
      }
      const bool bad = !gg.finite || !all_finite4(v[u]);
      if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.status, kStatusOverflow);
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kPushUnroll = 4;

template <int BITS, bool COMP>
cudaError_t launch_t(const CallArgs& a, cudaStream_t s, bool pdl) {
  static int grid_cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int& grid = grid_cache[dev & 63];
  if (grid == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, push_kernel<BITS, COMP, kPushUnroll>,
                                                  kThreads, 0);
    grid = sms * (per_sm > 0 ? per_sm : 1);
  }
  const int64_t W = (int64_t)a.P * (a.P - 1) * a.Gs;
  const int64_t warps_needed = (W + kPushUnroll - 1) / kPushUnroll;
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
  return cudaLaunchKernelEx(&cfg, push_kernel<BITS, COMP, kPushUnroll>, a);
}

}  // namespace

cudaError_t launch_push(const CallArgs& a, int bits, cudaStream_t s, bool pdl) {
  const bool comp = a.comp != nullptr;
  if (bits == 4) return comp ? launch_t<4, true>(a, s, pdl) : launch_t<4, false>(a, s, pdl);
  return comp ? launch_t<8, true>(a, s, pdl) : launch_t<8, false>(a, s, pdl);
}

}  // namespace echo
