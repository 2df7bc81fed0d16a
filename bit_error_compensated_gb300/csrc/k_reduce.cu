// k_reduce.cu -- the owner's reduce and the requantization for the gather
// ("Echo: Error-Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)):
// the owner of a segment decodes the P-1 code tiles it received, adds them to
// its own unquantized segment in fp32 in ascending rank order, quantizes the
// sum once, and keeps the error of that last rounding (sum minus the bf16
// value every rank will receive) as its compensator state for the segment.
// The entry pass of the compensator (adding the owner's held error to its own
// segment) is fused in as well.
//
// One thread block per owner tile of kReduceTile groups.  One thread issues
// 1-D bulk copies (cp.async.bulk, the TMA engine) of the P-1 received code
// tiles, their meta words, the owner's bf16 tile and its fp32 state tile into
// shared memory, all completing on one mbarrier; the block then works from
// shared memory, one warp per group.  The wait on the mbarrier is bounded: if
// it gives up, the block records ECHO_ERR_TIMEOUT in the status word, waits
// once more (also bounded) for its copies, and returns.
//
// With `FUSED` the block also writes the decoded gather value to all P output
// buffers, so the separate gather kernel is skipped.
#include "echo_internal.h"
#include "quant.cuh"

namespace echo {
namespace {

constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done != 0;
}

// Wait for phase `parity` of the barrier, giving up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

template <int BITS, bool COMP, bool FUSED>
__global__ void __launch_bounds__(kThreads)
reduce_kernel(const CallArgs a, int64_t tiles_per_seg) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr int CB = 16 * BITS;            // code bytes per group
  constexpr int T = kReduceTile;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;

  const int P = a.P;
  const int o = (int)(blockIdx.x / tiles_per_seg);
  const int64_t j0 = (blockIdx.x - (int64_t)o * tiles_per_seg) * T;
  const int t = (int)((a.Gs - j0) < T ? (a.Gs - j0) : T);   // groups in this tile

  uint8_t* s_codes = smem;                                     // [P-1][T][CB]
  uint32_t* s_meta = reinterpret_cast<uint32_t*>(smem + (P - 1) * T * CB);   // [P-1][T]
  uint2* s_x = reinterpret_cast<uint2*>(smem + (P - 1) * T * (CB + 4));      // [T][32] of 4 bf16
  float4* s_e = reinterpret_cast<float4*>(smem + (P - 1) * T * (CB + 4) + T * 256);  // [T][32]

  const uint32_t bar_a = smem_addr(&bar);
  const int64_t seg_group0 = (int64_t)o * a.Gs + j0;           // first group of the tile in the rank tensor
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar_a) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (threadIdx.x == 0) {
    // The owner's own tile does not depend on the push kernel, so with P > 1
    // its copies are issued before waiting for the push to finish.  (The push
    // kernel itself waited for everything before it, so what it did not write
    // is already final.)  With P == 1 there is no push kernel and the
    // preceding kernel may still be writing that tile: wait first.
    if (P == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t meta_bytes = (uint32_t)(((t + 3) & ~3) * 4);
    const uint32_t total = (uint32_t)((P - 1) * (t * CB + meta_bytes) + t * 256 + (COMP ? t * 512 : 0));
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar_a), "r"(total) : "memory");
    bulk_g2s(smem_addr(s_x), a.in[o] + seg_group0 * kGroup, (uint32_t)(t * 256), bar_a);
    if (COMP) {
      bulk_g2s(smem_addr(s_e), a.comp + (int64_t)o * a.n + seg_group0 * kGroup, (uint32_t)(t * 512), bar_a);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int js = 0; js < P - 1; ++js) {
      const int64_t slot = (int64_t)o * (P - 1) + js;
      bulk_g2s(smem_addr(s_codes + js * T * CB), a.codes1 + (slot * a.Gs + j0) * CB,
               (uint32_t)(t * CB), bar_a);
      bulk_g2s(smem_addr(s_meta + js * T), a.meta1 + slot * a.Gs_pad + j0, meta_bytes, bar_a);
    }
  } else {
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }

  if (!mbar_wait_bounded(bar_a, 0)) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTimeout);
    mbar_wait_bounded(bar_a, 0);   // let copies in flight land before leaving
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int gl = warp; gl < t; gl += kThreads / 32) {
    float acc[4];
#pragma unroll 1
    for (int p = 0; p < P; ++p) {
      float term[4];
      if (p == o) {
        bf16x4_to_f32(s_x[gl * 32 + lane], term);
        if (COMP) {
          const float4 e = s_e[gl * 32 + lane];
          term[0] = __fadd_rn(term[0], e.x);
          term[1] = __fadd_rn(term[1], e.y);
          term[2] = __fadd_rn(term[2], e.z);
          term[3] = __fadd_rn(term[3], e.w);
        }
      } else {
        const int js = p < o ? p : p - 1;
        float s;
        int z;
        unpack_meta(s_meta[js * T + gl], s, z);
        uint32_t w;
        if (BITS == 4) {
          w = reinterpret_cast<const uint16_t*>(s_codes + (js * T + gl) * CB)[lane];
        } else {
          w = reinterpret_cast<const uint32_t*>(s_codes + (js * T + gl) * CB)[lane];
        }
        int q[4];
        unpack4<BITS>(w, q);
#pragma unroll
        for (int k = 0; k < 4; ++k) term[k] = decode(q[k], z, s);
      }
      if (p == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = term[k];
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = __fadd_rn(acc[k], term[k]);
      }
    }

    // Quantize the sum once for the gather.
    float lo, hi;
    warp_range(acc, lo, hi);
    const GroupGrid gg = make_grid(lo, hi, L);
    int q[4];
    float deq[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      q[k] = encode(acc[k], gg, L);
      deq[k] = decode(q[k], gg.z, gg.s);
    }
    const int64_t grp = seg_group0 + gl;           // group index in the rank tensor
    const uint32_t word = pack4<BITS>(q);
    if (BITS == 4) {
      reinterpret_cast<uint16_t*>(a.codes2 + grp * CB)[lane] = (uint16_t)word;
    } else {
      reinterpret_cast<uint32_t*>(a.codes2 + grp * CB)[lane] = word;
    }
    if (lane == 0) a.meta2[(int64_t)o * a.Gs_pad + j0 + gl] = gg.meta;

    float yb[4];
    const uint2 y = f32x4_to_bf16(deq, yb);
    const int64_t elem = grp * kGroup + 4 * lane;
    if (COMP) {
      float4 en;
      en.x = __fsub_rn(acc[0], yb[0]);
      en.y = __fsub_rn(acc[1], yb[1]);
      en.z = __fsub_rn(acc[2], yb[2]);
      en.w = __fsub_rn(acc[3], yb[3]);
      *reinterpret_cast<float4*>(a.comp + (int64_t)o * a.n + elem) = en;
    }
    if (FUSED) {
      for (int r = 0; r < P; ++r) __stcs(reinterpret_cast<uint2*>(a.out[r] + elem), y);
    }
    const bool bad = !gg.finite || !all_finite4(acc);
    if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.status, kStatusOverflow);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int BITS, bool COMP, bool FUSED>
size_t smem_bytes(int P) {
  constexpr int CB = 16 * BITS;
  return (size_t)(P - 1) * kReduceTile * (CB + 4) + kReduceTile * 256 + (COMP ? kReduceTile * 512 : 0);
}

template <int BITS, bool COMP, bool FUSED>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(reduce_kernel<BITS, COMP, FUSED>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes<BITS, COMP, FUSED>(ECHO_MAX_RANKS));
}

template <int BITS, bool COMP, bool FUSED>
cudaError_t launch_t(const CallArgs& a, cudaStream_t s, bool pdl) {
  const int64_t tiles_per_seg = (a.Gs + kReduceTile - 1) / kReduceTile;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles_per_seg * a.P));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes<BITS, COMP, FUSED>(a.P);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, reduce_kernel<BITS, COMP, FUSED>, a, tiles_per_seg);
}

}  // namespace

cudaError_t launch_reduce(const CallArgs& a, int bits, bool fused, cudaStream_t s, bool pdl) {
  const bool comp = a.comp != nullptr;
  if (bits == 4) {
    if (comp) return fused ? launch_t<4, true, true>(a, s, pdl) : launch_t<4, true, false>(a, s, pdl);
    return fused ? launch_t<4, false, true>(a, s, pdl) : launch_t<4, false, false>(a, s, pdl);
  }
  if (comp) return fused ? launch_t<8, true, true>(a, s, pdl) : launch_t<8, true, false>(a, s, pdl);
  return fused ? launch_t<8, false, true>(a, s, pdl) : launch_t<8, false, false>(a, s, pdl);
}

cudaError_t prepare_kernels() {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_attr<4, true, true>()) != cudaSuccess) e = r;
  if ((r = set_attr<4, true, false>()) != cudaSuccess) e = r;
  if ((r = set_attr<4, false, true>()) != cudaSuccess) e = r;
  if ((r = set_attr<4, false, false>()) != cudaSuccess) e = r;
  if ((r = set_attr<8, true, true>()) != cudaSuccess) e = r;
  if ((r = set_attr<8, true, false>()) != cudaSuccess) e = r;
  if ((r = set_attr<8, false, true>()) != cudaSuccess) e = r;
  if ((r = set_attr<8, false, false>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace echo
