// k_tile.cu -- the whole call for one owner tile in one block ("Echo: Error-
// Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)): the pushes
// of the P-1 senders, the owner's fp32 sum and the gather of a tile of the
// owner's segment depend on the P ranks' inputs and held errors at the same
// element positions only, so with every rank in one GPU's memory a single
// block can take all of them, and no block waits on another.
//
// The block walks the ranks in ascending order.  For rank p it loads p's
// input and held error for the tile (1-D bulk copies, cp.async.bulk, into a
// ring of two shared-memory stages, so that rank p+1's tile is in flight
// while rank p's is computed) and forms v = x + e.  A sender (p != owner)
// quantizes v, writes the codes and meta word to the owner's receive slot as
// the push does, keeps v - deq(q) as its held error, and contributes the
// decoded value; the owner contributes v itself.  The contributions are summed
// in fp32 in rank order, starting from rank 0's, then the sum is quantized
// once: the gather codes and meta are written, every rank's output receives
// the decoded bf16 value, and the owner keeps sum - output.  Every value and
// every byte of the receive slots is the two-kernel path's; what is saved is
// the kernel boundary between push and reduce and the owner's read of the
// push codes, which it decodes from the values it has just encoded instead.
//
// One-shot blocks of kReduceWarps warps over kReduceTileElems-element tiles
// (g/16 lanes per group, as everywhere), placed by the hardware as SMs free
// up.  Waits are bounded and block-uniform; on timeout the block records
// ECHO_ERR_TIMEOUT, waits (bounded) for its copies in flight and returns.
#include "stages.cuh"

namespace echo {
namespace {

constexpr int kTE = kReduceTileElems;
constexpr int kTThreads = 32 * kReduceWarps;

// Resident blocks of 256 threads per SM the register allocation must allow
// (as the reduce kernel's bound): 4 leaves 64 registers a thread.
#ifndef ECHO_TILE_MIN_BLOCKS
#define ECHO_TILE_MIN_BLOCKS 4
#endif
constexpr int kTileMinBlocks = ECHO_TILE_MIN_BLOCKS * kThreads / kTThreads;

// One rank's tile in a stage: bf16 inputs, then the held errors.
template <int SF>
constexpr uint32_t tile_stage_bytes() { return (uint32_t)kTE * (2 + state_bytes<SF>()); }

template <int BITS, int SF, int MODE, int G>
__global__ void __launch_bounds__(kTThreads, kTileMinBlocks)
tile_kernel(const CallArgs a, int64_t tiles_per_seg) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr int T = tile_groups<G, kTE>();
  constexpr int NL = G / 16;
  constexpr int GPW = 32 / NL;
  constexpr int CB = G * BITS / 8;
  constexpr int EB = state_bytes<SF>();
  constexpr bool COMP = SF != kNoState;
  constexpr uint32_t SB = tile_stage_bytes<SF>();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[2];

  const int P = a.P;
  const int64_t tile = blockIdx.x;
  const int o = (int)(tile / tiles_per_seg);
  const int64_t j0 = (tile - (int64_t)o * tiles_per_seg) * T;   // first group of the tile
  const int t = (int)((a.Gs - j0) < T ? (a.Gs - j0) : T);         // groups in the tile
  const int64_t e0 = ((int64_t)o * a.Gs + j0) * G;                 // first element, in a rank
  const uint32_t full0 = smem_addr(&full[0]);
  if (threadIdx.x == 0) {
    mbar_init(full0, 1);
    mbar_init(full0 + 8, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Inputs, held errors and receive slots may all have been written by the
  // kernel before this one (the previous call).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint64_t pol = 0;
  if (threadIdx.x == 0) pol = policy_evict_first();   // everything loaded is read once
  // Thread 0: rank p's tile into stage st.
  auto issue = [&](int p, int st) {
    const uint32_t bar = full0 + 8 * st;
    uint8_t* stage = smem + (size_t)st * SB;
    mbar_expect_tx(bar, (uint32_t)(t * G * (2 + EB)));
    bulk_g2s(smem_addr(stage), a.in[p] + e0, (uint32_t)(t * G * 2), bar, pol);
    if (COMP)
      bulk_g2s(smem_addr(stage + kTE * 2),
               reinterpret_cast<const uint8_t*>(a.comp) + ((int64_t)p * a.n + e0) * EB,
               (uint32_t)(t * G * EB), bar, pol);
  };
  if (threadIdx.x == 0) {
    issue(0, 0);
    if (P > 1) issue(1, 1);
  }

  const uint64_t codes_pol = kCodesPolicyLast ? policy_evict_last() : policy_evict_normal();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / NL;
  const int q = lane % NL;
  const int gl = warp * GPW + sub;                 // group within the tile (one pass)
  const bool valid = gl < t;
  const int64_t grp = (int64_t)o * a.Gs + j0 + gl; // the group, within a rank tensor
  static_assert(T <= GPW * kReduceWarps, "tile: one pass of the block's warps");

  float acc[16];
  for (int p = 0; p < P; ++p) {
    const int st = p & 1;
    if (!mbar_wait_block(full0 + 8 * st, (uint32_t)((p >> 1) & 1))) {   // same outcome for all
      if (threadIdx.x == 0) {
        atomicOr(a.status, kStatusTimeout);
        for (int pp = p; pp < P && pp < p + 2; ++pp)                    // copies in flight
          mbar_wait_bounded(full0 + 8 * (pp & 1), (uint32_t)((pp >> 1) & 1));
      }
      return;
    }
    // This lane's 16 values of rank p: x, plus the held error when compensated.
    float v[16];
    const uint8_t* stage = smem + (size_t)st * SB;
    if (valid) {
      push_load<SF, G>(stage, stage + kTE * 2, gl, q, v);
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = 0.0f;   // idle lanes of a short tile
    }
    // The stage is in registers: hand it to rank p+2's copies.
    fence_proxy_async();
    __syncthreads();
    if (threadIdx.x == 0 && p + 2 < P) issue(p + 2, st);

    float term[16];
    if (p == o) {
#pragma unroll
      for (int k = 0; k < 16; ++k) term[k] = v[k];
    } else {
      // The push of sender p: codes and meta into the owner's receive slot,
      // the sender keeps v - deq(q); the owner's term is deq(q).
      const int js = p < o ? p : p - 1;
      const int64_t slot = (int64_t)o * (P - 1) + js;
      uint8_t* cs = a.codes1 + slot * a.Gs * CB;
      const GroupGrid gg = group_grid<MODE, NL>(v, L);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float c[8];
        quantize8_mode<MODE>(v + 8 * hh, gg, L, c, term + 8 * hh);
        if (valid) {
          store_codes8<BITS>(cs + (j0 + gl) * CB + half_code_byte<BITS, NL>(hh, q), c, codes_pol);
          if constexpr (COMP) {
            float r[8];
            sub_n<8>(r, v + 8 * hh, term + 8 * hh);
            uint8_t* ep = reinterpret_cast<uint8_t*>(a.comp) + (int64_t)p * a.n * EB;
            state_store8<SF, true>(ep, grp * G + half_at<NL>(hh, q), r, a.decay);
          }
        }
      }
      if (valid && q == 0) {
        st_hint_u32(a.meta1 + slot * a.Gs_pad + j0 + gl, gg.meta, codes_pol);
        if (!gg.finite) atomicOr(a.status, kStatusOverflow);
      }
    }
    // Ascending rank order, starting from rank 0's term.
    if (p == 0) {
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = term[k];
    } else {
      add_n<16>(acc, acc, term);
    }
  }

  // The gather: the sum quantized once; every rank receives the same value.
  const GroupGrid gg = group_grid<MODE, NL>(acc, L);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float c[8], deq[8];
    quantize8_mode<MODE>(acc + 8 * hh, gg, L, c, deq);
    if (!valid) continue;
    store_codes8<BITS>(a.codes2 + grp * CB + half_code_byte<BITS, NL>(hh, q), c, codes_pol);
    float yb[8];
    const uint4 y = f32x8_to_bf16(deq, yb);
    const int64_t e = grp * G + half_at<NL>(hh, q);
    if constexpr (COMP) {
      uint8_t* eo = reinterpret_cast<uint8_t*>(a.comp) + (int64_t)o * a.n * EB;
      float r[8];
      sub_n<8>(r, acc + 8 * hh, yb);
      state_store8<SF, true>(eo, e, r, a.decay);
    }
    for (int r = 0; r < P; ++r) __stcs(reinterpret_cast<uint4*>(a.out[r] + e), y);
  }
  if (valid && q == 0) {
    st_hint_u32(a.meta2 + (int64_t)o * a.Gs_pad + j0 + gl, gg.meta, codes_pol);
    if (!gg.finite) atomicOr(a.status, kStatusOverflow);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int BITS, int SF, int MODE, int G>
cudaError_t launch_t(const CallArgs& a, cudaStream_t s, bool pdl) {
  constexpr int T = tile_groups<G, kTE>();
  const int64_t tiles_per_seg = (a.Gs + T - 1) / T;
  const int64_t blocks = tiles_per_seg * a.P;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = 2 * tile_stage_bytes<SF>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tile_kernel<BITS, SF, MODE, G>, a, tiles_per_seg);
}

template <int MODE, int G>
cudaError_t launch_mode(const CallArgs& a, int bits, cudaStream_t s, bool pdl) {
  const int sf = state_fmt_of(a.comp, a.state_fmt);
  if (bits == 4) {
    if (sf == kStateF32) return launch_t<4, kStateF32, MODE, G>(a, s, pdl);
    if (sf == kStateBF16) return launch_t<4, kStateBF16, MODE, G>(a, s, pdl);
    if (sf == kStateF16) return launch_t<4, kStateF16, MODE, G>(a, s, pdl);
    return launch_t<4, kNoState, MODE, G>(a, s, pdl);
  }
  if (sf == kStateF32) return launch_t<8, kStateF32, MODE, G>(a, s, pdl);
  if (sf == kStateBF16) return launch_t<8, kStateBF16, MODE, G>(a, s, pdl);
  if (sf == kStateF16) return launch_t<8, kStateF16, MODE, G>(a, s, pdl);
  return launch_t<8, kNoState, MODE, G>(a, s, pdl);
}

}  // namespace

template <int G>
cudaError_t launch_tile_g(const CallArgs& a, int bits, cudaStream_t s, bool pdl) {
  if (a.mode == kNaiveZeroPoint) return launch_mode<kNaiveZeroPoint, G>(a, bits, s, pdl);
  if (a.mode == kSymmetric) return launch_mode<kSymmetric, G>(a, bits, s, pdl);
  return launch_mode<kZeroAware, G>(a, bits, s, pdl);
}

#ifndef ECHO_G
#define ECHO_G 128
#endif
static_assert(group_supported(ECHO_G), "ECHO_G: 64, 128 or 256");
template cudaError_t launch_tile_g<ECHO_G>(const CallArgs&, int, cudaStream_t, bool);

}  // namespace echo
