// k_reduce.cu -- the owner's reduce and the requantization for the gather
// ("Echo: Error-Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)):
// the owner of a segment decodes the P-1 code tiles it received, adds them to
// its own unquantized segment in fp32 in ascending rank order, quantizes the
// sum once, and keeps the error of that last rounding (sum minus the bf16
// value every rank will receive) as its compensator state for the segment.
// The entry pass of the compensator (adding the owner's held error to its own
// segment) is fused in as well.
//
// Blocks walk owner tiles of kReduceTileElems elements (kReduceTileElems / g
// groups) through a ring of kReduceRing shared-memory stages.  Thread 0 fills
// a stage with 1-D bulk copies (cp.async.bulk, the TMA engine) of the tile's
// P-1 received code tiles, their meta words, the owner's bf16 tile and its
// state tile, all completing on the stage's mbarrier; the block works from
// shared memory (g/16 lanes per group) and stores its results straight to
// global memory,
// and thread 0 refills the stage with the block's next tile as soon as every
// thread is done reading it, so the next tile loads while this one is
// computed.  With a ring of 1 every block takes exactly one tile.  The waits
// on the mbarriers are bounded and their outcome is the same for the whole
// block: if one gives up, the block records ECHO_ERR_TIMEOUT in the status
// word, waits once more (also bounded) for its copies in flight, and returns.
//
// With `FUSED` the block also writes the decoded gather value to all P output
// buffers, so the separate gather kernel is skipped.
#include "echo_internal.h"
#include "quant.cuh"
#include "tma.cuh"

#ifndef ECHO_REDUCE_RING
#define ECHO_REDUCE_RING 2
#endif
// Blocks per SM the register allocation must allow.  The shared-memory ring
// already caps residency near this (about 62 KB a block at 4 ranks), so a
// lower figure buys registers without costing occupancy.
#ifndef ECHO_REDUCE_MIN_BLOCKS
#define ECHO_REDUCE_MIN_BLOCKS 3
#endif

namespace echo {
namespace {

constexpr int kReduceRing = ECHO_REDUCE_RING;   // tiles in flight per block

// Groups per tile.
template <int G>
constexpr int tile_groups() { return kReduceTileElems / G; }

// Shared-memory stage of one tile of T groups: [P-1][T][CB] received codes,
// [P-1][T] meta words, [T][G] owner bf16 input, [T][G] owner state (when
// compensated).  Every region starts on a 16-byte boundary.
template <int BITS, int SF, int G>
__host__ __device__ inline uint32_t stage_bytes(int P) {
  constexpr int T = tile_groups<G>();
  return (uint32_t)((P - 1) * T * (G * BITS / 8 + 4) + T * G * 2 + T * G * state_bytes<SF>());
}

// Computes one owner tile (t groups from j0 of segment o) held in a stage,
// writing the gather codes, meta, new owner state and (FUSED) all P outputs
// to global memory.  Every thread of the block takes part.
template <int BITS, int SF, bool FUSED, int MODE, int G>
__device__ __forceinline__ void reduce_tile(const CallArgs& a, const uint8_t* stage, int o,
                                            int64_t j0, int t) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr bool COMP = SF != kNoState;
  constexpr int EB = state_bytes<SF>();
  constexpr int NL = G / 16;                 // lanes per group
  constexpr int GPW = 32 / NL;               // groups per warp per pass
  constexpr int CB = G * BITS / 8;
  constexpr int T = tile_groups<G>();
  const int P = a.P;
  const uint8_t* s_codes = stage;
  const uint32_t* s_meta = reinterpret_cast<const uint32_t*>(stage + (P - 1) * T * CB);
  const uint2* s_x = reinterpret_cast<const uint2*>(stage + (P - 1) * T * (CB + 4));
  const uint8_t* s_e = stage + (P - 1) * T * (CB + 4) + T * G * 2;         // [T] group states
  // The gather kernel reads these codes next: keep them in L2.
  const uint64_t codes_pol = kCodesPolicyLast ? policy_evict_last() : policy_evict_normal();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / NL;
  const int q = lane % NL;
  // GPW groups per warp per pass (NL lanes each, see quant.cuh).
  for (int gq = GPW * warp; gq < t; gq += GPW * (kThreads / 32)) {
    const int gl = gq + sub;                       // group within the tile
    const bool valid = gl < t;
    const int gs = valid ? gl : gq;                // idle lanes read a valid group
    // Decoded term of sender p (p != o), from its receive slot.
    auto sender_term = [&](int p, float term[16]) {
      const int js = p < o ? p : p - 1;
      float s, zf;
      unpack_meta(s_meta[js * T + gs], s, zf);
      const uint8_t* cg = s_codes + (js * T + gs) * CB;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint8_t* cw = cg + chunk_code_byte<BITS, NL>(c, q);
        const uint32_t w = BITS == 4 ? (uint32_t)*reinterpret_cast<const uint16_t*>(cw)
                                     : *reinterpret_cast<const uint32_t*>(cw);
        decode4_mode<BITS, MODE>(w, s, zf, term + 4 * c);
      }
    };
    // The owner's own term: its bf16 input plus (compensated) its held error.
    auto own_term = [&](float term[16]) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        bf16x4_to_f32(s_x[(gs * G + chunk_at<NL>(c, q)) / 4], term + 4 * c);
        if constexpr (COMP) {
          float e[4];
          state_load4<SF>(s_e, gs * G + chunk_at<NL>(c, q), e);
#pragma unroll
          for (int k = 0; k < 4; ++k) term[4 * c + k] = __fadd_rn(term[4 * c + k], e[k]);
        }
      }
    };
    // Ascending rank order, starting from rank 0's term: the senders below
    // the owner, the owner's own term, the senders above.
    float acc[16], term[16];
    if (o == 0) {
      own_term(acc);
    } else {
      sender_term(0, acc);
      for (int p = 1; p < o; ++p) {
        sender_term(p, term);
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = __fadd_rn(acc[k], term[k]);
      }
      own_term(term);
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = __fadd_rn(acc[k], term[k]);
    }
    for (int p = o + 1; p < P; ++p) {
      sender_term(p, term);
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = __fadd_rn(acc[k], term[k]);
    }

    // Quantize the sum once for the gather.
    const GroupGrid gg = group_grid<MODE, NL>(acc, L);
    const int64_t grp = (int64_t)o * a.Gs + j0 + gl;           // group index in the rank tensor
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {               // chunks 2hh and 2hh+1
      float c[8], deq[8];
      quantize8_mode<MODE>(acc + 8 * hh, gg, L, c, deq);
      if (!valid) continue;
      uint8_t* cg = a.codes2 + grp * CB;
      if (BITS == 4) {
        st_hint_u16(cg + chunk_code_byte<4, NL>(2 * hh, q), pack4<4>(c), codes_pol);
        st_hint_u16(cg + chunk_code_byte<4, NL>(2 * hh + 1, q), pack4<4>(c + 4), codes_pol);
      } else {
        st_hint_u32(cg + chunk_code_byte<8, NL>(2 * hh, q), pack4<8>(c), codes_pol);
        st_hint_u32(cg + chunk_code_byte<8, NL>(2 * hh + 1, q), pack4<8>(c + 4), codes_pol);
      }
      float yb[8];
      const uint2 ya = f32x4_to_bf16(deq, yb);
      const uint2 yv = f32x4_to_bf16(deq + 4, yb + 4);
      const int64_t ea = grp * G + chunk_at<NL>(2 * hh, q);
      const int64_t eb = grp * G + chunk_at<NL>(2 * hh + 1, q);
      if constexpr (COMP) {
        uint8_t* eo = reinterpret_cast<uint8_t*>(a.comp) + (int64_t)o * a.n * EB;
        const float* aa = acc + 8 * hh;
        float r[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) r[k] = __fsub_rn(aa[k], yb[k]);
        state_store4<SF>(eo, ea, r, a.decay);
        state_store4<SF>(eo, eb, r + 4, a.decay);
      }
      if (FUSED) {
        for (int r = 0; r < P; ++r) {
          __stcs(reinterpret_cast<uint2*>(a.out[r] + ea), ya);
          __stcs(reinterpret_cast<uint2*>(a.out[r] + eb), yv);
        }
      }
    }
    if (valid && q == 0) {
      st_hint_u32(a.meta2 + (int64_t)o * a.Gs_pad + j0 + gl, gg.meta, codes_pol);
      if (!gg.finite) atomicOr(a.status, kStatusOverflow);
    }
  }
}

template <int BITS, int SF, bool FUSED, int MODE, int G>
__global__ void __launch_bounds__(kThreads, ECHO_REDUCE_MIN_BLOCKS)
reduce_kernel(const CallArgs a, int64_t tiles_per_seg, int64_t ntiles) {
  constexpr int CB = G * BITS / 8;         // code bytes per group
  constexpr bool COMP = SF != kNoState;
  constexpr int EB = state_bytes<SF>();    // state bytes per element
  constexpr int T = tile_groups<G>();
  constexpr int R = kReduceRing;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[R];

  const int P = a.P;
  const uint32_t sbytes = stage_bytes<BITS, SF, G>(P);
  const uint32_t full0 = smem_addr(&full[0]);
  if (threadIdx.x == 0) {
    for (int st = 0; st < R; ++st) mbar_init(full0 + 8 * st, 1);
    fence_barrier_init();
  }
  __syncthreads();

  auto tile_of = [&](int64_t k, int& o, int64_t& j0, int& t) {
    const int64_t tile = (int64_t)blockIdx.x + k * gridDim.x;
    o = (int)(tile / tiles_per_seg);
    j0 = (tile - (int64_t)o * tiles_per_seg) * T;
    t = (int)((a.Gs - j0) < T ? (a.Gs - j0) : T);
  };
  auto exists = [&](int64_t k) { return (int64_t)blockIdx.x + k * gridDim.x < ntiles; };
  uint64_t pol = 0;
  // Thread 0: the owner's own input and state of block tile k into stage st
  // (arming the stage's barrier for the whole tile), then its received codes.
  auto issue_own = [&](int64_t k, int st) {
    int o, t;
    int64_t j0;
    tile_of(k, o, j0, t);
    const uint32_t meta_bytes = (uint32_t)(((t + 3) & ~3) * 4);
    const uint32_t bar = full0 + 8 * st;
    uint8_t* stage = smem + (size_t)st * sbytes;
    const int64_t g0 = (int64_t)o * a.Gs + j0;
    mbar_expect_tx(bar, (uint32_t)((P - 1) * (t * CB + meta_bytes) + t * G * (2 + EB)));
    bulk_g2s(smem_addr(stage + (P - 1) * T * (CB + 4)), a.in[o] + g0 * G, (uint32_t)(t * G * 2),
             bar, pol);
    if (COMP) bulk_g2s(smem_addr(stage + (P - 1) * T * (CB + 4) + T * G * 2),
                       reinterpret_cast<const uint8_t*>(a.comp) + ((int64_t)o * a.n + g0 * G) * EB,
                       (uint32_t)(t * G * EB), bar, pol);
  };
  auto issue_codes = [&](int64_t k, int st) {
    int o, t;
    int64_t j0;
    tile_of(k, o, j0, t);
    const uint32_t meta_bytes = (uint32_t)(((t + 3) & ~3) * 4);
    const uint32_t bar = full0 + 8 * st;
    uint8_t* stage = smem + (size_t)st * sbytes;
    for (int js = 0; js < P - 1; ++js) {
      const int64_t slot = (int64_t)o * (P - 1) + js;
      bulk_g2s(smem_addr(stage + js * T * CB), a.codes1 + (slot * a.Gs + j0) * CB,
               (uint32_t)(t * CB), bar, pol);
      bulk_g2s(smem_addr(stage + (P - 1) * T * CB + js * T * 4), a.meta1 + slot * a.Gs_pad + j0,
               meta_bytes, bar, pol);
    }
  };

  if (threadIdx.x == 0) {
    pol = policy_evict_first();                    // every byte loaded is read once per call
    // The owner's own tiles do not depend on the push kernel, so with P > 1
    // their copies are issued before waiting for the push to finish.  (The
    // push kernel itself waited for everything before it, so what it did not
    // write is already final.)  With P == 1 there is no push kernel and the
    // preceding kernel may still be writing them: wait first.
    if (P == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int st = 0; st < R; ++st) if (exists(st)) issue_own(st, st);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int st = 0; st < R; ++st) if (exists(st)) issue_codes(st, st);
  } else {
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }

  for (int64_t k = 0; exists(k); ++k) {
    const int st = (int)(k % R);
    if (!mbar_wait_block(full0 + 8 * st, (uint32_t)((k / R) & 1))) {   // same outcome for all
      if (threadIdx.x == 0) {
        atomicOr(a.status, kStatusTimeout);
        for (int64_t kk = k; kk < k + R && exists(kk); ++kk)   // copies still in flight
          mbar_wait_bounded(full0 + 8 * (int)(kk % R), (uint32_t)((kk / R) & 1));
      }
      return;
    }
    int o, t;
    int64_t j0;
    tile_of(k, o, j0, t);
    reduce_tile<BITS, SF, FUSED, MODE, G>(a, smem + (size_t)st * sbytes, o, j0, t);
    if (exists(k + R)) {                           // block-uniform
      fence_proxy_async();                         // this thread's reads before the refill
      __syncthreads();
      if (threadIdx.x == 0) {
        issue_own(k + R, st);
        issue_codes(k + R, st);
      }
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int BITS, int SF, int G>
size_t smem_bytes(int P) {
  return (size_t)kReduceRing * stage_bytes<BITS, SF, G>(P);
}

template <int BITS, int SF, bool FUSED, int MODE, int G>
cudaError_t launch_t(const CallArgs& a, cudaStream_t s, bool pdl) {
  static int resident_cache[64][ECHO_MAX_RANKS + 1] = {{0}};
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = smem_bytes<BITS, SF, G>(a.P);
  int& resident = resident_cache[dev & 63][a.P];
  if (resident == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reduce_kernel<BITS, SF, FUSED, MODE, G>,
                                                  kThreads, smem);
    resident = sms * (per_sm > 0 ? per_sm : 1);
  }
  constexpr int T = tile_groups<G>();
  const int64_t tiles_per_seg = (a.Gs + T - 1) / T;
  const int64_t ntiles = tiles_per_seg * a.P;
  // A ring of 1 is one tile per block; otherwise one resident wave of blocks.
  const int64_t blocks = (kReduceRing == 1 || ntiles < resident) ? ntiles : resident;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, reduce_kernel<BITS, SF, FUSED, MODE, G>, a, tiles_per_seg, ntiles);
}

template <int BITS, int SF, bool FUSED, int MODE, int G>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(reduce_kernel<BITS, SF, FUSED, MODE, G>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes<BITS, SF, G>(ECHO_MAX_RANKS));
}

template <int MODE, int G>
cudaError_t launch_mode(const CallArgs& a, int bits, bool fused, cudaStream_t s, bool pdl) {
  const int sf = a.comp == nullptr ? kNoState : (a.state_bf16 ? kStateBF16 : kStateF32);
#define ECHO_REDUCE_SF(B, SFV)                                                            \
  return fused ? launch_t<B, SFV, true, MODE, G>(a, s, pdl)                               \
               : launch_t<B, SFV, false, MODE, G>(a, s, pdl);
  if (bits == 4) {
    if (sf == kStateF32) { ECHO_REDUCE_SF(4, kStateF32) }
    if (sf == kStateBF16) { ECHO_REDUCE_SF(4, kStateBF16) }
    ECHO_REDUCE_SF(4, kNoState)
  }
  if (sf == kStateF32) { ECHO_REDUCE_SF(8, kStateF32) }
  if (sf == kStateBF16) { ECHO_REDUCE_SF(8, kStateBF16) }
  ECHO_REDUCE_SF(8, kNoState)
#undef ECHO_REDUCE_SF
}

template <int MODE, int G>
cudaError_t prepare_mode() {
  cudaError_t e = cudaSuccess, r;
#define ECHO_PREP(B, SFV)                                                                 \
  if ((r = set_attr<B, SFV, true, MODE, G>()) != cudaSuccess) e = r;                      \
  if ((r = set_attr<B, SFV, false, MODE, G>()) != cudaSuccess) e = r;
  ECHO_PREP(4, kNoState) ECHO_PREP(4, kStateF32) ECHO_PREP(4, kStateBF16)
  ECHO_PREP(8, kNoState) ECHO_PREP(8, kStateF32) ECHO_PREP(8, kStateBF16)
#undef ECHO_PREP
  return e;
}

}  // namespace

template <int G>
cudaError_t launch_reduce_g(const CallArgs& a, int bits, bool fused, cudaStream_t s, bool pdl) {
  if (a.mode == kNaiveZeroPoint) return launch_mode<kNaiveZeroPoint, G>(a, bits, fused, s, pdl);
  if (a.mode == kSymmetric) return launch_mode<kSymmetric, G>(a, bits, fused, s, pdl);
  return launch_mode<kZeroAware, G>(a, bits, fused, s, pdl);
}

template <int G>
cudaError_t prepare_reduce_g() {
  cudaError_t e = prepare_mode<kZeroAware, G>(), r;
  if ((r = prepare_mode<kNaiveZeroPoint, G>()) != cudaSuccess) e = r;
  if ((r = prepare_mode<kSymmetric, G>()) != cudaSuccess) e = r;
  return e;
}

#ifndef ECHO_G
#define ECHO_G 128
#endif
static_assert(group_supported(ECHO_G), "ECHO_G: 64, 128 or 256");
template cudaError_t launch_reduce_g<ECHO_G>(const CallArgs&, int, bool, cudaStream_t, bool);
template cudaError_t prepare_reduce_g<ECHO_G>();

}  // namespace echo
