// k_tile.cu -- the whole call for one owner tile in one block ("Echo: Error-
// Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)): the pushes
// of the P-1 senders, the owner's fp32 sum and the gather of a tile of the
// owner's segment depend on the P ranks' inputs and held errors at the same
// element positions only, so with every rank in one GPU's memory a single
// block can take all of them, and no block waits on another.
//
// For each rank p the block loads p's input and held error for the tile (1-D
// bulk copies, cp.async.bulk) and forms v = x + e.  A sender (p != owner)
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
// Two forms, both one-shot blocks over kReduceTileElems-element tiles (g/16
// lanes per group, as everywhere), placed by the hardware as SMs free up:
//  - rank loop (tile_kernel): a block of kReduceWarps warps walks the ranks in
//    ascending order through a ring of shared-memory stages (two; four without
//    state, whose stages are a third as large), so that the next ranks' tiles
//    are in flight while rank p's is computed.  Small blocks, many per SM: the
//    form for grids that fill the GPU several times over.
//  - rank-parallel (tile_rp_kernel): a block of P x kReduceWarps warps, one
//    warp pair per rank, all P ranks' tiles copied at once; each pair pushes
//    its rank and leaves its fp32 terms in shared memory, and rank 0's pair
//    sums them in rank order and does the gather.  A block's critical path is
//    then one push and one gather instead of P pushes: the form for grids too
//    small to fill the GPU, where that path is the call's latency.
// Waits are bounded and block-uniform; on timeout the block records
// ECHO_ERR_TIMEOUT, waits (bounded) for its copies in flight and returns.
#include "stages.cuh"

namespace echo {
namespace {

constexpr int kTE = kReduceTileElems;
constexpr int kTThreads = 32 * kReduceWarps;
// The rank-parallel block holds kTThreads threads per rank.
constexpr int kRpMaxThreads = kTThreads * kTileRpMaxP;
constexpr int kRpMaxP = kTileRpMaxP;
static_assert(kRpMaxThreads <= 1024, "rank-parallel block: at most 1024 threads");

// Resident blocks of 256 threads per SM the register allocation of the rank
// loop must allow (as the reduce kernel's bound): 3 leaves 80 registers a
// thread with fp32 state, 4 leaves 64 with a 2-byte state or none, whose
// bodies are shorter and gain more from the extra resident blocks.
#ifndef ECHO_TILE_MIN_BLOCKS_F32
#define ECHO_TILE_MIN_BLOCKS_F32 3
#endif
#ifndef ECHO_TILE_MIN_BLOCKS
#define ECHO_TILE_MIN_BLOCKS 4
#endif
template <int SF>
constexpr int tile_min_blocks() {
  return (SF == kStateF32 ? ECHO_TILE_MIN_BLOCKS_F32 : ECHO_TILE_MIN_BLOCKS) * kThreads / kTThreads;
}

// One rank's tile in a stage: bf16 inputs, then the held errors.
template <int SF>
constexpr uint32_t tile_stage_bytes() { return (uint32_t)kTE * (2 + state_bytes<SF>()); }
// Stages of the rank loop's ring: with no state a stage holds only the 2 KB
// of inputs, and two of them leave too few bytes in flight per SM.
#ifndef ECHO_TILE_STAGES_NOSTATE
#define ECHO_TILE_STAGES_NOSTATE 4
#endif
template <int SF>
constexpr int tile_stages() { return SF == kNoState ? ECHO_TILE_STAGES_NOSTATE : 2; }
static_assert(ECHO_TILE_STAGES_NOSTATE >= 2 && ECHO_TILE_STAGES_NOSTATE <= 8, "tile ring: 2..8");
// Rank-parallel: per rank a stage, and the rank's fp32 terms.
template <int SF>
constexpr uint32_t rp_rank_bytes() { return tile_stage_bytes<SF>() + (uint32_t)kTE * 4; }

// Where a thread's values sit: the tile's owner and first group, its length
// in groups, and the thread's group (gl, within the tile) and lane within it.
struct TilePos {
  int o;
  int64_t j0;     // first group of the tile, within the owner's segment
  int t;          // groups in the tile
  int64_t e0;     // first element, within a rank
  int gl;
  int q;
  bool valid;     // gl < t
  int64_t grp;    // the group, within a rank tensor
};

template <int G>
__device__ __forceinline__ TilePos tile_pos(const CallArgs& a, int64_t tile, int64_t tiles_per_seg,
                                            int tid) {
  constexpr int T = tile_groups<G, kTE>();
  constexpr int NL = G / 16;
  constexpr int GPW = 32 / NL;
  static_assert(T <= GPW * kReduceWarps, "tile: one pass of kReduceWarps warps");
  TilePos tp;
  tp.o = (int)(tile / tiles_per_seg);
  tp.j0 = (tile - (int64_t)tp.o * tiles_per_seg) * T;
  tp.t = (int)((a.Gs - tp.j0) < T ? (a.Gs - tp.j0) : T);
  tp.e0 = ((int64_t)tp.o * a.Gs + tp.j0) * G;
  const int lane = tid & 31;
  tp.q = lane % NL;
  tp.gl = (tid >> 5) * GPW + lane / NL;
  tp.valid = tp.gl < tp.t;
  tp.grp = (int64_t)tp.o * a.Gs + tp.j0 + tp.gl;
  return tp;
}

// One thread: rank p's tile (inputs, then held errors) into `stage`, on `bar`.
template <int SF, int G>
__device__ __forceinline__ void tile_issue(const CallArgs& a, const TilePos& tp, int p,
                                           uint8_t* stage, uint32_t bar, uint64_t pol) {
  constexpr int EB = state_bytes<SF>();
  mbar_expect_tx(bar, (uint32_t)(tp.t * G * (2 + EB)));
  bulk_g2s(smem_addr(stage), a.in[p] + tp.e0, (uint32_t)(tp.t * G * 2), bar, pol);
  if (SF != kNoState)
    bulk_g2s(smem_addr(stage + kTE * 2),
             reinterpret_cast<const uint8_t*>(a.comp) + ((int64_t)p * a.n + tp.e0) * EB,
             (uint32_t)(tp.t * G * EB), bar, pol);
}

// This lane's 16 values of a rank from a stage: x, plus the held error when
// compensated (zero on the idle lanes of a short tile).
template <int SF, int G>
__device__ __forceinline__ void tile_values(const uint8_t* stage, const TilePos& tp, float v[16]) {
  if (tp.valid) {
    push_load<SF, G>(stage, stage + kTE * 2, tp.gl, tp.q, v);
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = 0.0f;
  }
}

// The push of sender p: codes and meta into the owner's receive slot, the
// sender keeps v - deq(q); the owner's term is deq(q).
template <int BITS, int SF, int MODE, int G>
__device__ __forceinline__ void tile_push(const CallArgs& a, const TilePos& tp, int p,
                                          const float v[16], float term[16], uint64_t codes_pol) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr int NL = G / 16;
  constexpr int CB = G * BITS / 8;
  constexpr int EB = state_bytes<SF>();
  const int js = p < tp.o ? p : p - 1;
  const int64_t slot = (int64_t)tp.o * (a.P - 1) + js;
  uint8_t* cs = a.codes1 + slot * a.Gs * CB;
  const GroupGrid gg = group_grid<MODE, NL>(v, L);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float c[8];
    quantize8_mode<MODE>(v + 8 * hh, gg, L, c, term + 8 * hh);
    if (tp.valid) {
      store_codes8<BITS>(cs + (tp.j0 + tp.gl) * CB + half_code_byte<BITS, NL>(hh, tp.q), c,
                         codes_pol);
      if constexpr (SF != kNoState) {
        float r[8];
        sub_n<8>(r, v + 8 * hh, term + 8 * hh);
        uint8_t* ep = reinterpret_cast<uint8_t*>(a.comp) + (int64_t)p * a.n * EB;
        state_store8<SF, true>(ep, tp.grp * G + half_at<NL>(hh, tp.q), r, a.decay);
      }
    }
  }
  if (tp.valid && tp.q == 0) {
    st_hint_u32(a.meta1 + slot * a.Gs_pad + tp.j0 + tp.gl, gg.meta, codes_pol);
    if (!gg.finite) atomicOr(a.status, kStatusOverflow);
  }
}

// The gather: the sum quantized once; every rank receives the same value and
// the owner keeps sum - output.
template <int BITS, int SF, int MODE, int G>
__device__ __forceinline__ void tile_gather(const CallArgs& a, const TilePos& tp,
                                            const float acc[16], uint64_t codes_pol) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr int NL = G / 16;
  constexpr int CB = G * BITS / 8;
  constexpr int EB = state_bytes<SF>();
  const GroupGrid gg = group_grid<MODE, NL>(acc, L);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float c[8], deq[8];
    quantize8_mode<MODE>(acc + 8 * hh, gg, L, c, deq);
    if (!tp.valid) continue;
    store_codes8<BITS>(a.codes2 + tp.grp * CB + half_code_byte<BITS, NL>(hh, tp.q), c, codes_pol);
    float yb[8];
    const uint4 y = f32x8_to_bf16(deq, yb);
    const int64_t e = tp.grp * G + half_at<NL>(hh, tp.q);
    if constexpr (SF != kNoState) {
      uint8_t* eo = reinterpret_cast<uint8_t*>(a.comp) + (int64_t)tp.o * a.n * EB;
      float r[8];
      sub_n<8>(r, acc + 8 * hh, yb);
      state_store8<SF, true>(eo, e, r, a.decay);
    }
    for (int r = 0; r < a.P; ++r) __stcs(reinterpret_cast<uint4*>(a.out[r] + e), y);
  }
  if (tp.valid && tp.q == 0) {
    st_hint_u32(a.meta2 + (int64_t)tp.o * a.Gs_pad + tp.j0 + tp.gl, gg.meta, codes_pol);
    if (!gg.finite) atomicOr(a.status, kStatusOverflow);
  }
}

// ---- rank loop ----------------------------------------------------------

template <int BITS, int SF, int MODE, int G>
__global__ void __launch_bounds__(kTThreads, tile_min_blocks<SF>())
tile_kernel(const CallArgs a, int64_t tiles_per_seg) {
  constexpr uint32_t SB = tile_stage_bytes<SF>();
  constexpr int S = tile_stages<SF>();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[S];

  const int P = a.P;
  const TilePos tp = tile_pos<G>(a, blockIdx.x, tiles_per_seg, threadIdx.x);
  const uint32_t full0 = smem_addr(&full[0]);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int st = 0; st < S; ++st) mbar_init(full0 + 8 * st, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Inputs, held errors and receive slots may all have been written by the
  // kernel before this one (the previous call).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint64_t pol = 0;
  if (threadIdx.x == 0) pol = policy_evict_first();   // everything loaded is read once
  if (threadIdx.x == 0) {
    for (int p = 0; p < P && p < S; ++p)
      tile_issue<SF, G>(a, tp, p, smem + (size_t)p * SB, full0 + 8 * p, pol);
  }
  const uint64_t codes_pol = kCodesPolicyLast ? policy_evict_last() : policy_evict_normal();

  float acc[16];
  for (int p = 0; p < P; ++p) {
    const int st = p % S;
    if (!mbar_wait_block(full0 + 8 * st, (uint32_t)((p / S) & 1))) {   // same outcome for all
      if (threadIdx.x == 0) {
        atomicOr(a.status, kStatusTimeout);
        for (int pp = p; pp < P && pp < p + S; ++pp)                    // copies in flight
          mbar_wait_bounded(full0 + 8 * (pp % S), (uint32_t)((pp / S) & 1));
      }
      return;
    }
    float v[16];
    tile_values<SF, G>(smem + (size_t)st * SB, tp, v);
    // The stage is in registers: hand it to rank p+S's copies.
    fence_proxy_async();
    __syncthreads();
    if (threadIdx.x == 0 && p + S < P)
      tile_issue<SF, G>(a, tp, p + S, smem + (size_t)st * SB, full0 + 8 * st, pol);

    float term[16];
    if (p == tp.o) {
#pragma unroll
      for (int k = 0; k < 16; ++k) term[k] = v[k];
    } else {
      tile_push<BITS, SF, MODE, G>(a, tp, p, v, term, codes_pol);
    }
    // Ascending rank order, starting from rank 0's term.
    if (p == 0) {
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = term[k];
    } else {
      add_n<16>(acc, acc, term);
    }
  }
  tile_gather<BITS, SF, MODE, G>(a, tp, acc, codes_pol);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- rank-parallel ------------------------------------------------------

template <int BITS, int SF, int MODE, int G>
__global__ void __launch_bounds__(kRpMaxThreads, 1)
tile_rp_kernel(const CallArgs a, int64_t tiles_per_seg) {
  constexpr uint32_t SB = tile_stage_bytes<SF>();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kRpMaxP];

  const int P = a.P;
  const int r = threadIdx.x / kTThreads;          // the rank this warp pair serves
  const int tid = threadIdx.x % kTThreads;
  const TilePos tp = tile_pos<G>(a, blockIdx.x, tiles_per_seg, tid);
  uint8_t* stage = smem + (size_t)r * SB;
  // terms[p][j][tid]: float4 j of thread tid's 16 values of rank p
  float4* terms = reinterpret_cast<float4*>(smem + (size_t)P * SB);
  const uint32_t bar = smem_addr(&full[r]);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) tile_issue<SF, G>(a, tp, r, stage, bar, policy_evict_first());
  const uint64_t codes_pol = kCodesPolicyLast ? policy_evict_last() : policy_evict_normal();

  float term[16];
  const bool ok = mbar_wait_warp(bar, 0);
  if (ok) {
    float v[16];
    tile_values<SF, G>(stage, tp, v);
    if (r == tp.o) {
#pragma unroll
      for (int k = 0; k < 16; ++k) term[k] = v[k];
    } else {
      tile_push<BITS, SF, MODE, G>(a, tp, r, v, term, codes_pol);
    }
    if (r > 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        terms[((size_t)r * 4 + j) * kTThreads + tid] =
            make_float4(term[4 * j], term[4 * j + 1], term[4 * j + 2], term[4 * j + 3]);
    }
  }
  if (!__syncthreads_and(ok ? 1 : 0)) {           // same outcome for all
    if (tid == 0) {
      atomicOr(a.status, kStatusTimeout);
      mbar_wait_bounded(bar, 0);                  // this rank's copies, if still in flight
    }
    return;
  }
  if (r == 0) {
    // Ascending rank order, starting from rank 0's term (in registers).
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = term[k];
    for (int p = 1; p < P; ++p) {
      float t[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 f = terms[((size_t)p * 4 + j) * kTThreads + tid];
        t[4 * j] = f.x;
        t[4 * j + 1] = f.y;
        t[4 * j + 2] = f.z;
        t[4 * j + 3] = f.w;
      }
      add_n<16>(acc, acc, t);
    }
    tile_gather<BITS, SF, MODE, G>(a, tp, acc, codes_pol);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int SF>
constexpr size_t rp_smem_bytes(int P) { return (size_t)P * rp_rank_bytes<SF>(); }

template <int BITS, int SF, int MODE, int G>
cudaError_t launch_t(const CallArgs& a, bool rank_parallel, cudaStream_t s, bool pdl) {
  constexpr int T = tile_groups<G, kTE>();
  const int64_t tiles_per_seg = (a.Gs + T - 1) / T;
  const int64_t blocks = tiles_per_seg * a.P;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  if (rank_parallel) {
    cfg.blockDim = dim3(kTThreads * a.P);
    cfg.dynamicSmemBytes = rp_smem_bytes<SF>(a.P);
  } else {
    cfg.blockDim = dim3(kTThreads);
    cfg.dynamicSmemBytes = tile_stages<SF>() * tile_stage_bytes<SF>();
  }
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (rank_parallel)
    return cudaLaunchKernelEx(&cfg, tile_rp_kernel<BITS, SF, MODE, G>, a, tiles_per_seg);
  return cudaLaunchKernelEx(&cfg, tile_kernel<BITS, SF, MODE, G>, a, tiles_per_seg);
}

template <int MODE, int G>
cudaError_t launch_mode(const CallArgs& a, int bits, bool rp, cudaStream_t s, bool pdl) {
  const int sf = state_fmt_of(a.comp, a.state_fmt);
  if (bits == 4) {
    if (sf == kStateF32) return launch_t<4, kStateF32, MODE, G>(a, rp, s, pdl);
    if (sf == kStateBF16) return launch_t<4, kStateBF16, MODE, G>(a, rp, s, pdl);
    if (sf == kStateF16) return launch_t<4, kStateF16, MODE, G>(a, rp, s, pdl);
    return launch_t<4, kNoState, MODE, G>(a, rp, s, pdl);
  }
  if (sf == kStateF32) return launch_t<8, kStateF32, MODE, G>(a, rp, s, pdl);
  if (sf == kStateBF16) return launch_t<8, kStateBF16, MODE, G>(a, rp, s, pdl);
  if (sf == kStateF16) return launch_t<8, kStateF16, MODE, G>(a, rp, s, pdl);
  return launch_t<8, kNoState, MODE, G>(a, rp, s, pdl);
}

// The rank-parallel kernels' shared memory above the default 48 KB, for the
// largest block they take.
template <int BITS, int SF, int G>
cudaError_t set_rp_attr() {
  cudaError_t e = cudaSuccess, r;
  const int bytes = (int)rp_smem_bytes<SF>(kRpMaxP);
  if ((r = cudaFuncSetAttribute(tile_rp_kernel<BITS, SF, kZeroAware, G>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    e = r;
  if ((r = cudaFuncSetAttribute(tile_rp_kernel<BITS, SF, kNaiveZeroPoint, G>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    e = r;
  if ((r = cudaFuncSetAttribute(tile_rp_kernel<BITS, SF, kSymmetric, G>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    e = r;
  return e;
}

}  // namespace

template <int G>
cudaError_t launch_tile_g(const CallArgs& a, int bits, bool rank_parallel, cudaStream_t s,
                          bool pdl) {
  const bool rp = rank_parallel && a.P <= kRpMaxP;
  if (a.mode == kNaiveZeroPoint) return launch_mode<kNaiveZeroPoint, G>(a, bits, rp, s, pdl);
  if (a.mode == kSymmetric) return launch_mode<kSymmetric, G>(a, bits, rp, s, pdl);
  return launch_mode<kZeroAware, G>(a, bits, rp, s, pdl);
}

template <int G>
cudaError_t prepare_tile_g() {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_rp_attr<4, kStateF32, G>()) != cudaSuccess) e = r;
  if ((r = set_rp_attr<4, kStateBF16, G>()) != cudaSuccess) e = r;
  if ((r = set_rp_attr<4, kStateF16, G>()) != cudaSuccess) e = r;
  if ((r = set_rp_attr<4, kNoState, G>()) != cudaSuccess) e = r;
  if ((r = set_rp_attr<8, kStateF32, G>()) != cudaSuccess) e = r;
  if ((r = set_rp_attr<8, kStateBF16, G>()) != cudaSuccess) e = r;
  if ((r = set_rp_attr<8, kStateF16, G>()) != cudaSuccess) e = r;
  if ((r = set_rp_attr<8, kNoState, G>()) != cudaSuccess) e = r;
  return e;
}

#ifndef ECHO_G
#define ECHO_G 128
#endif
static_assert(group_supported(ECHO_G), "ECHO_G: 64, 128 or 256");
template cudaError_t launch_tile_g<ECHO_G>(const CallArgs&, int, bool, cudaStream_t, bool);
template cudaError_t prepare_tile_g<ECHO_G>();

}  // namespace echo
