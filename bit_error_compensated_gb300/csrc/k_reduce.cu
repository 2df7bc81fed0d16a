// k_reduce.cu -- the owner's reduce and the requantization for the gather
// ("Echo: Error-Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)):
// the owner of a segment decodes the P-1 code tiles it received, adds them to
// its own unquantized segment in fp32 in ascending rank order, quantizes the
// sum once, and keeps the error of that last rounding (sum minus the bf16
// value every rank will receive) as its compensator state for the segment.
// The entry pass of the compensator (adding the owner's held error to its own
// segment) is fused in as well.
//
// Each block takes one owner tile of kReduceTileElems elements
// (kReduceTileElems / g groups).  Thread 0 fills a shared-memory stage with
// 1-D bulk copies (cp.async.bulk, the TMA engine) of the tile's P-1 received
// code tiles, their meta words, the owner's bf16 tile and its state tile, all
// completing on the stage's mbarrier; the block works from shared memory
// (g/16 lanes per group) and stores its results straight to global memory.
// Many short blocks, placed by the hardware as SMs free up, keep the copy
// engines and HBM busy to the end of the grid; with ECHO_REDUCE_RING = R > 1
// a single resident wave of blocks walks the tiles instead, through a ring of
// R stages that thread 0 refills as soon as every thread is done reading one
// (measured slower: the last tiles of the wave leave HBM idle).  The waits on
// the mbarriers are bounded and their outcome is the same for the whole
// block: if one gives up, the block records ECHO_ERR_TIMEOUT in the status
// word, waits once more (also bounded) for its copies in flight, and returns.
//
// With `FUSED` the block also writes the decoded gather value to all P output
// buffers, so the separate gather kernel is skipped.
#include "stages.cuh"

#ifndef ECHO_REDUCE_RING
#define ECHO_REDUCE_RING 1
#endif
// Tiles per block (0: one resident wave of blocks walking all the tiles).
#ifndef ECHO_REDUCE_TILES_PER_BLOCK
#define ECHO_REDUCE_TILES_PER_BLOCK 1
#endif

namespace echo {
namespace {

constexpr int kReduceRing = ECHO_REDUCE_RING;   // tiles in flight per block

constexpr int kTE = kReduceTileElems;
constexpr int kRThreads = 32 * kReduceWarps;

// Resident threads per SM the compiler must allow for: the fused kernels fit
// 1024 (64 registers a thread) without spilling, the unfused ones 768.
#ifndef ECHO_REDUCE_MIN_BLOCKS_FUSED
#define ECHO_REDUCE_MIN_BLOCKS_FUSED 4
#endif
template <bool FUSED>
constexpr int reduce_min_blocks() {
  return (FUSED ? ECHO_REDUCE_MIN_BLOCKS_FUSED : ECHO_REDUCE_MIN_BLOCKS) * kThreads / kRThreads;
}

template <int BITS, int SF, bool FUSED, int MODE, int G>
__global__ void __launch_bounds__(kRThreads, reduce_min_blocks<FUSED>())
reduce_kernel(const CallArgs a, int64_t tiles_per_seg, int64_t ntiles) {
  constexpr int T = tile_groups<G, kTE>();
  constexpr int R = kReduceRing;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[R];

  const int P = a.P;
  const uint32_t sbytes = reduce_stage_bytes<BITS, SF, G, kTE>(P);
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
    reduce_issue_own<BITS, SF, G, kTE>(a, smem + (size_t)st * sbytes, full0 + 8 * st, o, j0, t, pol);
  };
  auto issue_codes = [&](int64_t k, int st) {
    int o, t;
    int64_t j0;
    tile_of(k, o, j0, t);
    reduce_issue_codes<BITS, SF, G, kTE>(a, smem + (size_t)st * sbytes, full0 + 8 * st, o, j0, t, pol);
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
    reduce_tile<BITS, SF, FUSED, MODE, G, kTE, kReduceWarps>(a, smem + (size_t)st * sbytes, o, j0, t);
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
  return (size_t)kReduceRing * reduce_stage_bytes<BITS, SF, G, kTE>(P);
}

template <int BITS, int SF, bool FUSED, int MODE, int G>
cudaError_t launch_t(const CallArgs& a, cudaStream_t s, bool pdl) {
  static CachedInt resident_cache[64][ECHO_MAX_RANKS + 1];
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = smem_bytes<BITS, SF, G>(a.P);
  CachedInt& cached = resident_cache[dev & 63][a.P];
  int resident = cached.get();
  if (resident == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reduce_kernel<BITS, SF, FUSED, MODE, G>,
                                                  kRThreads, smem);
    resident = sms * (per_sm > 0 ? per_sm : 1);
    cached.set(resident);
  }
  constexpr int T = tile_groups<G, kTE>();
  const int64_t tiles_per_seg = (a.Gs + T - 1) / T;
  const int64_t ntiles = tiles_per_seg * a.P;
  constexpr int64_t TPB = ECHO_REDUCE_TILES_PER_BLOCK;
  int64_t blocks = TPB > 0 ? (ntiles + TPB - 1) / TPB : (ntiles < resident ? ntiles : resident);
  if (a.grid_cap > 0 && blocks > a.grid_cap) blocks = a.grid_cap;   // blocks stride over tiles
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kRThreads);
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
  const int sf = state_fmt_of(a.comp, a.state_fmt);
#define ECHO_REDUCE_SF(B, SFV)                                                            \
  return fused ? launch_t<B, SFV, true, MODE, G>(a, s, pdl)                               \
               : launch_t<B, SFV, false, MODE, G>(a, s, pdl);
  if (bits == 4) {
    if (sf == kStateF32) { ECHO_REDUCE_SF(4, kStateF32) }
    if (sf == kStateBF16) { ECHO_REDUCE_SF(4, kStateBF16) }
    if (sf == kStateF16) { ECHO_REDUCE_SF(4, kStateF16) }
    ECHO_REDUCE_SF(4, kNoState)
  }
  if (sf == kStateF32) { ECHO_REDUCE_SF(8, kStateF32) }
  if (sf == kStateBF16) { ECHO_REDUCE_SF(8, kStateBF16) }
  if (sf == kStateF16) { ECHO_REDUCE_SF(8, kStateF16) }
  ECHO_REDUCE_SF(8, kNoState)
#undef ECHO_REDUCE_SF
}

template <int MODE, int G>
cudaError_t prepare_mode() {
  cudaError_t e = cudaSuccess, r;
#define ECHO_PREP(B, SFV)                                                                 \
  if ((r = set_attr<B, SFV, true, MODE, G>()) != cudaSuccess) e = r;                      \
  if ((r = set_attr<B, SFV, false, MODE, G>()) != cudaSuccess) e = r;
  ECHO_PREP(4, kNoState) ECHO_PREP(4, kStateF32) ECHO_PREP(4, kStateBF16) ECHO_PREP(4, kStateF16)
  ECHO_PREP(8, kNoState) ECHO_PREP(8, kStateF32) ECHO_PREP(8, kStateBF16) ECHO_PREP(8, kStateF16)
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
