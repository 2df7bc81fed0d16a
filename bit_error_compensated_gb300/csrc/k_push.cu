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
// Grid: blockIdx.y is a (sender p, owner o) segment pair; blockIdx.x and the
// warp pick units of the segment's groups, so no division is needed per
// group.  g/16 lanes per group of g elements (quant.cuh); a warp works on 512
// adjacent elements at a time (a "unit": 512/g groups, 1 KB of bf16 input and
// 2 KB of fp32 or 1 KB of 2-byte state, contiguous).
//
// Blocks are small and short: 2 warps taking one unit each with fp32 state,
// 1 warp taking four units with a 2-byte state or none.  Lane 0 issues 1-D
// bulk copies (cp.async.bulk, the TMA engine) of a unit's input and state into
// the warp's shared-memory stage, completing on the stage's mbarrier; the warp
// quantizes the unit from shared memory and stores codes, meta and the new
// state straight to global memory.  With several units per warp, push_stages
// stages keep the next units' copies in flight during compute without holding
// registers.  Many short blocks, placed by the hardware as SMs free up, keep
// HBM busy to the end of the grid: measured faster than one resident wave of
// blocks striding over the segment.  The waits are bounded and their outcome
// is the same for the whole warp: on timeout the warp records
// ECHO_ERR_TIMEOUT, waits once more (bounded) for each copy it still has in
// flight, and returns.  HBM-bound: per element 2 B of input and the state
// read, the state and b/8 B of codes written, plus 4 B of meta a group.
#include "stages.cuh"

namespace echo {
namespace {

// Units per warp: each block's warps take push_units<SF>() units each (0: one
// resident wave of blocks striding over the segment).  An fp32-state unit
// moves 3 KB and one per warp measured fastest; a 2-byte-state (or stateless)
// unit moves 2 KB (1 KB) and four per warp did, two in flight at a time.
#ifndef ECHO_PUSH_UNITS_F32
#define ECHO_PUSH_UNITS_F32 1
#endif
#ifndef ECHO_PUSH_UNITS_2B
#define ECHO_PUSH_UNITS_2B 4
#endif
#ifndef ECHO_PUSH_STAGES
#define ECHO_PUSH_STAGES 2
#endif
template <int SF>
constexpr int push_units() { return SF == kStateF32 ? ECHO_PUSH_UNITS_F32 : ECHO_PUSH_UNITS_2B; }

// Units in flight per warp: no more stages than units.
template <int SF>
constexpr int push_stages() {
  return push_units<SF>() > 0 && push_units<SF>() < ECHO_PUSH_STAGES ? push_units<SF>()
                                                                       : ECHO_PUSH_STAGES;
}

// Warps per push block: small blocks, so that the hardware can fill SMs as
// they free up, but not so many blocks that launching them limits the rate.
#ifndef ECHO_PUSH_WARPS_F32
#define ECHO_PUSH_WARPS_F32 2
#endif
#ifndef ECHO_PUSH_WARPS_2B
#define ECHO_PUSH_WARPS_2B 1
#endif
template <int SF>
constexpr int push_threads() {
  return 32 * (SF == kStateF32 ? ECHO_PUSH_WARPS_F32 : ECHO_PUSH_WARPS_2B);
}

template <int SF>
constexpr size_t push_smem_bytes() {
  return (size_t)(push_threads<SF>() / 32) * push_stages<SF>() * push_unit_bytes<SF>();
}

// Resident blocks per SM the compiler must allow for (0: its own choice).
#ifndef ECHO_PUSH_MIN_BLOCKS
#define ECHO_PUSH_MIN_BLOCKS 0
#endif
#if ECHO_PUSH_MIN_BLOCKS > 0
#define ECHO_PUSH_BOUNDS __launch_bounds__(push_threads<SF>(), ECHO_PUSH_MIN_BLOCKS)
#else
#define ECHO_PUSH_BOUNDS __launch_bounds__(push_threads<SF>())
#endif

template <int BITS, int SF, int MODE, int G>
__global__ void ECHO_PUSH_BOUNDS
push_kernel(const CallArgs a) {
  constexpr int NL = G / 16;                        // lanes per group
  constexpr int GPW = 32 / NL;                      // groups per unit
  constexpr int S = push_stages<SF>();
  constexpr int SB = push_unit_bytes<SF>();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[push_threads<SF>() / 32][S];

  const int P = a.P;
  const int p = (int)blockIdx.y / (P - 1);          // sender
  const int oi = (int)blockIdx.y - p * (P - 1);
  const int o = oi + (oi >= p ? 1 : 0);             // owner of the segment
  const PushPlace pl = push_place<BITS, SF, G>(a, p, o);
  const int64_t Gs = a.Gs;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / NL;                        // group within the unit
  const int q = lane % NL;                          // lane within the group
  const int64_t wg = (int64_t)blockIdx.x * (push_threads<SF>() / 32) + warp;
  const int64_t nw = (int64_t)gridDim.x * (push_threads<SF>() / 32);
  const int64_t nunits = (Gs + GPW - 1) / GPW;
  uint8_t* wbuf = smem + (size_t)warp * S * SB;
  const uint32_t bar0 = smem_addr(&bars[warp][0]);

  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < S; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
  }
  __syncwarp();
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint64_t pol = 0;
  if (lane == 0) pol = policy_evict_first();        // input and state are read once per call
  const uint64_t codes_pol = kCodesPolicyLast ? policy_evict_last() : policy_evict_normal();
  // Lane 0: start the copies of iteration i into stage st.
  auto issue = [&](int64_t i, int st) {
    const int64_t ud = wg + i * nw;
    if (ud >= nunits) return;
    const int64_t g0 = GPW * ud;
    const uint32_t ng = (uint32_t)((Gs - g0) < GPW ? (Gs - g0) : GPW);
    push_issue<SF, G>(pl, g0, ng, wbuf + st * SB, bar0 + 8 * st, pol);
  };
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < S; ++st) issue(st, st);
  }

  for (int64_t i = 0; wg + i * nw < nunits; ++i) {
    const int st = (int)(i % S);
    const uint32_t parity = (uint32_t)((i / S) & 1);
    if (!mbar_wait_warp(bar0 + 8 * st, parity)) {        // same outcome for every lane
      if (lane == 0) {
        atomicOr(a.status, kStatusTimeout);
        for (int k = 0; k < S; ++k) {             // copies still in flight
          const int64_t ii = i + k;
          if (wg + ii * nw < nunits)
            mbar_wait_bounded(bar0 + 8 * (int)(ii % S), (uint32_t)((ii / S) & 1));
        }
      }
      return;
    }
    const int64_t j = GPW * (wg + i * nw) + sub;     // this lane's group
    const bool valid = j < Gs;
    float v[16];
    if (valid) {
      push_load<SF, G>(wbuf + st * SB, wbuf + st * SB + kUnitX, sub, q, v);
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = 0.0f;      // idle lanes of a short unit
    }
    // The stage has been read into registers: hand it back to the copy engine.
    __syncwarp();
    if (lane == 0) {
      fence_proxy_async();
      issue(i + S, st);
    }
    if (SF != kNoState && a.decay != 1.0f)           // uniform: decayed error feedback
      push_finish<BITS, SF, MODE, G, true>(a, v, valid, j, q, pl.es, pl.cs, pl.ms, codes_pol);
    else
      push_finish<BITS, SF, MODE, G, false>(a, v, valid, j, q, pl.es, pl.cs, pl.ms, codes_pol);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int BITS, int SF, int MODE, int G>
cudaError_t launch_t(const CallArgs& a, cudaStream_t s, bool pdl) {
  static CachedInt resident_cache[64];
  int dev = 0;
  cudaGetDevice(&dev);
  CachedInt& cached = resident_cache[dev & 63];
  int resident = cached.get();
  if (resident == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(push_kernel<BITS, SF, MODE, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)push_smem_bytes<SF>());
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, push_kernel<BITS, SF, MODE, G>,
                                                  push_threads<SF>(), push_smem_bytes<SF>());
    resident = sms * (per_sm > 0 ? per_sm : 1);
    cached.set(resident);
  }
  const int pairs = a.P * (a.P - 1);
  // Blocks per segment: push_units units for each warp, or one resident wave
  // across all segments; never more than one unit for each warp.
  const int64_t per_block = (int64_t)(push_threads<SF>() / 32) * (32 / (G / 16));
  const int64_t need = (a.Gs + per_block - 1) / per_block;
  constexpr int U = push_units<SF>();
  int64_t bx = U > 0 ? (need + U - 1) / U : (resident + pairs - 1) / pairs;
  if (bx > need) bx = need;
  if (a.grid_cap > 0 && bx > a.grid_cap) bx = a.grid_cap;
  if (bx < 1) bx = 1;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)bx, (unsigned)pairs);
  cfg.blockDim = dim3(push_threads<SF>());
  cfg.dynamicSmemBytes = push_smem_bytes<SF>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, push_kernel<BITS, SF, MODE, G>, a);
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
cudaError_t launch_push_g(const CallArgs& a, int bits, cudaStream_t s, bool pdl) {
  if (a.mode == kNaiveZeroPoint) return launch_mode<kNaiveZeroPoint, G>(a, bits, s, pdl);
  if (a.mode == kSymmetric) return launch_mode<kSymmetric, G>(a, bits, s, pdl);
  return launch_mode<kZeroAware, G>(a, bits, s, pdl);
}

#ifndef ECHO_G
#define ECHO_G 128
#endif
static_assert(group_supported(ECHO_G), "ECHO_G: 64, 128 or 256");
template cudaError_t launch_push_g<ECHO_G>(const CallArgs&, int, cudaStream_t, bool);

}  // namespace echo
