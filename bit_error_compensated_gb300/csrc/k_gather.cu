// k_gather.cu -- the gather of the quantized P2P all-reduce ("Echo: Error-
// Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)): every rank,
// the owner included, decodes the same gather codes of every segment, so all
// P outputs hold identical bits.  With the ranks in one GPU's memory, the
// all-gather is one read of each segment's codes and P writes of the decoded
// bf16 values.
//
// g/8 lanes per group of g elements, 8 consecutive elements per lane: a warp
// reads the codes and meta words of 256/g adjacent groups (256 elements) and
// writes, per rank, one 16-byte streaming store per lane (512 B per warp).
// U such runs per warp are read before any is written, to keep several code
// reads in flight.  Write-bound: P * 2 bytes out per element.
#include "stages.cuh"

namespace echo {
namespace {

template <int BITS, int U, int MODE, int G>
__global__ void __launch_bounds__(kThreads)
gather_kernel(const CallArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t wg = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const int64_t nw = (int64_t)gridDim.x * (kThreads / 32);
  const int64_t runs = (a.Gs * G + kRun - 1) / kRun;
  gather_runs<BITS, U, MODE, G>(a, (int)blockIdx.y, wg, nw, runs);   // blockIdx.y: owner segment
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#ifndef ECHO_GATHER_UNROLL
#define ECHO_GATHER_UNROLL 4
#endif
constexpr int kGatherUnroll = ECHO_GATHER_UNROLL;  // warp runs in flight per warp

// 1: one pass of kGatherUnroll runs per warp, as many blocks as that takes;
// 0: one resident wave of blocks striding over the segment.
#ifndef ECHO_GATHER_ONE_PASS
#define ECHO_GATHER_ONE_PASS 1
#endif

template <int BITS, int MODE, int G>
cudaError_t launch_t(const CallArgs& a, cudaStream_t s, bool pdl) {
  static CachedInt grid_cache[64];
  int dev = 0;
  cudaGetDevice(&dev);
  CachedInt& cached = grid_cache[dev & 63];
  int grid = cached.get();
  if (grid == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_kernel<BITS, kGatherUnroll, MODE, G>,
                                                  kThreads, 0);
    grid = sms * (per_sm > 0 ? per_sm : 1);
    cached.set(grid);
  }
  // Blocks per owner segment: one pass per warp (or one resident wave across
  // the P segments), but no more than the segment has warp runs for.
  const int64_t per_block = (int64_t)(kThreads / 32) * kGatherUnroll * (256 / G);
  const int64_t need = (a.Gs + per_block - 1) / per_block;
  int64_t bx = ECHO_GATHER_ONE_PASS ? need : (grid + a.P - 1) / a.P;
  if (bx > need) bx = need;
  if (a.grid_cap > 0 && bx > a.grid_cap) bx = a.grid_cap;
  if (bx < 1) bx = 1;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)bx, (unsigned)a.P);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gather_kernel<BITS, kGatherUnroll, MODE, G>, a);
}

template <int MODE, int G>
cudaError_t launch_mode(const CallArgs& a, int bits, cudaStream_t s, bool pdl) {
  return bits == 4 ? launch_t<4, MODE, G>(a, s, pdl) : launch_t<8, MODE, G>(a, s, pdl);
}

}  // namespace

template <int G>
cudaError_t launch_gather_g(const CallArgs& a, int bits, cudaStream_t s, bool pdl) {
  if (a.mode == kNaiveZeroPoint) return launch_mode<kNaiveZeroPoint, G>(a, bits, s, pdl);
  if (a.mode == kSymmetric) return launch_mode<kSymmetric, G>(a, bits, s, pdl);
  return launch_mode<kZeroAware, G>(a, bits, s, pdl);
}

#ifndef ECHO_G
#define ECHO_G 128
#endif
static_assert(group_supported(ECHO_G), "ECHO_G: 64, 128 or 256");
template cudaError_t launch_gather_g<ECHO_G>(const CallArgs&, int, cudaStream_t, bool);

}  // namespace echo
