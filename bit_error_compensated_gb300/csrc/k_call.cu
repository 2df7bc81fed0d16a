// k_call.cu -- one whole all-reduce call ("Echo: Error-Compensated 4-Bit
// Tensor-Parallel Communication", Fig. 2) in a single persistent kernel, the
// one-GPU counterpart of the paper's staggered push / reduce / gather tiles
// (Fig. 2(b)): a reduce tile starts as soon as its P-1 pushes are done and a
// gather tile as soon as its reduce is, with no kernel boundary in between.
//
// Work items, in ticket order, come in rounds: round r holds the push of
// tile r from every sender to every owner, the reduce of tile r - D of every
// owner and (unless the reduce writes the outputs itself) the gather of tile
// r - 2D, where the lag D is about three waves of items in flight
// (kCallLagWaves; one and two waves measured 5% and 0.5% slower), so a reduce
// tile is claimed when its pushes are most likely done and published, and
// pushes, reduces and gathers, which load memory and ALU differently, share
// the GPU.  Slots
// whose tile is out of range are skipped.  A tile is kCallTileElems elements
// of a segment.  A reduce item waits for a per-tile counter of finished
// pushes, a gather item for a per-tile reduce flag; each consumer resets what
// it consumed, and the last block to finish resets the ticket counter, so the
// words are zero again for the next call.
//
// A block is kThreads/32 compute warps and one control warp, which share a
// ring of shared-memory stages (NS of them, two or three, chosen at launch),
// each with a "full" and an "empty" mbarrier.  The control warp's lane 0 does
// all the scheduling: it claims tickets from one atomic counter (the next one
// fetched ahead), waits for an item's inputs, fills a stage with the item's
// bulk copies (cp.async.bulk) completing on its full barrier, and, once the
// compute warps have arrived on the stage's empty barrier, publishes the
// item's completion to the other blocks (a release add or store) and refills
// the stage.  The compute warps only wait on full barriers, compute, and
// arrive on empty barriers: no block barrier and no memory fence is ever on
// their path, so the latencies of the claims, the flags and the release
// fences overlap the arithmetic.
//
// Deadlock freedom: an item only ever waits on items with smaller tickets,
// the launch is cooperative (all blocks co-resident), and the control warp
// never waits for an item's inputs while it holds an item it has not
// published: when the next item's inputs are not final it first lets the
// compute warps finish what it issued and publishes it.  So the waiting item
// with the smallest ticket always has all its inputs on their way, and every
// wait ends.
//
// Every wait is bounded (kWaitLimitNs) and also gives up when another block
// has set the abort word; whoever gives up records ECHO_ERR_TIMEOUT in the
// status word and sets the abort word; the control warp lets the copies it
// issued land (bounded) before the block exits.  echo_get_status clears the
// schedule words after a timeout.
#include "stages.cuh"

namespace echo {
namespace {

constexpr int kPushItem = 0, kReduceItem = 1, kGatherItem = 2, kEmptyItem = 3;
// A push item is one 512-element unit per warp, a gather item two or more
// 256-element runs per warp.
static_assert(kCallTileElems == kUnit * (kThreads / 32), "tile: one push unit per warp");
static_assert(kCallTileElems % (kRun * (kThreads / 32)) == 0, "tile: whole gather runs per warp");

#ifndef ECHO_CALL_LAG_WAVES
#define ECHO_CALL_LAG_WAVES 3
#endif
constexpr int kCallLagWaves = ECHO_CALL_LAG_WAVES;

struct Item {
  int kind, p, o;
  int64_t k;
  int64_t t;        // its ticket
};

// Tickets and rounds fit 32 bits (echo_set_persistent refuses a problem with
// 2^31 or more work items), so the decoding divides in 32 bits, a few times
// cheaper than the 64-bit division on the control thread's path.
__device__ __forceinline__ Item item_of(const CallArgs& a, const CallSched& sch, int64_t t) {
  const int P = a.P;
  const int pairs = P * (P - 1);
  const uint32_t rd = (uint32_t)sch.round;
  const uint32_t r32 = (uint32_t)t / rd;
  const int64_t r = r32;
  const int slot = (int)((uint32_t)t - r32 * rd);
  Item it;
  if (slot < pairs) {
    it.kind = kPushItem;
    it.k = r;
    it.p = slot / (P - 1);
    const int oi = slot - it.p * (P - 1);
    it.o = oi + (oi >= it.p ? 1 : 0);
  } else if (slot < pairs + P) {
    it.kind = kReduceItem;
    it.k = r - sch.lag;
    it.o = it.p = slot - pairs;
  } else {
    it.kind = kGatherItem;
    it.k = r - 2 * sch.lag;
    it.o = it.p = slot - pairs - P;
  }
  if (it.k < 0 || it.k >= sch.tiles) it.kind = kEmptyItem;
  it.t = t;
  return it;
}

// Release forms of the completion signals: the block's results (ordered
// before thread 0 by the barrier) become visible before the counter or flag.
__device__ __forceinline__ void add_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Orders this thread's earlier generic-proxy view of global memory (the
// acquire of a flag) before its later bulk copies reading that memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// A wait that has lasted this long starts reading the abort word (ns).
#ifndef ECHO_ABORT_POLL_NS
#define ECHO_ABORT_POLL_NS 20000
#endif
constexpr uint64_t kAbortPollNs = ECHO_ABORT_POLL_NS;

// The control thread: waits until *w == want, or gives up (bounded, or when
// the abort word is set).  Returns false on giving up.
__device__ __forceinline__ bool wait_word(const uint32_t* w, uint32_t want, const uint32_t* abort) {
  if (ld_acquire(w) == want) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (ld_acquire(w) == want) return true;
    const uint64_t dt = global_ns() - t0;
    if (dt > kWaitLimitNs || (dt > kAbortPollNs && ld_relaxed(abort) != 0)) return false;
  }
}

// Compute warps per block and the block size (plus the control warp).
constexpr int kCallWarps = kThreads / 32;
constexpr int kCallBlockThreads = kThreads + 32;
// Resident blocks per SM the register allocation must allow: 3 blocks of 288
// threads leave 72 registers a thread.
#ifndef ECHO_CALL_MIN_BLOCKS
#define ECHO_CALL_MIN_BLOCKS 3
#endif
constexpr int64_t kSentinel = -1;              // no ticket held in a stage
// Most stages a block's ring can have (the launcher picks 2 or 3 unless
// ECHO_CALL_STAGES asks for more).
constexpr int kCallMaxStages = 4;

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// Finished items the control thread publishes together, behind one GPU-scope
// fence (1: each item by its own release add or store).
#ifndef ECHO_CALL_PUBLISH_BATCH
#define ECHO_CALL_PUBLISH_BATCH 1
#endif
constexpr int kPublishBatch = ECHO_CALL_PUBLISH_BATCH;
static_assert(kPublishBatch >= 1 && kPublishBatch <= 4, "publish batch: 1 to 4 items");

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void add_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Bounded wait on a barrier phase that also gives up once the abort word is
// set.  The abort word is read only once a wait has lasted kAbortPollNs (no
// wait of a healthy call comes near it): thousands of waiting warps reading
// it on every try would load the L2 slice that also serves the ticket
// counter next to it.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   const uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t dt = global_ns() - t0;
    if (dt > kWaitLimitNs || (dt > kAbortPollNs && ld_relaxed(abort) != 0)) return false;
  }
}

template <int BITS, int SF, int MODE, int G, bool FUSED>
__global__ void __launch_bounds__(kCallBlockThreads, ECHO_CALL_MIN_BLOCKS)
call_kernel(const CallArgs a, const CallSched sch, const int NS) {
  constexpr int T = tile_groups<G, kCallTileElems>();
  constexpr int NL = G / 16;
  constexpr int GPW = 32 / NL;
  constexpr int EB = state_bytes<SF>();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kCallMaxStages];
  __shared__ __align__(8) uint64_t empty[kCallMaxStages];
  __shared__ Item s_item[kCallMaxStages];        // the item in each stage (kEmptyItem: stop)
  __shared__ int64_t s_held[kCallMaxStages];     // control: ticket issued into each stage

  const int P = a.P;
  const int64_t Gs = a.Gs;
  const uint32_t sbytes = reduce_stage_bytes<BITS, SF, G, kCallTileElems>(P);
  const uint32_t full0 = smem_addr(&full[0]);
  const uint32_t empty0 = smem_addr(&empty[0]);
  uint32_t* const ticket = sch.ctrl;
  uint32_t* const finished = sch.ctrl + 1;
  uint32_t* const abort = sch.ctrl + 2;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(full0 + 8 * st, 1);
      mbar_init(empty0 + 8 * st, kCallWarps);
      s_held[st] = kSentinel;
    }
    fence_barrier_init();
  }
  __syncthreads();                               // the block's only barrier

  if (warp == kCallWarps) {
    // ------------------------------------------------------------ control ----
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();   // inputs and state are read once per call
    if (ld_relaxed(abort) != 0) atomicOr(a.status, kStatusTimeout);   // an earlier call gave up
    // Is the input of item `it` final?  1 yes (and consumed: the counter or
    // flag is reset for the next call), 0 not yet (only when not `blocking`),
    // -1 gave up (the abort word is then set).
    auto inputs_ready = [&](const Item& it, bool blocking) -> int {
      if (it.kind == kPushItem || (it.kind == kReduceItem && P == 1)) return 1;
      const int64_t tile = (int64_t)it.o * sch.tiles + it.k;
      uint32_t* w = it.kind == kReduceItem ? sch.push_done + tile : sch.reduce_done + tile;
      const uint32_t want = it.kind == kReduceItem ? (uint32_t)(P - 1) : 1u;
      if (blocking) {
        if (!wait_word(w, want, abort)) return -1;
      } else if (ld_acquire(w) != want) {
        return 0;
      }
      *w = 0;                                    // consumed; zero for the next call
      fence_proxy_async_global();                // before bulk copies of what it guards
      return 1;
    };
    // Fills stage st with item `it`: its bulk copies, or for a
    // gather item (which reads the codes from global memory) a plain arrival.
    auto issue = [&](const Item& it, int st) {
      s_item[st] = it;
      const uint32_t bar = full0 + 8 * st;
      uint8_t* stage = smem + (size_t)st * sbytes;
      const int64_t j0 = it.k * T;
      const int tg = (int)((Gs - j0) < T ? (Gs - j0) : T);     // groups in the tile
      if (it.kind == kPushItem) {
        const PushPlace pl = push_place<BITS, SF, G>(a, it.p, it.o);
        mbar_expect_tx(bar, (uint32_t)tg * G * (2u + EB));
        bulk_g2s(smem_addr(stage), pl.xs + j0 * G, (uint32_t)tg * G * 2u, bar, pol);
        if (SF != kNoState)
          bulk_g2s(smem_addr(stage + T * G * 2), pl.es + j0 * G * EB, (uint32_t)tg * G * EB, bar, pol);
      } else if (it.kind == kReduceItem) {
        reduce_issue_own<BITS, SF, G, kCallTileElems>(a, stage, bar, it.o, j0, tg, pol);
        reduce_issue_codes<BITS, SF, G, kCallTileElems>(a, stage, bar, it.o, j0, tg, pol);
      } else {
        mbar_arrive(bar);
      }
    };
    // Publishes the completion of ticket t to the other blocks: the compute
    // warps' writes, ordered before their arrival on the empty barrier that
    // this thread has waited for, are made visible at GPU scope first.
    // Items finished and not yet published, published kPublishBatch at a
    // time behind one fence (a fence, then relaxed writes, is a release of
    // each of them).
    int64_t pend[kPublishBatch];
    int npend = 0;
    auto flush = [&]() {
      if (npend == 0) return;
      if (kPublishBatch > 1) fence_acq_rel_gpu();
      for (int b = 0; b < npend; ++b) {
        const int64_t t = pend[b];
        const Item it = item_of(a, sch, t);
        if (it.kind == kGatherItem || t == sch.hold) continue;
        const int64_t tile = (int64_t)it.o * sch.tiles + it.k;
        if (kPublishBatch == 1) {
          if (it.kind == kPushItem) add_release(sch.push_done + tile, 1u);
          else if (!FUSED) st_release(sch.reduce_done + tile, 1u);
        } else {
          if (it.kind == kPushItem) add_relaxed(sch.push_done + tile, 1u);
          else if (!FUSED) st_relaxed(sch.reduce_done + tile, 1u);
        }
      }
      npend = 0;
    };
    auto publish = [&](int64_t t) {
      pend[npend++] = t;
      if (npend == kPublishBatch) flush();
    };
    // Per stage: the ticket issued into it and not yet published (s_held,
    // in shared memory), and the parity of its next empty and next full
    // phase (bit st of ep and fp, in registers, so that nothing goes to
    // local memory).
    uint32_t ep = 0u, fp = 0u;
    // Waits until the compute warps are done with stage st, which is then
    // free; `done` receives the ticket they finished there (kSentinel if the
    // stage held none or the wait gave up), still to be published.  False if
    // the wait gave up.
    auto free_stage = [&](int st, int64_t& done) -> bool {
      const int64_t h = s_held[st];
      done = kSentinel;
      if (h == kSentinel) return true;
      if (!mbar_wait_or_abort(empty0 + 8 * st, (ep >> st) & 1u, abort)) return false;
      done = h;
      ep ^= 1u << st;
      s_held[st] = kSentinel;
      return true;
    };
    // Frees the stages after st, oldest item first (st + 1, ..., st + NS - 1),
    // publishing what they held.  False if a wait gave up.
    auto drain_others = [&](int st) -> bool {
      for (int k = 1; k < NS; ++k) {
        const int s2 = st + k < NS ? st + k : st + k - NS;
        int64_t d2;
        if (!free_stage(s2, d2)) return false;
        if (d2 != kSentinel) publish(d2);
      }
      return true;
    };
    // The next non-empty ticket, or sch.total when there is none.  The ticket
    // after it is fetched right away and used next time, so the atomic's
    // latency passes while the compute warps work.
    int64_t pre = (int64_t)atomicAdd(ticket, 1u);
    auto take = [&](Item& it) -> int64_t {
      int64_t t = pre;
      for (;;) {
        if (t >= sch.total) {
          pre = sch.total;
          return sch.total;
        }
        it = item_of(a, sch, t);
        if (it.kind != kEmptyItem) break;
        t = (int64_t)atomicAdd(ticket, 1u);
      }
      pre = (int64_t)atomicAdd(ticket, 1u);
      return t;
    };

    bool ok = true;
    int st = 0;                                  // the stage of the next item issued
    int64_t done = kSentinel;                    // finished, not yet published
    for (;;) {
      if (!(ok = free_stage(st, done))) break;
      Item it;
      const int64_t t = take(it);
      if (t >= sch.total) break;
      int r = inputs_ready(it, false);
      if (r == 0) {
        // Not final yet: publish everything this block holds before waiting,
        // so that no block waits while holding an item it has not published.
        if (done != kSentinel) publish(done);
        done = kSentinel;
        if (!(ok = drain_others(st))) break;
        flush();
        r = inputs_ready(it, true);
      }
      if (r < 0) {
        ok = false;
        break;
      }
      // Publish the freed stage's item, then refill the stage.  (Refilling
      // first, so that the release fence waits beside the new copies, measured
      // 4-6% slower: consumers in other blocks then see the item later.)
      if (done != kSentinel) publish(done);
      done = kSentinel;
      issue(it, st);
      fp ^= 1u << st;
      s_held[st] = t;
      st = st + 1 < NS ? st + 1 : 0;
    }
    if (done != kSentinel) publish(done);        // freed at the top of the last pass
    if (ok) ok = drain_others(st);               // the last items issued
    flush();
    if (ok) {
      // Stop the compute warps: a sentinel in the stage they wait on next
      // (free: its item was freed at the top of the loop's last pass).
      s_item[st].kind = kEmptyItem;
      mbar_arrive(full0 + 8 * st);
      fp ^= 1u << st;
    } else {
      atomicOr(a.status, kStatusTimeout);
      atomicExch(abort, 1u);
    }
    // Copies still in flight land before the block can exit (bounded).
    for (int s2 = 0; s2 < NS; ++s2) mbar_wait_bounded(full0 + 8 * s2, ((fp >> s2) & 1u) ^ 1u);
    // The last block to stop claiming resets the ticket counter for the next call.
    __threadfence();
    if (atomicAdd(finished, 1u) == gridDim.x - 1) {
      atomicExch(ticket, 0u);
      atomicExch(finished, 0u);
    }
    return;
  }

  // -------------------------------------------------------------- compute ----
  const uint64_t codes_pol = kCodesPolicyLast ? policy_evict_last() : policy_evict_normal();
  const int64_t runs_total = (Gs * G + kRun - 1) / kRun;
  int st = 0;                                    // the next item's stage and its phase parity
  uint32_t par = 0u;
  for (;;) {
    const bool got = __all_sync(kFull, mbar_wait_or_abort(full0 + 8 * st, par, abort)) != 0;
    if (!got) {
      if (lane == 0) {
        atomicOr(a.status, kStatusTimeout);
        atomicExch(abort, 1u);
      }
      break;
    }
    const volatile Item& vi = s_item[st];
    Item it;
    it.kind = vi.kind;
    if (it.kind == kEmptyItem) break;
    it.p = vi.p;
    it.o = vi.o;
    it.k = vi.k;
    it.t = vi.t;
    const int64_t j0 = it.k * T;
    const int tg = (int)((Gs - j0) < T ? (Gs - j0) : T);
    const uint8_t* stage = smem + (size_t)st * sbytes;
    if (it.kind == kPushItem) {
      // One 512-element unit per warp: groups [j0 + warp*GPW, +GPW) of the tile.
      const PushPlace pl = push_place<BITS, SF, G>(a, it.p, it.o);
      const int sub = lane / NL;
      const int q = lane % NL;
      const int gl = warp * GPW + sub;           // group within the tile
      const bool valid = gl < tg;
      float v[16];
      if (valid) {
        push_load<SF, G>(stage + warp * kUnitX, stage + T * G * 2 + warp * kUnit * EB, sub, q, v);
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = 0.0f;
      }
      push_finish<BITS, SF, MODE, G>(a, v, valid, j0 + gl, q, pl.es, pl.cs, pl.ms, codes_pol);
    } else if (it.kind == kReduceItem) {
      reduce_tile<BITS, SF, FUSED, MODE, G, kCallTileElems, kCallWarps>(a, stage, it.o, j0, tg);
    } else {
      const int64_t r0 = it.k * (T * G / kRun);
      const int64_t r1 = r0 + T * G / kRun < runs_total ? r0 + T * G / kRun : runs_total;
      gather_runs<BITS, (T * G / kRun) / kCallWarps, MODE, G>(a, it.o, r0 + warp, kCallWarps, r1);
    }
    fence_proxy_async();                         // this lane's stage reads before a refill
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    if (++st == NS) {
      st = 0;
      par ^= 1u;
    }
  }
}

// Stages of a block's ring: 0 lets the launcher choose (three when that
// leaves as many resident blocks per SM as two, else two); 2 to 4 asks for
// that many, or as many as fit.  A third stage bought with a resident block
// measured slower (P = 4, fp32 state: 776 against 850 GB/s on 2048 x 4096
// per rank, 882 against 958 on 8192 x 4096): more blocks, each with its own
// scheduling thread, keep more items moving than a deeper ring per block.
// At no cost in blocks (P = 4 with bf16 state, three blocks either way) it
// gained 2% (1017 against 996 GB/s).
#ifndef ECHO_CALL_STAGES
#define ECHO_CALL_STAGES 0
#endif
static_assert(ECHO_CALL_STAGES == 0 || (ECHO_CALL_STAGES >= 2 && ECHO_CALL_STAGES <= kCallMaxStages),
              "persistent kernel: 0 (chosen at launch) or 2..kCallMaxStages stages");

template <int BITS, int SF, int MODE, int G, bool FUSED>
cudaError_t launch_t(const CallArgs& a, const CallSched& sch, cudaStream_t s) {
  // Per device and P: resident blocks x 8 + stages.
  static CachedInt layout_cache[64][ECHO_MAX_RANKS + 1];
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t stage_bytes = reduce_stage_bytes<BITS, SF, G, kCallTileElems>(a.P);
  CachedInt& cached = layout_cache[dev & 63][a.P];
  int layout = cached.get();
  if (layout == 0) {
    auto kernel = call_kernel<BITS, SF, MODE, G, FUSED>;
    int sms = 0, optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    const int dyn_max = optin - (int)fa.sharedSizeBytes;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
    if (e != cudaSuccess) return e;
    // Resident blocks per SM with ns stages (0 when a block does not fit).
    auto per_sm_with = [&](int ns, int& blocks) -> cudaError_t {
      blocks = 0;
      if ((size_t)ns * stage_bytes > (size_t)dyn_max) return cudaSuccess;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, kCallBlockThreads,
                                                           (size_t)ns * stage_bytes);
    };
    int ns = 2, per_sm = 0;
    if ((e = per_sm_with(2, per_sm)) != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    for (int want = 3; want <= (ECHO_CALL_STAGES ? ECHO_CALL_STAGES : 3); ++want) {
      int p2 = 0;
      if ((e = per_sm_with(want, p2)) != cudaSuccess) return e;
      if (p2 >= (ECHO_CALL_STAGES ? 1 : per_sm)) {
        ns = want;
        per_sm = p2;
      }
    }
    layout = sms * per_sm * 8 + ns;
    cached.set(layout);
  }
  const int resident = layout / 8;
  const int NS = layout % 8;
  const size_t smem = (size_t)NS * stage_bytes;
  // Rounds of P(P-1) pushes, P reduces and (unfused) P gathers; the lag is
  // about kCallLagWaves waves of items in flight (one per stage of a block).
  CallSched sc = sch;
  const int P = a.P;
  sc.round = (int64_t)P * (P - 1) + P + (FUSED ? 0 : P);
  int64_t lag = (kCallLagWaves * NS * (int64_t)resident + sc.round - 1) / sc.round;
  if (P == 1) lag = 0;                           // nothing to wait for
  sc.lag = lag < sc.tiles ? lag : sc.tiles;
  sc.total = sc.round * (sc.tiles + (FUSED ? 1 : 2) * sc.lag);
  // Every block resident at once (a cooperative launch checks it), and no
  // more blocks than items.
  const int64_t items = (FUSED ? 1 : 2) * (int64_t)P * sc.tiles + (int64_t)P * (P - 1) * sc.tiles;
  int64_t blocks = items < resident ? items : resident;
  if (a.grid_cap > 0 && blocks > a.grid_cap) blocks = a.grid_cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kCallBlockThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, call_kernel<BITS, SF, MODE, G, FUSED>, a, sc, NS);
}

template <int MODE, int G>
cudaError_t launch_mode(const CallArgs& a, const CallSched& sch, int bits, bool fused,
                        cudaStream_t s) {
  const int sf = state_fmt_of(a.comp, a.state_fmt);
#define ECHO_CALL_SF(B, SFV)                                                                 \
  return fused ? launch_t<B, SFV, MODE, G, true>(a, sch, s) : launch_t<B, SFV, MODE, G, false>(a, sch, s);
  if (bits == 4) {
    if (sf == kStateF32) { ECHO_CALL_SF(4, kStateF32) }
    if (sf == kStateBF16) { ECHO_CALL_SF(4, kStateBF16) }
    if (sf == kStateF16) { ECHO_CALL_SF(4, kStateF16) }
    ECHO_CALL_SF(4, kNoState)
  }
  if (sf == kStateF32) { ECHO_CALL_SF(8, kStateF32) }
  if (sf == kStateBF16) { ECHO_CALL_SF(8, kStateBF16) }
  if (sf == kStateF16) { ECHO_CALL_SF(8, kStateF16) }
  ECHO_CALL_SF(8, kNoState)
#undef ECHO_CALL_SF
}

}  // namespace

template <int G>
cudaError_t launch_call_g(const CallArgs& a, const CallSched& sch, int bits, bool fused,
                          cudaStream_t s) {
  if (a.mode == kNaiveZeroPoint) return launch_mode<kNaiveZeroPoint, G>(a, sch, bits, fused, s);
  if (a.mode == kSymmetric) return launch_mode<kSymmetric, G>(a, sch, bits, fused, s);
  return launch_mode<kZeroAware, G>(a, sch, bits, fused, s);
}

#ifndef ECHO_G
#define ECHO_G 128
#endif
static_assert(group_supported(ECHO_G), "ECHO_G: 64, 128 or 256");
template cudaError_t launch_call_g<ECHO_G>(const CallArgs&, const CallSched&, int, bool, cudaStream_t);

}  // namespace echo
