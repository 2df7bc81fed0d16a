// echo_api.cu -- host side of libecho.so: plans, argument checks, launches.
// The operation and every call's contract are described in include/echo.h.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "echo_internal.h"

using echo::CallArgs;

struct echo_plan_s {
  int P = 0, g = 0, bits = 0, device = 0;
  int64_t n = 0, m = 0, Gs = 0, Gs_pad = 0, CB = 0;
  uint8_t* wire = nullptr;          // push codes/meta, gather codes/meta (inside wire_alloc)
  uint8_t* wire_alloc = nullptr;    // the allocation: guard band, wire, guard band
  size_t wire_bytes = 0;
  int64_t off[4] = {0, 0, 0, 0};
  float* comp = nullptr;            // the plan's own compensator state (inside comp_alloc)
  uint8_t* comp_alloc = nullptr;    // guard band, state (fp32-sized), guard band
  size_t comp_bytes = 0;
  int* status = nullptr;            // device status word
  cudaStream_t last_stream = nullptr;
  int fused = 1;                    // the reduce kernel writes the outputs (no gather kernel)
  int mode = ECHO_QUANT_ZERO_AWARE;
  int state_fmt = ECHO_STATE_F32;   // ECHO_STATE_*
  float decay = 1.0f;
  int persistent = 0;               // one persistent kernel per call (k_call.cu)
  int tile = ECHO_TILE_AUTO;        // one kernel, each block a whole owner tile (k_tile.cu)
  int sms = 0;                      // SMs of the plan's device
  uint32_t* sched = nullptr;        // its schedule words, zero between calls
  int64_t tiles = 0;                // reduce tiles per segment
  int64_t hold = -1;                // test hook, see echo_debug_hold_push
  int grid_cap = 0;                 // debug: see echo_debug_set_grid
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  int timing = 0;
};

namespace {

thread_local cudaError_t g_last_cuda = cudaSuccess;

int cuda_fail(cudaError_t e) {
  g_last_cuda = e;
  return ECHO_ERR_CUDA;
}

#define ECHO_CUDA(call)                              \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return cuda_fail(e_);     \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool overlap(uintptr_t a, uintptr_t b, size_t bytes) {
  return a < b + bytes && b < a + bytes;
}

int check_device(const echo_plan_s* plan) {
  int dev = -1;
  ECHO_CUDA(cudaGetDevice(&dev));
  return dev == plan->device ? ECHO_OK : ECHO_ERR_ARG;
}

bool g_kernels_prepared[64] = {false};   // guarded by g_prepare_mutex
std::mutex g_prepare_mutex;

// Guard bands around the plan's receive slots and state: filled with a fixed
// byte at plan time and checked by echo_debug_check_guards.
constexpr size_t kGuard = 256;
constexpr int kGuardByte = 0xA5;

// NVTX ranges (domain "echo") around each call, for timeline tools; without
// a tool attached they cost a branch.
nvtxDomainHandle_t nvtx_domain() {
  static nvtxDomainHandle_t d = nvtxDomainCreateA("echo");
  return d;
}
struct NvtxRange {
  explicit NvtxRange(const char* name) {
    nvtxEventAttributes_t attr = {};
    attr.version = NVTX_VERSION;
    attr.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    attr.messageType = NVTX_MESSAGE_TYPE_ASCII;
    attr.message.ascii = name;
    nvtxDomainRangePushEx(nvtx_domain(), &attr);
  }
  ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
};

}  // namespace

namespace echo {
int note_cuda_error(cudaError_t e) { return cuda_fail(e); }

#define ECHO_BY_GROUP(g, call) ((g) == 64 ? call<64> : (g) == 256 ? call<256> : call<128>)

cudaError_t launch_push(const CallArgs& a, int g, int bits, cudaStream_t s, bool pdl) {
  return ECHO_BY_GROUP(g, launch_push_g)(a, bits, s, pdl);
}
cudaError_t launch_reduce(const CallArgs& a, int g, int bits, bool fused, cudaStream_t s, bool pdl) {
  return ECHO_BY_GROUP(g, launch_reduce_g)(a, bits, fused, s, pdl);
}
cudaError_t launch_gather(const CallArgs& a, int g, int bits, cudaStream_t s, bool pdl) {
  return ECHO_BY_GROUP(g, launch_gather_g)(a, bits, s, pdl);
}
cudaError_t launch_call(const CallArgs& a, const CallSched& sch, int g, int bits, bool fused,
                        cudaStream_t s) {
  return ECHO_BY_GROUP(g, launch_call_g)(a, sch, bits, fused, s);
}
cudaError_t launch_tile(const CallArgs& a, int g, int bits, bool rank_parallel, cudaStream_t s,
                        bool pdl) {
  return ECHO_BY_GROUP(g, launch_tile_g)(a, bits, rank_parallel, s, pdl);
}
#undef ECHO_BY_GROUP

cudaError_t prepare_kernels() {
  cudaError_t e = cudaSuccess, r;
  if ((r = prepare_reduce_g<64>()) != cudaSuccess) e = r;
  if ((r = prepare_reduce_g<128>()) != cudaSuccess) e = r;
  if ((r = prepare_reduce_g<256>()) != cudaSuccess) e = r;
  if ((r = prepare_tile_g<64>()) != cudaSuccess) e = r;
  if ((r = prepare_tile_g<128>()) != cudaSuccess) e = r;
  if ((r = prepare_tile_g<256>()) != cudaSuccess) e = r;
  return e;
}
}  // namespace echo

namespace {
// The tile schedule's form for a call of the plan: rank-parallel blocks when
// the grid (one block per owner tile) is too small to keep the SMs busy with
// the rank loop's small blocks, whose per-block path is P pushes long.
#ifndef ECHO_TILE_RP_TILES_PER_SM
#define ECHO_TILE_RP_TILES_PER_SM 4
#endif
bool tile_rank_parallel(const echo_plan_s* plan) {
  if (plan->tile == ECHO_TILE_RANK_PARALLEL) return true;
  if (plan->tile != ECHO_TILE_AUTO || plan->P < 2) return false;
  const int64_t T = echo::kReduceTileElems / plan->g;
  const int64_t blocks = (plan->Gs + T - 1) / T * plan->P;
  return blocks <= (int64_t)ECHO_TILE_RP_TILES_PER_SM * plan->sms;
}
}  // namespace

extern "C" {

int echo_plan(int P, int64_t n, int g, int bits, echo_plan_t* out) {
  if (out == nullptr) return ECHO_ERR_ARG;
  *out = nullptr;
  if (P < 1 || P > ECHO_MAX_RANKS || g < 1) return ECHO_ERR_ARG;
  if (bits != 4 && bits != 8) return ECHO_ERR_UNSUPPORTED;
  if (!echo::group_supported(g)) return ECHO_ERR_UNSUPPORTED;
  if (n < 0 || n % ((int64_t)P * g) != 0) return ECHO_ERR_SHAPE;
  if (n > ((int64_t)1 << 40)) return ECHO_ERR_SHAPE;

  echo_plan_s* p = new (std::nothrow) echo_plan_s();
  if (p == nullptr) return ECHO_ERR_ARG;
  p->P = P;
  p->g = g;
  p->bits = bits;
  p->n = n;
  p->m = n / P;
  p->Gs = p->m / g;
  p->Gs_pad = (p->Gs + 3) / 4 * 4;
  p->CB = (int64_t)g * bits / 8;

  const size_t codes1 = (size_t)P * (P - 1) * p->Gs * p->CB;
  const size_t meta1 = (size_t)P * (P - 1) * p->Gs_pad * 4;
  const size_t codes2 = (size_t)P * p->Gs * p->CB;
  const size_t meta2 = (size_t)P * p->Gs_pad * 4;
  p->off[0] = 0;
  p->off[1] = (int64_t)align_up(p->off[0] + codes1, 256);
  p->off[2] = (int64_t)align_up(p->off[1] + meta1, 256);
  p->off[3] = (int64_t)align_up(p->off[2] + codes2, 256);
  p->wire_bytes = align_up(p->off[3] + meta2, 256);
  p->comp_bytes = (size_t)P * n * sizeof(float);
  const int64_t T = echo::kCallTileElems / g;       // tiles of the persistent schedule
  p->tiles = (p->Gs + T - 1) / T;
  const size_t sched_bytes = (size_t)echo::sched_words(P, p->tiles) * sizeof(uint32_t);

  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e == cudaSuccess && p->device >= 0 && p->device < 64) {
    std::lock_guard<std::mutex> lock(g_prepare_mutex);
    if (!g_kernels_prepared[p->device]) {
      e = echo::prepare_kernels();
      if (e == cudaSuccess) g_kernels_prepared[p->device] = true;
    }
  }
  if (e == cudaSuccess && p->wire_bytes > 0) {
    e = cudaMalloc((void**)&p->wire_alloc, p->wire_bytes + 2 * kGuard);
    p->wire = p->wire_alloc + kGuard;
    if (e == cudaSuccess) e = cudaMemset(p->wire_alloc, kGuardByte, kGuard);
    if (e == cudaSuccess) e = cudaMemset(p->wire + p->wire_bytes, kGuardByte, kGuard);
  }
  if (e == cudaSuccess && p->comp_bytes > 0) {
    e = cudaMalloc((void**)&p->comp_alloc, p->comp_bytes + 2 * kGuard);
    p->comp = reinterpret_cast<float*>(p->comp_alloc + kGuard);
    if (e == cudaSuccess) e = cudaMemset(p->comp_alloc, kGuardByte, kGuard);
    if (e == cudaSuccess) e = cudaMemset(p->comp_alloc + kGuard + p->comp_bytes, kGuardByte, kGuard);
  }
  if (e == cudaSuccess) e = cudaMalloc((void**)&p->status, sizeof(int));
  if (e == cudaSuccess) e = cudaMalloc((void**)&p->sched, sched_bytes);
  if (e == cudaSuccess) e = cudaMemset(p->sched, 0, sched_bytes);
  if (e == cudaSuccess && p->wire_bytes > 0) e = cudaMemset(p->wire, 0, p->wire_bytes);
  if (e == cudaSuccess && p->comp_bytes > 0) e = cudaMemset(p->comp, 0, p->comp_bytes);
  if (e == cudaSuccess) e = cudaMemset(p->status, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    echo_plan_destroy(p);
    return cuda_fail(e);
  }
  *out = p;
  return ECHO_OK;
}

int echo_allreduce(echo_plan_t plan, const void* const* in, void* const* out,
                   void* comp_state, void* stream) {
  if (plan == nullptr || in == nullptr || out == nullptr) return ECHO_ERR_ARG;
  const int P = plan->P;
  const size_t bytes = (size_t)plan->n * 2;
  for (int p = 0; p < P; ++p) {
    if (in[p] == nullptr || out[p] == nullptr) return ECHO_ERR_ARG;
    if (!aligned16(in[p]) || !aligned16(out[p])) return ECHO_ERR_ALIGN;
  }
  float* comp = nullptr;
  if (comp_state == ECHO_COMP_DEFAULT) {
    comp = plan->comp;
  } else if (comp_state != nullptr) {
    if (((uintptr_t)comp_state & 31u) != 0) return ECHO_ERR_ALIGN;   // 32-byte state stores
    comp = static_cast<float*>(comp_state);
  }
  // Aliasing: out[p] may be in[p]; otherwise outputs overlap nothing, and the
  // state overlaps no input or output.
  for (int p = 0; p < P; ++p) {
    const uintptr_t op = (uintptr_t)out[p];
    for (int q = 0; q < P; ++q) {
      const uintptr_t iq = (uintptr_t)in[q];
      if (op == iq && p == q) continue;
      if (overlap(op, iq, bytes)) return ECHO_ERR_ARG;
      if (q != p && overlap(op, (uintptr_t)out[q], bytes)) return ECHO_ERR_ARG;
    }
    if (comp != nullptr && plan->comp_bytes > 0) {
      const uintptr_t c = (uintptr_t)comp;
      if (c < op + bytes && op < c + plan->comp_bytes) return ECHO_ERR_ARG;
      if (c < (uintptr_t)in[p] + bytes && (uintptr_t)in[p] < c + plan->comp_bytes) return ECHO_ERR_ARG;
    }
  }
  int rc = check_device(plan);
  if (rc != ECHO_OK) return rc;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  plan->last_stream = s;
  if (plan->n == 0) return ECHO_OK;

  CallArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int p = 0; p < P; ++p) {
    a.in[p] = static_cast<const __nv_bfloat16*>(in[p]);
    a.out[p] = static_cast<__nv_bfloat16*>(out[p]);
  }
  a.comp = comp;
  a.codes1 = plan->wire + plan->off[0];
  a.meta1 = reinterpret_cast<uint32_t*>(plan->wire + plan->off[1]);
  a.codes2 = plan->wire + plan->off[2];
  a.meta2 = reinterpret_cast<uint32_t*>(plan->wire + plan->off[3]);
  a.status = plan->status;
  a.n = plan->n;
  a.Gs = plan->Gs;
  a.Gs_pad = plan->Gs_pad;
  a.P = P;
  a.mode = plan->mode;
  a.state_fmt = plan->state_fmt;
  a.decay = plan->decay;
  a.grid_cap = plan->grid_cap;
  NvtxRange range(plan->persistent ? "echo_allreduce (persistent)"
                  : plan->tile && plan->fused ? "echo_allreduce (tile-fused)"
                  : plan->fused ? "echo_allreduce" : "echo_allreduce (separate gather)");

  // Programmatic dependent launch lets each kernel's blocks be scheduled while
  // the previous kernel drains; every kernel waits (griddepcontrol.wait) before
  // touching data the previous one wrote.  Timing events in between make each
  // launch an ordinary stream-ordered one.
  if (plan->tile && plan->fused && !plan->persistent) {
    if (plan->timing) ECHO_CUDA(cudaEventRecord(plan->ev[0], s));
    ECHO_CUDA(echo::launch_tile(a, plan->g, plan->bits, tile_rank_parallel(plan), s,
                                plan->timing == 0));
    if (plan->timing) {
      for (int k = 1; k < 4; ++k) ECHO_CUDA(cudaEventRecord(plan->ev[k], s));
    }
    return ECHO_OK;
  }
  if (plan->persistent) {
    echo::CallSched sch;
    sch.tiles = plan->tiles;
    sch.round = sch.lag = sch.total = 0;       // set by the launcher
    sch.hold = plan->hold;
    sch.push_done = plan->sched;
    sch.reduce_done = plan->sched + (int64_t)P * plan->tiles;
    sch.ctrl = plan->sched + 2 * (int64_t)P * plan->tiles;
    if (plan->timing) ECHO_CUDA(cudaEventRecord(plan->ev[0], s));
    ECHO_CUDA(echo::launch_call(a, sch, plan->g, plan->bits, plan->fused != 0, s));
    if (plan->timing) {
      for (int k = 1; k < 4; ++k) ECHO_CUDA(cudaEventRecord(plan->ev[k], s));
    }
    return ECHO_OK;
  }
  const bool pdl = plan->timing == 0;
  if (plan->timing) ECHO_CUDA(cudaEventRecord(plan->ev[0], s));
  if (P > 1) ECHO_CUDA(echo::launch_push(a, plan->g, plan->bits, s, pdl));
  if (plan->timing) ECHO_CUDA(cudaEventRecord(plan->ev[1], s));
  ECHO_CUDA(echo::launch_reduce(a, plan->g, plan->bits, plan->fused != 0, s, pdl));
  if (plan->timing) ECHO_CUDA(cudaEventRecord(plan->ev[2], s));
  if (!plan->fused) ECHO_CUDA(echo::launch_gather(a, plan->g, plan->bits, s, pdl));
  if (plan->timing) ECHO_CUDA(cudaEventRecord(plan->ev[3], s));
  return ECHO_OK;
}

int echo_reset_comp(echo_plan_t plan) {
  if (plan == nullptr) return ECHO_ERR_ARG;
  return echo_reset_comp_async(plan, ECHO_COMP_DEFAULT, plan->last_stream);
}

int echo_reset_comp_async(echo_plan_t plan, void* comp_state, void* stream) {
  if (plan == nullptr || comp_state == nullptr) return ECHO_ERR_ARG;
  void* dst = comp_state == ECHO_COMP_DEFAULT ? (void*)plan->comp : comp_state;
  if (plan->comp_bytes == 0) return ECHO_OK;
  int rc = check_device(plan);
  if (rc != ECHO_OK) return rc;
  ECHO_CUDA(cudaMemsetAsync(dst, 0, plan->comp_bytes, static_cast<cudaStream_t>(stream)));
  return ECHO_OK;
}

size_t echo_comp_bytes(echo_plan_t plan) { return plan ? plan->comp_bytes : 0; }

size_t echo_wire_bytes(echo_plan_t plan) { return plan ? plan->wire_bytes : 0; }

int echo_wire_layout(echo_plan_t plan, int64_t* desc) {
  if (plan == nullptr || desc == nullptr) return ECHO_ERR_ARG;
  for (int k = 0; k < 4; ++k) desc[k] = plan->off[k];
  desc[4] = plan->Gs;
  desc[5] = plan->Gs_pad;
  desc[6] = plan->CB;
  desc[7] = (int64_t)plan->wire_bytes;
  return ECHO_OK;
}

int echo_get_status(echo_plan_t plan, void* stream, int* status) {
  if (plan == nullptr || status == nullptr) return ECHO_ERR_ARG;
  int rc = check_device(plan);
  if (rc != ECHO_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  ECHO_CUDA(cudaMemcpyAsync(&word, plan->status, sizeof(int), cudaMemcpyDeviceToHost, s));
  ECHO_CUDA(cudaMemsetAsync(plan->status, 0, sizeof(int), s));
  ECHO_CUDA(cudaStreamSynchronize(s));
  *status = (word & echo::kStatusTimeout) ? ECHO_ERR_TIMEOUT
            : (word & echo::kStatusOverflow) ? ECHO_ERR_OVERFLOW : ECHO_OK;
  if (word & echo::kStatusTimeout) {
    // A persistent call that gave up leaves its schedule words part-way:
    // clear them so that the next call starts clean.
    ECHO_CUDA(cudaMemsetAsync(plan->sched, 0,
                              (size_t)echo::sched_words(plan->P, plan->tiles) * sizeof(uint32_t), s));
    ECHO_CUDA(cudaStreamSynchronize(s));
  }
  return ECHO_OK;
}

int echo_debug_wire(echo_plan_t plan, void* host_dst, size_t bytes, void* stream) {
  if (plan == nullptr || host_dst == nullptr) return ECHO_ERR_ARG;
  if (bytes < plan->wire_bytes) return ECHO_ERR_ARG;
  if (plan->wire_bytes == 0) return ECHO_OK;
  int rc = check_device(plan);
  if (rc != ECHO_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ECHO_CUDA(cudaMemcpyAsync(host_dst, plan->wire, plan->wire_bytes, cudaMemcpyDeviceToHost, s));
  ECHO_CUDA(cudaStreamSynchronize(s));
  return ECHO_OK;
}

int echo_set_fused(echo_plan_t plan, int fused) {
  if (plan == nullptr || (fused != 0 && fused != 1)) return ECHO_ERR_ARG;
  plan->fused = fused;
  return ECHO_OK;
}

int echo_set_tile_fused(echo_plan_t plan, int on) {
  if (plan == nullptr || on < ECHO_TILE_OFF || on > ECHO_TILE_RANK_PARALLEL) return ECHO_ERR_ARG;
  plan->tile = on;
  return ECHO_OK;
}

int echo_set_persistent(echo_plan_t plan, int on) {
  if (plan == nullptr || (on != 0 && on != 1)) return ECHO_ERR_ARG;
  // Tickets are 32-bit: at most 3 tiles rounds of P (P+1) tickets (plus the
  // claims that find none).
  if (on && 3 * (int64_t)plan->P * (plan->P + 1) * plan->tiles > ((int64_t)1 << 31))
    return ECHO_ERR_UNSUPPORTED;
  plan->persistent = on;
  return ECHO_OK;
}

int echo_debug_set_grid(echo_plan_t plan, int blocks) {
  if (plan == nullptr || blocks < 0) return ECHO_ERR_ARG;
  plan->grid_cap = blocks;
  return ECHO_OK;
}

int echo_debug_check_guards(echo_plan_t plan, int* intact) {
  if (plan == nullptr || intact == nullptr) return ECHO_ERR_ARG;
  *intact = 1;
  int rc = check_device(plan);
  if (rc != ECHO_OK) return rc;
  const size_t state_alloc = (size_t)plan->P * plan->n * sizeof(float);
  const uint8_t* bands[4] = {
      plan->wire_alloc, plan->wire_alloc ? plan->wire + plan->wire_bytes : nullptr,
      plan->comp_alloc, plan->comp_alloc ? plan->comp_alloc + kGuard + state_alloc : nullptr};
  uint8_t host[kGuard];
  for (const uint8_t* b : bands) {
    if (b == nullptr) continue;
    ECHO_CUDA(cudaMemcpy(host, b, kGuard, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < kGuard; ++i)
      if (host[i] != kGuardByte) *intact = 0;
  }
  return ECHO_OK;
}

int echo_debug_hold_push(echo_plan_t plan, int64_t item) {
  if (plan == nullptr || item < -1) return ECHO_ERR_ARG;
  plan->hold = item;
  return ECHO_OK;
}

int echo_set_quantizer(echo_plan_t plan, int mode) {
  if (plan == nullptr || mode < ECHO_QUANT_ZERO_AWARE || mode > ECHO_QUANT_SYMMETRIC) return ECHO_ERR_ARG;
  plan->mode = mode;
  return ECHO_OK;
}

int echo_set_state(echo_plan_t plan, int format, float decay) {
  if (plan == nullptr || (format != ECHO_STATE_F32 && format != ECHO_STATE_BF16 &&
                          format != ECHO_STATE_F16))
    return ECHO_ERR_ARG;
  if (!(decay > 0.0f && decay <= 1.0f)) return ECHO_ERR_ARG;      // also rejects NaN
  if (format != plan->state_fmt) {
    int rc = check_device(plan);
    if (rc != ECHO_OK) return rc;
    // The held values mean nothing in another format: start from zero.  The
    // allocation (fp32-sized) serves every format.
    if (plan->comp != nullptr && plan->comp_bytes > 0)
      ECHO_CUDA(cudaMemsetAsync(plan->comp, 0, (size_t)plan->P * plan->n * sizeof(float),
                                plan->last_stream));
    plan->state_fmt = format;
    plan->comp_bytes = (size_t)plan->P * plan->n * (format == ECHO_STATE_F32 ? 4 : 2);
  }
  plan->decay = decay;
  return ECHO_OK;
}

int echo_set_timing(echo_plan_t plan, void* const* events, int count) {
  if (plan == nullptr) return ECHO_ERR_ARG;
  if (count == 0) {
    plan->timing = 0;
    return ECHO_OK;
  }
  if (count != 4 || events == nullptr) return ECHO_ERR_ARG;
  for (int k = 0; k < 4; ++k) {
    if (events[k] == nullptr) return ECHO_ERR_ARG;
    plan->ev[k] = static_cast<cudaEvent_t>(events[k]);
  }
  plan->timing = 1;
  return ECHO_OK;
}

void echo_plan_destroy(echo_plan_t plan) {
  if (plan == nullptr) return;
  if (plan->wire_alloc) cudaFree(plan->wire_alloc);
  if (plan->comp_alloc) cudaFree(plan->comp_alloc);
  if (plan->status) cudaFree(plan->status);
  if (plan->sched) cudaFree(plan->sched);
  delete plan;
}

const char* echo_strerror(int status) {
  switch (status) {
    case ECHO_OK: return "ok";
    case ECHO_ERR_ARG: return "invalid argument";
    case ECHO_ERR_SHAPE: return "n must be a non-negative multiple of P*g";
    case ECHO_ERR_UNSUPPORTED: return "unsupported configuration (bits must be 4 or 8, g must be 64, 128 or 256)";
    case ECHO_ERR_ALIGN: return "device pointer not 16-byte aligned (32 for a compensator state)";
    case ECHO_ERR_CUDA: return cudaGetErrorString(g_last_cuda);
    case ECHO_ERR_OVERFLOW: return "non-finite input or fp16 step overflow in some group";
    case ECHO_ERR_TIMEOUT: return "a device-side wait gave up";
    case ECHO_ERR_TOO_LARGE:
      return "problem needs more receive-slot space than the fixed no-allocation area holds";
    default: return "unknown status";
  }
}

}  // extern "C"
