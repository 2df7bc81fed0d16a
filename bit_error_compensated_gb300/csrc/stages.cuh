// stages.cuh -- the work of each step of one all-reduce call ("Echo: Error-
// Compensated 4-Bit Tensor-Parallel Communication", Fig. 2(a)) on one piece
// of data held in shared memory or registers, shared by the per-step kernels
// (k_push.cu, k_reduce.cu, k_gather.cu) and the single persistent kernel
// (k_call.cu).
//
//   push    a sender quantizes v = x + e of a group of a segment it does not
//           own, sends the codes and meta word to the owner's receive slot and
//           keeps v - deq(q) as its held error;
//   reduce  the owner decodes the P-1 received code tiles, adds them to its own
//           x + e in fp32 in ascending rank order, quantizes the sum once for
//           the gather and keeps sum - y as its held error (y the bf16 value
//           every rank receives);
//   gather  every rank decodes the owner's gather codes.
//
// Group of g elements: g/16 lanes of 16 values each (quant.cuh).
#pragma once

#include "echo_internal.h"
#include "quant.cuh"
#include "tma.cuh"

namespace echo {

// ------------------------------------------------------------------ push ----

// Elements of a push unit: what one warp quantizes at a time (512/g groups).
constexpr int kUnit = 512;
constexpr int kUnitX = kUnit * 2;                  // bf16 bytes of a unit

template <int SF>
constexpr int push_unit_bytes() { return kUnitX + kUnit * state_bytes<SF>(); }

// This lane's 16 values of group `sub` of a unit staged in shared memory (bf16
// input at sx, state at se): x, plus the held error when compensated.
template <int SF, int G>
__device__ __forceinline__ void push_load(const uint8_t* sx, const uint8_t* se, int sub, int q,
                                          float v[16]) {
  constexpr int NL = G / 16;
  const uint4* x8 = reinterpret_cast<const uint4*>(sx);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = sub * G + half_at<NL>(h, q);
    if constexpr (SF != kNoState) {
      float e[8];
      state_load8<SF>(se, i, e);
      entry8(x8[i / 8], e, v + 8 * h);
    } else {
      bf16x8_to_f32(x8[i / 8], v + 8 * h);
    }
  }
}

// The 8 codes of a half (integer-valued floats) packed into one word and
// stored with an L2 policy: 32 bits for 4-bit codes, 64 for 8-bit.
template <int BITS>
__device__ __forceinline__ void store_codes8(uint8_t* p, const float c[8], uint64_t pol) {
  uint32_t w0, w1;
  pack8<BITS>(c, w0, w1);
  if (BITS == 4) st_hint_u32(p, w0 | (w1 << 16), pol);
  else st_hint_u64(p, (uint64_t)w0 | ((uint64_t)w1 << 32), pol);
}

// Quantizes group j of a sender's segment (all 32 lanes call it; lanes whose
// group is not `valid` compute on zeros and store nothing).  cs, ms: the
// receive slot's codes and meta; es: the sender's state of the segment.
template <int BITS, int SF, int MODE, int G, bool DECAY = true>
__device__ __forceinline__ void push_finish(const CallArgs& a, const float v[16], bool valid,
                                            int64_t j, int q, uint8_t* es, uint8_t* cs,
                                            uint32_t* ms, uint64_t codes_pol) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr int NL = G / 16;
  constexpr int CB = G * BITS / 8;
  const GroupGrid gg = group_grid<MODE, NL>(v, L);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {                 // the lane's two halves
    float c[8], d[8];
    quantize8_mode<MODE>(v + 8 * hh, gg, L, c, d);
    if (valid) {
      store_codes8<BITS>(cs + j * CB + half_code_byte<BITS, NL>(hh, q), c, codes_pol);
      if constexpr (SF != kNoState) {
        float r[8];
        sub_n<8>(r, v + 8 * hh, d);
        state_store8<SF, DECAY>(es, j * G + half_at<NL>(hh, q), r, a.decay);
      }
    }
  }
  if (valid && q == 0) {
    st_hint_u32(ms + j, gg.meta, codes_pol);
    if (!gg.finite) atomicOr(a.status, kStatusOverflow);
  }
}

// Where sender p's push of owner o's segment reads and writes.
struct PushPlace {
  const __nv_bfloat16* xs;   // sender's input, segment start
  uint8_t* es;               // sender's state, segment start (nullptr uncompensated)
  uint8_t* cs;               // receive slot codes
  uint32_t* ms;              // receive slot meta
};

template <int BITS, int SF, int G>
__device__ __forceinline__ PushPlace push_place(const CallArgs& a, int p, int o) {
  constexpr int CB = G * BITS / 8;
  const int P = a.P;
  const int slot = o * (P - 1) + (p < o ? p : p - 1);
  PushPlace pl;
  pl.xs = a.in[p] + (int64_t)o * a.Gs * G;
  pl.es = SF != kNoState ? reinterpret_cast<uint8_t*>(a.comp) +
                               ((int64_t)p * a.n + (int64_t)o * a.Gs * G) * state_bytes<SF>()
                         : nullptr;
  pl.cs = a.codes1 + (int64_t)slot * a.Gs * CB;
  pl.ms = a.meta1 + (int64_t)slot * a.Gs_pad;
  return pl;
}

// Lane 0: bulk copies of groups [g0, g0 + ng) of a push place into a unit
// buffer, completing on `bar`.  ng <= 512/g.
template <int SF, int G>
__device__ __forceinline__ void push_issue(const PushPlace& pl, int64_t g0, uint32_t ng,
                                           uint8_t* buf, uint32_t bar, uint64_t pol) {
  constexpr int EB = state_bytes<SF>();
  mbar_expect_tx(bar, ng * G * (2u + EB));
  bulk_g2s(smem_addr(buf), pl.xs + g0 * G, ng * G * 2u, bar, pol);
  if (SF != kNoState) bulk_g2s(smem_addr(buf + kUnitX), pl.es + g0 * G * EB, ng * G * EB, bar, pol);
}

// ---------------------------------------------------------------- reduce ----

// Groups per reduce tile of TE elements.
template <int G, int TE>
constexpr int tile_groups() { return TE / G; }

// Shared-memory stage of one reduce tile of T groups: [P-1][T][CB] received
// codes, [P-1][T] meta words, [T][G] owner bf16 input, [T][G] owner state
// (when compensated).  Every region starts on a 16-byte boundary.
template <int BITS, int SF, int G, int TE>
__host__ __device__ inline uint32_t reduce_stage_bytes(int P) {
  constexpr int T = tile_groups<G, TE>();
  return (uint32_t)((P - 1) * T * (G * BITS / 8 + 4) + T * G * 2 + T * G * state_bytes<SF>());
}

// Thread 0: arms `bar` for the whole tile (t groups from j0 of segment o) and
// copies the owner's own input and state tile into the stage.
template <int BITS, int SF, int G, int TE>
__device__ __forceinline__ void reduce_issue_own(const CallArgs& a, uint8_t* stage, uint32_t bar,
                                                 int o, int64_t j0, int t, uint64_t pol) {
  constexpr int CB = G * BITS / 8;
  constexpr int EB = state_bytes<SF>();
  constexpr int T = tile_groups<G, TE>();
  const int P = a.P;
  const uint32_t meta_bytes = (uint32_t)(((t + 3) & ~3) * 4);
  const int64_t g0 = (int64_t)o * a.Gs + j0;
  mbar_expect_tx(bar, (uint32_t)((P - 1) * (t * CB + meta_bytes) + t * G * (2 + EB)));
  bulk_g2s(smem_addr(stage + (P - 1) * T * (CB + 4)), a.in[o] + g0 * G, (uint32_t)(t * G * 2), bar,
           pol);
  if (SF != kNoState)
    bulk_g2s(smem_addr(stage + (P - 1) * T * (CB + 4) + T * G * 2),
             reinterpret_cast<const uint8_t*>(a.comp) + ((int64_t)o * a.n + g0 * G) * EB,
             (uint32_t)(t * G * EB), bar, pol);
}

// Thread 0: copies the tile's P-1 received code tiles and meta words.  The
// meta copy is rounded up to 4 words (the slot rows are padded to Gs_pad).
template <int BITS, int SF, int G, int TE>
__device__ __forceinline__ void reduce_issue_codes(const CallArgs& a, uint8_t* stage, uint32_t bar,
                                                   int o, int64_t j0, int t, uint64_t pol) {
  constexpr int CB = G * BITS / 8;
  constexpr int T = tile_groups<G, TE>();
  const int P = a.P;
  const uint32_t meta_bytes = (uint32_t)(((t + 3) & ~3) * 4);
  for (int js = 0; js < P - 1; ++js) {
    const int64_t slot = (int64_t)o * (P - 1) + js;
    bulk_g2s(smem_addr(stage + js * T * CB), a.codes1 + (slot * a.Gs + j0) * CB, (uint32_t)(t * CB),
             bar, pol);
    bulk_g2s(smem_addr(stage + (P - 1) * T * CB + js * T * 4), a.meta1 + slot * a.Gs_pad + j0,
             meta_bytes, bar, pol);
  }
}

// Computes one owner tile (t groups from j0 of segment o) held in a stage,
// writing the gather codes, meta, new owner state and (FUSED) all P outputs
// to global memory.  The NW warps of the block take part; no block barrier.
template <int BITS, int SF, bool FUSED, int MODE, int G, int TE, int NW, bool DECAY = true>
__device__ __forceinline__ void reduce_tile(const CallArgs& a, const uint8_t* stage, int o,
                                            int64_t j0, int t) {
  constexpr float L = (float)((1 << BITS) - 1);
  constexpr bool COMP = SF != kNoState;
  constexpr int EB = state_bytes<SF>();
  constexpr int NL = G / 16;                 // lanes per group
  constexpr int GPW = 32 / NL;               // groups per warp per pass
  constexpr int CB = G * BITS / 8;
  constexpr int T = tile_groups<G, TE>();
  const int P = a.P;
  const uint8_t* s_codes = stage;
  const uint32_t* s_meta = reinterpret_cast<const uint32_t*>(stage + (P - 1) * T * CB);
  const uint4* s_x = reinterpret_cast<const uint4*>(stage + (P - 1) * T * (CB + 4));
  const uint8_t* s_e = stage + (P - 1) * T * (CB + 4) + T * G * 2;         // [T] group states
  // The gather reads these codes next: keep them in L2.
  const uint64_t codes_pol = kCodesPolicyLast ? policy_evict_last() : policy_evict_normal();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / NL;
  const int q = lane % NL;
  // GPW groups per warp per pass (NL lanes each, see quant.cuh).
  for (int gq = GPW * warp; gq < t; gq += GPW * NW) {
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
      for (int h = 0; h < 2; ++h) {
        const uint8_t* cw = cg + half_code_byte<BITS, NL>(h, q);
        if (BITS == 4) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(cw);
          decode4_mode<4, MODE>(w, s, zf, term + 8 * h);
          decode4_mode<4, MODE>(w >> 16, s, zf, term + 8 * h + 4);
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(cw);
          decode4_mode<8, MODE>(w.x, s, zf, term + 8 * h);
          decode4_mode<8, MODE>(w.y, s, zf, term + 8 * h + 4);
        }
      }
    };
    // The owner's own term: its bf16 input plus (compensated) its held error.
    auto own_term = [&](float term[16]) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = gs * G + half_at<NL>(h, q);
        if constexpr (COMP) {
          float e[8];
          state_load8<SF>(s_e, i, e);
          entry8(s_x[i / 8], e, term + 8 * h);
        } else {
          bf16x8_to_f32(s_x[i / 8], term + 8 * h);
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
        add_n<16>(acc, acc, term);
      }
      own_term(term);
      add_n<16>(acc, acc, term);
    }
    for (int p = o + 1; p < P; ++p) {
      sender_term(p, term);
      add_n<16>(acc, acc, term);
    }

    // Quantize the sum once for the gather.
    const GroupGrid gg = group_grid<MODE, NL>(acc, L);
    const int64_t grp = (int64_t)o * a.Gs + j0 + gl;           // group index in the rank tensor
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {               // the lane's two halves
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
        state_store8<SF, DECAY>(eo, e, r, a.decay);
      }
      if (FUSED) {
        for (int r = 0; r < P; ++r) __stcs(reinterpret_cast<uint4*>(a.out[r] + e), y);
      }
    }
    if (valid && q == 0) {
      st_hint_u32(a.meta2 + (int64_t)o * a.Gs_pad + j0 + gl, gg.meta, codes_pol);
      if (!gg.finite) atomicOr(a.status, kStatusOverflow);
    }
  }
}

// ---------------------------------------------------------------- gather ----

// Elements of a gather run: what one warp decodes at a time (256/g groups,
// g/8 lanes each, 8 consecutive elements per lane).
constexpr int kRun = 256;

// One warp decodes runs run0, run0 + stride, ... (< run_end) of owner o's
// gather codes and writes every rank's output: U runs are read before any is
// written, to keep several code reads in flight.
template <int BITS, int U, int MODE, int G>
__device__ __forceinline__ void gather_runs(const CallArgs& a, int o, int64_t run0, int64_t stride,
                                            int64_t run_end) {
  constexpr int CB = G * BITS / 8;
  constexpr int LG = G / 8;         // lanes per group
  constexpr int GW = 32 / LG;       // groups per run
  const int lane = threadIdx.x & 31;
  const int sub = lane / LG;
  const int h = lane % LG;          // lane h of a group decodes elements [8h, 8h+8)
  const int P = a.P;
  const int64_t Gs = a.Gs;
  const uint8_t* cs = a.codes2 + (int64_t)o * Gs * CB;
  const uint32_t* ms = a.meta2 + (int64_t)o * a.Gs_pad;
  for (int64_t r0 = run0; r0 < run_end; r0 += stride * U) {
    uint2 word[U];
    uint32_t meta[U];
    int64_t w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t run = r0 + (int64_t)u * stride;
      w[u] = run < run_end ? GW * run + sub : Gs;
      if (w[u] < Gs) {
        // L2-only loads: in the persistent kernel these codes were written by
        // another SM during the same launch.
        meta[u] = __ldcg(ms + w[u]);
        const uint8_t* cg = cs + w[u] * CB;
        if (BITS == 4) {
          word[u].x = __ldcg(reinterpret_cast<const uint32_t*>(cg) + h);
          word[u].y = 0;
        } else {
          word[u] = __ldcg(reinterpret_cast<const uint2*>(cg) + h);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (w[u] >= Gs) continue;
      float s, zf;
      unpack_meta(meta[u], s, zf);
      float deq[8], yb[8];
      if (BITS == 4) {
        decode4_mode<4, MODE>(word[u].x, s, zf, deq);
        decode4_mode<4, MODE>(word[u].x >> 16, s, zf, deq + 4);
      } else {
        decode4_mode<8, MODE>(word[u].x, s, zf, deq);
        decode4_mode<8, MODE>(word[u].y, s, zf, deq + 4);
      }
      const uint4 y = f32x8_to_bf16(deq, yb);
      const int64_t e0 = ((int64_t)o * Gs + w[u]) * G + 8 * h;
      for (int r = 0; r < P; ++r) __stcs(reinterpret_cast<uint4*>(a.out[r] + e0), y);
    }
  }
}

}  // namespace echo
