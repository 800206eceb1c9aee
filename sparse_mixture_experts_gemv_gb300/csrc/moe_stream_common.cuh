// Pieces shared by the record-streaming decode kernels (bf16 experts in
// moe_stream.cu, MXFP4 experts in moe_stream_mx.cu): the CTA layout (16
// consumer warps + 1 producer warp), the router with tagged logits, the
// per-CTA top-k and slot list of a token window, the record ranges of a CTA,
// and the exchange that adds the CTAs' partial outputs.
//
// Tagged words: a 64-bit global word {call tag (high 32 bits), fp32 value}
// written with one single-copy-atomic store. A reader that sees the current
// call's tag also sees the value written with it, so publishing data needs no
// fence and reading it needs no separate barrier. The tag of a call is
// (calls completed) + 1, where calls completed = ctr / G and every CTA adds 1
// to ctr when it leaves: no CTA leaves a call before it has read everything
// the other CTAs of that call publish, and every CTA reads ctr before it
// publishes anything.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_sm100.cuh"

namespace moe {
namespace stream {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;            // + one producer warp
constexpr int kMaxRingGroups = 16;
constexpr int kMaxRouterRows = 16;                   // router rows per CTA
constexpr int kSmemMax = 212 * 1024;                 // dynamic shared memory budget
constexpr long long kSpinBudget = 4000000000LL;      // ~2 s of SM cycles: then give up

MOE_DEV unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Same load without a compiler memory barrier, so that a batch of them can be
// issued back to back (each is still a single-copy-atomic relaxed load).
MOE_DEV unsigned long long ld_relaxed_u64_nc(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
MOE_DEV void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
MOE_DEV void st_relaxed_v2u64(unsigned long long* p, unsigned long long v0, unsigned long long v1) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" :: "l"(p), "l"(v0), "l"(v1) : "memory");
}
MOE_DEV void ld_relaxed_v2u64(const unsigned long long* p, unsigned long long& v0, unsigned long long& v1) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(v0), "=l"(v1) : "l"(p));
}
MOE_DEV unsigned long long tagged(unsigned long long tag, float v) {
  return (tag << 32) | (unsigned long long)__float_as_uint(v);
}
// Barrier among the 16 consumer warps only (the producer warp never joins it).
MOE_DEV void consumers_sync() { asm volatile("bar.sync 1, %0;" :: "n"(kConsumers) : "memory"); }

// Routing of the window, in shared memory.
struct RouteSmem {
  int idx[kMaxDecodeT * kMaxTopK];        // [t][j] selected experts, descending logits
  float w[kMaxDecodeT * kMaxTopK];        // [t][j] renormalised softmax weights
  int slot_of[kMaxDecodeT * kMaxTopK];    // scratch of the slot build
  unsigned tmask[kMaxSlots];              // tokens using each slot
  DecodeMeta meta;                        // slots: distinct experts, first-appearance order
};

// Record range of this CTA. Shared-expert records [sh0, sh1) are known before
// routing; routed records [u0, u1) index the window's D x I (slot, feature)
// pairs. When there are at least G routed pairs the two ranges are balanced
// jointly (a CTA with one more shared record gets one fewer routed record).
// All counts fit 32 bits (U <= 64 slots x 4096 features, G < 1024), and only
// unsigned 32-bit division is used: 64-bit division is a long software
// sequence that would sit on the producer's critical path.
struct Ranges {
  int sh0, sh1;
  int u0, u1;
};
MOE_DEV Ranges cta_ranges(unsigned b, unsigned G, unsigned Is, unsigned U) {
  Ranges r;
  r.sh0 = (int)(b * Is / G);
  r.sh1 = (int)((b + 1) * Is / G);
  if (U >= G) {
    const unsigned N = U + Is;
    r.u0 = (int)(b * N / G) - r.sh0;
    r.u1 = (int)((b + 1) * N / G) - r.sh1;
  } else {
    r.u0 = (int)(b * U / G);
    r.u1 = (int)((b + 1) * U / G);
  }
  return r;
}

// Poll one token's E tagged logit words until all carry `tag`, then select its
// top-k (bounded: false after ~2 s without every word arriving).
template <int GK>
MOE_DEV bool poll_topk(const unsigned long long* words, int E, int k, unsigned long long tag, int lane, int* out_e,
                       float* out_w) {
  uint32_t key[GK][8];
  int jj[GK][8];
  const unsigned long long want = tag & 0xFFFFFFFFull;
  const long long t0 = clock64();
  bool ok = false;
  while (true) {
    unsigned long long w[GK][8];
#pragma unroll
    for (int g = 0; g < GK; ++g)   // every load in flight before any is used
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = lane + 32 * (8 * g + q);
        w[g][q] = (e < E) ? ld_relaxed_u64_nc(words + e) : (want << 32);
      }
    bool mine = true;
#pragma unroll
    for (int g = 0; g < GK; ++g)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = lane + 32 * (8 * g + q);
        mine &= (w[g][q] >> 32) == want;
        key[g][q] = (e < E) ? f32_order_key(__uint_as_float((uint32_t)w[g][q])) : 0u;
      }
    ok = __all_sync(0xFFFFFFFFu, mine);
    if (ok || clock64() - t0 > kSpinBudget) break;
  }
  warp_topk_keys<GK>(key, jj, k, lane, out_e, out_w);
  return ok;
}

// Consumer warps: this CTA's router logits (rows b, b + G, ... of the fp32
// router, at most kMaxRouterRows), split into parts over the 16 warps, summed
// in warp order, plus the router bias and the optional per-token logit bias,
// published as tagged words [t][E]. The row loads are issued before waiting
// for x (x_bar). Every consumer thread has waited on x_bar when this returns.
template <int TMAX>
MOE_DEV void router_publish(const uint16_t* xs, int XP, int T, int H, int E, const float* router_t,
                            const float* router_bias, const float* logit_bias, unsigned long long* words,
                            unsigned long long tag, uint64_t* x_bar, int* err, int* s_abort,
                            float (*s_rpart)[TMAX]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int nr_rows = (E - b + G - 1) / G;
  const int P = max(1, kConsumerWarps / max(nr_rows, 1));     // warps per row
  const int items = nr_rows * P;
  const int H4 = H / 4;
  bool x_ready = false;
  if (warp < items) {
    const int m = warp / P, p = warp - m * P;
    const float* row = router_t + (size_t)(b + m * G) * H;
    const int c0 = p * H4 / P, c1 = (p + 1) * H4 / P;
    float acc[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
    for (int cb = c0; cb < c1; cb += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = cb + lane + 32 * q;
        if (c < c1) v[q] = ldg_stream(row + 4 * c);
      }
      if (!x_ready) {
        volatile int never = 0;
        if (!sm100::mbar_wait(x_bar, 0, err, &never, kSpinBudget, false)) *s_abort = 1;
        x_ready = true;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = cb + lane + 32 * q;
        if (c < c1) {
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (t < T) {
              const uint2 xx = *reinterpret_cast<const uint2*>(xs + t * XP + 4 * c);
              float s = acc[t];
              s = fmaf(__uint_as_float(v[q].x), bf16_lo(xx.x), s);
              s = fmaf(__uint_as_float(v[q].y), bf16_hi(xx.x), s);
              s = fmaf(__uint_as_float(v[q].z), bf16_lo(xx.y), s);
              s = fmaf(__uint_as_float(v[q].w), bf16_hi(xx.y), s);
              acc[t] = s;
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const float sum = warp_sum(acc[t]);
        if (lane == 0) s_rpart[warp][t] = sum;
      }
    }
  }
  if (!x_ready) {   // x is needed later by every warp
    volatile int never = 0;
    if (!sm100::mbar_wait(x_bar, 0, err, &never, kSpinBudget, false)) *s_abort = 1;
  }
  consumers_sync();
  if ((int)threadIdx.x < nr_rows * T) {   // logit = partial sums in warp order + biases
    const int m = threadIdx.x / T, t = threadIdx.x - m * T;
    const int e = b + m * G;
    float sl = 0.f;
    for (int p = 0; p < P; ++p) sl += s_rpart[m * P + p][t];
    sl += router_bias[e];
    if (logit_bias) sl += logit_bias[(size_t)t * E + e];
    st_relaxed_u64(words + (size_t)t * E + e, tagged(tag, sl));
  }
}

// Consumer warps: top-k of every token (warp t polls token t's logits), then
// warp 0 lists the distinct experts of the window in first-appearance order
// (slots) with, per slot, the position j of its expert in each token's top-k
// (-1 if the token did not choose it) and the mask of tokens using it.
// The caller synchronises the CTA before the slots are read.
MOE_DEV void route_window(const unsigned long long* words, int T, int E, int k, unsigned long long tag, RouteSmem& rs,
                          int* err, int* s_abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < T) {
    const int t = warp;
    bool ok;
    if (E <= 256) ok = poll_topk<1>(words + (size_t)t * E, E, k, tag, lane, rs.idx + t * k, rs.w + t * k);
    else ok = poll_topk<2>(words + (size_t)t * E, E, k, tag, lane, rs.idx + t * k, rs.w + t * k);
    if (!ok) {
      if (lane == 0) set_error(err, kDevTimeout);
      *s_abort = 1;
    }
  }
  if (T > 1) consumers_sync();
  if (warp != 0) return;
  if (T == 1) {   // one token: its k experts are the slots, in order
    if (lane < k) {
      const int e = rs.idx[lane];
      if (e < 0 || e >= E) {   // only NaN logits can get here
        set_error(err, kDevCheck);
        *s_abort = 1;
      }
      rs.meta.slot_expert[lane] = e;
      rs.tmask[lane] = 1u;
#pragma unroll
      for (int t = 0; t < kMaxDecodeT; ++t) rs.meta.slot_j[lane][t] = (signed char)(t == 0 ? lane : -1);
    }
    if (lane == 0) rs.meta.num_slots = k;
    return;
  }
  const int n = T * k;
  bool first[2] = {false, false};
  int firstpos[2] = {0, 0};
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int ai = lane + 32 * h2;
    if (ai < n) {
      const int e = rs.idx[ai];
      if (e < 0 || e >= E) {
        set_error(err, kDevCheck);
        *s_abort = 1;
      }
      int q = 0;
      while (rs.idx[q] != e) ++q;
      first[h2] = (q == ai);
      firstpos[h2] = q;
    }
  }
  const unsigned m0 = __ballot_sync(0xFFFFFFFFu, first[0]);
  const unsigned m1 = __ballot_sync(0xFFFFFFFFu, first[1]);
  const unsigned lt = (1u << lane) - 1u;
  if (first[0]) rs.slot_of[lane] = __popc(m0 & lt);
  if (first[1]) rs.slot_of[lane + 32] = __popc(m0) + __popc(m1 & lt);
  __syncwarp();
  const int D = __popc(m0) + __popc(m1);
  for (int q = lane; q < D * kMaxDecodeT; q += 32) rs.meta.slot_j[q / kMaxDecodeT][q % kMaxDecodeT] = -1;
  for (int q = lane; q < D; q += 32) rs.tmask[q] = 0u;
  __syncwarp();
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int ai = lane + 32 * h2;
    if (ai < n) {
      const int slot = rs.slot_of[firstpos[h2]];
      if (first[h2]) rs.meta.slot_expert[slot] = rs.idx[ai];
      rs.meta.slot_j[slot][ai / k] = (signed char)(ai % k);
      atomicOr(&rs.tmask[slot], 1u << (ai / k));
    }
  }
  if (lane == 0) rs.meta.num_slots = D;
}

// Consumer warps, after this CTA published its partial outputs as tagged
// words at partial[(b * H + n) * TP + t] (TP = T rounded up to even): this
// CTA owns output rows [nb0, nb1) for every token. Each thread polls its share
// of the G x rows x TP words (16 bytes at a time) until they carry this call's
// tag and stages the values in shared memory (`stage`, G x rows x TP floats);
// then one warp per output adds the G partials in a fixed order and writes
// bf16. Ends with a consumer barrier.
MOE_DEV void collect_outputs(const unsigned long long* partial, float* stage, unsigned long long tag, int T, int H,
                             uint16_t* out, int* err, int* s_abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int TP = T + (T & 1);
  const int nb0 = (int)((unsigned)b * (unsigned)H / (unsigned)G);
  const int nb1 = (int)((unsigned)(b + 1) * (unsigned)H / (unsigned)G);
  const int nrow = nb1 - nb0;
  const int per = nrow * TP / 2;                      // 16-byte units per CTA partial
  const int units = G * per;
  const unsigned long long want = tag & 0xFFFFFFFFull;
  for (int q0 = threadIdx.x; q0 < units; q0 += 8 * kConsumers) {
    const long long t0 = clock64();
    while (true) {
      unsigned long long v[8][2];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int q = q0 + r * kConsumers;
        v[r][0] = v[r][1] = want << 32;
        if (q < units) {
          const int p = q / per, w2 = q - p * per;
          ld_relaxed_v2u64(partial + ((size_t)p * H + nb0) * TP + 2 * w2, v[r][0], v[r][1]);
        }
      }
      bool ok = true;   // (the pad token of odd T is written too, so both words are checked)
#pragma unroll
      for (int r = 0; r < 8; ++r) ok &= (v[r][0] >> 32) == want && (v[r][1] >> 32) == want;
      if (ok) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int q = q0 + r * kConsumers;
          if (q < units)
            *reinterpret_cast<float2*>(stage + 2 * (size_t)q) =
                make_float2(__uint_as_float((uint32_t)v[r][0]), __uint_as_float((uint32_t)v[r][1]));
        }
        break;
      }
      if (clock64() - t0 > kSpinBudget) {
        set_error(err, kDevTimeout);
        *s_abort = 1;
        break;
      }
    }
  }
  consumers_sync();
  if (!*s_abort) {
    for (int o = warp; o < nrow * T; o += kConsumerWarps) {
      const int nl = o / T, t = o - nl * T;
      float sum = 0.f;
      for (int p = lane; p < G; p += 32) sum += stage[((size_t)p * nrow + nl) * TP + t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
      if (lane == 0) out[(size_t)t * H + nb0 + nl] = f32_to_bf16_rne(sum);
    }
  }
  consumers_sync();
}

// Bytes of shared memory the exchange stages: G x ceil(H / G) x TP floats.
inline size_t collect_stage_bytes(int G, int H, int T) {
  return (size_t)G * ((size_t)(H + G - 1) / G) * (size_t)(T + (T & 1)) * 4;
}

}  // namespace stream
}  // namespace moe
