// Record-streaming decode kernel of the MoE layer for bf16 routed experts and
// small token windows (T <= MOE_DECODE_MAX_T).
//
// "Optimizing on-device inference for Apple Silicon", section "Decode: reduce
// bytes moved per token": at batch 1 the layer's time is the time to read its
// weight bytes once, so the kernel's job is to keep HBM busy from the first
// cycle to the last. Section "Reduce intermediate and state traffic": the
// gated gate/up projection and the down projection with its routing weight and
// the shared-expert result are one pass. Section "Overlap independent work":
// the shared expert does not depend on routing, so its weights are on their way
// while the router runs. "Three ways to speed up MoE inference on DGX Spark",
// section "Optimization 3": a verify window reads each distinct expert once for
// every token that chose it.
//
// Weight layout: one record per (expert, intermediate feature i), contiguous:
//   [ gate row i (H bf16) | up row i (H bf16) | down column i (H bf16) ]
// so that feature i's SwiGLU output h_i = silu(gate_i . x) * (up_i . x) and its
// whole contribution w * h_i * down[:, i] to the output come from one 6H-byte
// stream. Summing those contributions over the features a CTA owns gives a
// partial output vector per CTA; one grid-wide exchange adds the partials.
//
// One cooperative launch, one CTA per SM, 16 consumer warps + 1 producer warp:
//   producer   bulk-copies x, then this CTA's shared-expert records, then (once
//              routing is known) its routed records, group by group, into a
//              ring of slot groups in shared memory (full/empty mbarriers).
//   router     each CTA computes its 1-4 fp32 router logits and publishes each
//              as a 64-bit word {call tag, value}; readers poll until every
//              word carries the current call's tag (no separate barrier).
//   top-k      every CTA derives the routing from the published logits
//              (identical inputs and arithmetic on every CTA).
//   groups     4 records per group; 4 warps per record compute the gate/up dot
//              products over a quarter of H each; then every thread adds
//              w * h * down[n] for its own 4-output slices.
//   exchange   partial outputs [T][H] fp32 per CTA -> global; one bounded grid
//              barrier; each CTA sums its slice of outputs over all CTAs in a
//              fixed order (deterministic) and writes bf16.
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_sm100.cuh"

namespace moe {

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kStreamThreads = kConsumers + 32;     // + one producer warp
constexpr int kWarpsPerRecord = 4;
constexpr int kGroupRecords = kConsumerWarps / kWarpsPerRecord;   // records per ring group
constexpr int kMaxRingGroups = 16;
constexpr int kMaxRouterRows = 16;                  // router rows per CTA
constexpr int kStreamSmemMax = 220 * 1024;          // dynamic shared memory budget
constexpr int kMaxStreamH = 4096;
constexpr long long kSpinBudget = 4000000000LL;     // ~2 s of SM cycles: then give up

struct StreamArgs {
  const uint16_t* x;           // bf16 [T][H]
  int T, H, E, k, I, Is;
  const float* router_t;       // fp32 [E][H]
  const float* router_bias;    // fp32 [E]
  const float* logit_bias;     // fp32 [T][E] or nullptr
  const uint8_t* rec;          // routed records [E][I][3][H] bf16
  const uint8_t* rec_sh;       // shared-expert records [Is][3][H] bf16
  int rec_bytes;               // 6 * H
  int ring_groups;             // slot groups in the ring
  int x_bytes_al;              // bytes of the x region (128-aligned)
  unsigned long long* words;   // [kMaxDecodeT][E] tagged logits
  float* partial;              // [G][T][H] per-CTA partial outputs
  unsigned long long* ctr;     // monotonic arrival counter of the final exchange
  int* idx;                    // [T][k]  diagnostics (CTA 0)
  float* weights;              // [T][k]
  DecodeMeta* meta;
  uint16_t* out;               // bf16 [T][H]
  int* err;
  const int* never_set;
  int force_timeout;
};

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
MOE_DEV unsigned long long ld_acquire_u64_g(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
MOE_DEV void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
// Barrier among the 16 consumer warps only (the producer warp never joins it).
MOE_DEV void consumers_sync() { asm volatile("bar.sync 1, %0;" :: "n"(kConsumers) : "memory"); }

// Record range of this CTA. Shared-expert records [sh0, sh1) are known before
// routing; routed records [u0, u1) index the window's D x I (slot, feature)
// pairs. When there are at least G routed pairs the two ranges are balanced
// jointly (a CTA with one more shared record gets one fewer routed record).
// All counts fit 32 bits (U <= 64 slots x 4096 features, G < 1024), and the
// kernel uses unsigned 32-bit division only: 64-bit division is a long
// software sequence that would sit on the producer's critical path.
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

template <int TMAX>
__global__ void __launch_bounds__(kStreamThreads, 1) moe_decode_stream_kernel(const StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);   // x [T][H] bf16
  uint8_t* ring = smem + a.x_bytes_al;                // ring_groups x kGroupRecords records

  __shared__ __align__(8) uint64_t full_bar[kMaxRingGroups];
  __shared__ __align__(8) uint64_t empty_bar[kMaxRingGroups];
  __shared__ __align__(8) uint64_t x_bar;
  __shared__ float s_rpart[kConsumerWarps][TMAX];                    // router partial sums
  __shared__ float s_gu[kGroupRecords][kWarpsPerRecord][TMAX][2];    // gate/up partial dots
  __shared__ float s_c[kGroupRecords][TMAX];                         // w * h per record, token
  __shared__ int s_idx[kMaxDecodeT * kMaxTopK];
  __shared__ float s_w[kMaxDecodeT * kMaxTopK];
  __shared__ int s_slot_of[kMaxDecodeT * kMaxTopK];
  __shared__ unsigned s_tmask[kMaxSlots];
  __shared__ DecodeMeta s_meta;
  __shared__ unsigned long long s_tag;
  __shared__ int s_abort;

  const int T = a.T, H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int NG = a.ring_groups;
  const int rec_bytes = a.rec_bytes;
  const bool producer = (warp == kConsumerWarps);

  if (threadIdx.x == 0) {
    for (int g = 0; g < NG; ++g) {
      sm100::mbar_init(&full_bar[g], 1);
      sm100::mbar_init(&empty_bar[g], kConsumerWarps);
    }
    sm100::mbar_init(&x_bar, 1);
    sm100::fence_barrier_init();
    s_abort = 0;
    // Calls completed so far = arrivals at the final exchange / G; no CTA of
    // this call arrives there before every CTA has published its logits, which
    // each does after reading this value.
    s_tag = ld_relaxed_u64(a.ctr) / (unsigned long long)G + 1ull;
  }
  __syncthreads();
  const unsigned long long tag = s_tag;

  const Ranges rg0 = cta_ranges(b, G, Is, 0);   // shared range does not depend on routing
  const int ns = rg0.sh1 - rg0.sh0;
  const int nsg = (ns + kGroupRecords - 1) / kGroupRecords;    // shared groups

  // ---------------------------------------------------------------- producer: x + shared records
  // Whole producer warp: lane 0 posts the group's byte count, then lane r
  // copies record r of the group.
  auto issue_group = [&](int grp, int u0, int nr) {
    const int sg = grp % NG;
    int first, n;
    if (grp < nsg) {
      first = grp * kGroupRecords;
      n = min(kGroupRecords, ns - first);
    } else {
      first = (grp - nsg) * kGroupRecords;
      n = min(kGroupRecords, nr - first);
    }
    if (lane == 0) sm100::mbar_arrive_expect_tx(&full_bar[sg], (uint32_t)(n * rec_bytes));
    __syncwarp();
    if (lane < n) {
      const uint8_t* src;
      if (grp < nsg) {
        src = a.rec_sh + (size_t)(rg0.sh0 + first + lane) * rec_bytes;
      } else {
        const unsigned u = (unsigned)(u0 + first + lane);
        const unsigned d = u / (unsigned)I, i = u - d * (unsigned)I;
        src = a.rec + ((size_t)s_meta.slot_expert[d] * I + i) * rec_bytes;
      }
      sm100::bulk_copy_g2s(ring + ((size_t)sg * kGroupRecords + lane) * rec_bytes, src, (uint32_t)rec_bytes,
                           &full_bar[sg]);
    }
  };
  int issued = 0;   // groups issued (producer warp)
  if (producer) {
    if (lane == 0) {
      const uint32_t xbytes = (uint32_t)(T * H * 2);
      sm100::mbar_arrive_expect_tx(&x_bar, xbytes);
      for (uint32_t off = 0; off < xbytes; off += 32768u)
        sm100::bulk_copy_g2s(reinterpret_cast<uint8_t*>(xs) + off, reinterpret_cast<const uint8_t*>(a.x) + off,
                             min(32768u, xbytes - off), &x_bar);
    }
    for (; issued < nsg && issued < NG; ++issued) issue_group(issued, 0, 0);
  }

  // ---------------------------------------------------------------- consumers: router logits
  const int nr_rows = (E - b + G - 1) / G;   // router rows b, b + G, ... (<= kMaxRouterRows)
  if (!producer) {
    const int P = max(1, kConsumerWarps / max(nr_rows, 1));     // warps per row
    const int items = nr_rows * P;
    const int H4 = H / 4;
    if (threadIdx.x == 0 && a.force_timeout && b == 0 && !bounded_wait_flag(a.never_set, 2000000LL))
      set_error(a.err, kDevTimeout);
    if (warp < items) {
      const int m = warp / P, p = warp - m * P;
      const int e = b + m * G;
      const float* row = a.router_t + (size_t)e * H;
      const int c0 = p * H4 / P, c1 = (p + 1) * H4 / P;
      float acc[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
      bool x_ready = false;
      for (int cb = c0; cb < c1; cb += 32 * 8) {
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int c = cb + lane + 32 * q;
          if (c < c1) v[q] = ldg_stream(row + 4 * c);
        }
        if (!x_ready) {
          volatile int never = 0;
          if (!sm100::mbar_wait(&x_bar, 0, a.err, &never, kSpinBudget, false)) s_abort = 1;
          x_ready = true;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int c = cb + lane + 32 * q;
          if (c < c1) {
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
              if (t < T) {
                const uint2 xx = *reinterpret_cast<const uint2*>(xs + t * H + 4 * c);
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
      if (!x_ready) {
        volatile int never = 0;
        if (!sm100::mbar_wait(&x_bar, 0, a.err, &never, kSpinBudget, false)) s_abort = 1;
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const float sum = warp_sum(acc[t]);
          if (lane == 0) s_rpart[warp][t] = sum;
        }
      }
    } else {
      volatile int never = 0;   // x is needed later by every warp
      if (!sm100::mbar_wait(&x_bar, 0, a.err, &never, kSpinBudget, false)) s_abort = 1;
    }
    consumers_sync();
    if ((int)threadIdx.x < nr_rows * T) {   // logit = partial sums in warp order + biases
      const int m = threadIdx.x / T, t = threadIdx.x - m * T;
      const int e = b + m * G;
      float sl = 0.f;
      for (int p = 0; p < P; ++p) sl += s_rpart[m * P + p][t];
      sl += a.router_bias[e];
      if (a.logit_bias) sl += a.logit_bias[(size_t)t * E + e];
      st_relaxed_u64(a.words + (size_t)t * E + e, (tag << 32) | (unsigned long long)__float_as_uint(sl));
    }

    // ------------------------------------------------------------ top-k of every token, in every CTA
    if (warp < T) {
      const int t = warp;
      bool ok;
      if (E <= 256) ok = poll_topk<1>(a.words + (size_t)t * E, E, k, tag, lane, s_idx + t * k, s_w + t * k);
      else ok = poll_topk<2>(a.words + (size_t)t * E, E, k, tag, lane, s_idx + t * k, s_w + t * k);
      if (!ok) {
        if (lane == 0) set_error(a.err, kDevTimeout);
        s_abort = 1;
      }
    }
    consumers_sync();
    // distinct experts of the window in first-appearance order (slots), and
    // for each slot the position j of its expert in each token's top-k
    if (warp == 0) {
      const int n = T * k;
      bool first[2] = {false, false};
      int firstpos[2] = {0, 0};
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int ai = lane + 32 * h2;
        if (ai < n) {
          const int e = s_idx[ai];
          if (e < 0 || e >= E) {   // only NaN logits can get here
            set_error(a.err, kDevCheck);
            s_abort = 1;
          }
          int q = 0;
          while (s_idx[q] != e) ++q;
          first[h2] = (q == ai);
          firstpos[h2] = q;
        }
      }
      const unsigned m0 = __ballot_sync(0xFFFFFFFFu, first[0]);
      const unsigned m1 = __ballot_sync(0xFFFFFFFFu, first[1]);
      const unsigned lt = (1u << lane) - 1u;
      if (first[0]) s_slot_of[lane] = __popc(m0 & lt);
      if (first[1]) s_slot_of[lane + 32] = __popc(m0) + __popc(m1 & lt);
      __syncwarp();
      const int D = __popc(m0) + __popc(m1);
      for (int q = lane; q < D * kMaxDecodeT; q += 32) s_meta.slot_j[q / kMaxDecodeT][q % kMaxDecodeT] = -1;
      for (int q = lane; q < D; q += 32) s_tmask[q] = 0u;
      __syncwarp();
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int ai = lane + 32 * h2;
        if (ai < n) {
          const int slot = s_slot_of[firstpos[h2]];
          if (first[h2]) s_meta.slot_expert[slot] = s_idx[ai];
          s_meta.slot_j[slot][ai / k] = (signed char)(ai % k);
          atomicOr(&s_tmask[slot], 1u << (ai / k));
        }
      }
      if (lane == 0) s_meta.num_slots = D;
    }
  }
  __syncthreads();   // routing known to every warp, producer included
  if (s_abort) {
    // nothing routed was issued; let x and the shared-expert copies land first
    if (threadIdx.x == 0) {
      volatile int never = 0;
      sm100::mbar_wait(&x_bar, 0, a.err, &never, 20000000LL, false);
      for (int g2 = 0; g2 < nsg && g2 < NG; ++g2)
        sm100::mbar_wait(&full_bar[g2], 0, a.err, &never, 20000000LL, false);
    }
    return;
  }

  const int D = s_meta.num_slots;
  const int U = D * I;
  const Ranges rg = cta_ranges(b, G, Is, U);
  const int nr = (int)(rg.u1 - rg.u0);
  const int ngroups = nsg + (nr + kGroupRecords - 1) / kGroupRecords;

  if (b == 0 && !producer) {   // diagnostics copy of the routing
    for (int q = threadIdx.x; q < T * k; q += kConsumers) {
      a.idx[q] = s_idx[q];
      a.weights[q] = s_w[q];
    }
    const int* src = reinterpret_cast<const int*>(&s_meta);
    int* dst = reinterpret_cast<int*>(a.meta);
    for (int q = threadIdx.x; q < (int)(sizeof(DecodeMeta) / 4); q += kConsumers) dst[q] = src[q];
  }

  // ---------------------------------------------------------------- producer: routed records
  if (producer) {
    for (; issued < ngroups; ++issued) {
      bool go = !s_abort;
      if (go && issued >= NG && lane == 0) {
        const int sg = issued % NG;
        const uint32_t par = (uint32_t)((issued / NG) - 1) & 1u;
        go = sm100::mbar_wait(&empty_bar[sg], par, a.err, &s_abort, kSpinBudget);
      }
      if (!__shfl_sync(0xFFFFFFFFu, go, 0)) break;
      issue_group(issued, rg.u0, nr);
    }
    return;   // the consumers outlive every copy issued here (they wait for each)
  }

  // ---------------------------------------------------------------- consumers: groups
  constexpr int NCH = kMaxStreamH / 4 / kConsumers;   // 4-output chunks per thread (2)
  float acc[NCH][TMAX][4];
#pragma unroll
  for (int ci = 0; ci < NCH; ++ci)
#pragma unroll
    for (int t = 0; t < TMAX; ++t)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[ci][t][j] = 0.f;

  const int H8 = H / 8, H4 = H / 4;
  const int rr = warp / kWarpsPerRecord, qq = warp % kWarpsPerRecord;
  const int cq0 = qq * H8 / kWarpsPerRecord, cq1 = (qq + 1) * H8 / kWarpsPerRecord;
  int grp = 0;
  for (; grp < ngroups; ++grp) {
    const int sg = grp % NG;
    const bool shared = grp < nsg;
    const int first = shared ? grp * kGroupRecords : (grp - nsg) * kGroupRecords;
    const int nvalid = min(kGroupRecords, (shared ? ns : nr) - first);
    const uint8_t* gbase = ring + (size_t)sg * kGroupRecords * rec_bytes;
    if (!sm100::mbar_wait(&full_bar[sg], (uint32_t)(grp / NG) & 1u, a.err, &s_abort, kSpinBudget)) {
      // fall through to the barrier; every warp sees s_abort there
    }
    // gate/up dot products: warp (rr, qq) covers 16-byte chunks [cq0, cq1) of record rr
    unsigned tmask = 0u;
    if (rr < nvalid) {
      tmask = shared ? (1u << T) - 1u : s_tmask[(unsigned)(rg.u0 + first + rr) / (unsigned)I];
      const uint8_t* rec = gbase + (size_t)rr * rec_bytes;
      float ag[TMAX], au[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) ag[t] = au[t] = 0.f;
      for (int c = cq0 + lane; c < cq1; c += 32) {
        const uint4 gv = *reinterpret_cast<const uint4*>(rec + 16 * c);
        const uint4 uv = *reinterpret_cast<const uint4*>(rec + 2 * H + 16 * c);
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t < T && ((tmask >> t) & 1u)) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * H + 8 * c);
            ag[t] = fma8_bf16(gv, xv, ag[t]);
            au[t] = fma8_bf16(uv, xv, au[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T && ((tmask >> t) & 1u)) {
          const float gs = warp_sum(ag[t]);
          const float us = warp_sum(au[t]);
          if (lane == 0) {
            s_gu[rr][qq][t][0] = gs;
            s_gu[rr][qq][t][1] = us;
          }
        }
      }
    }
    consumers_sync();
    if ((int)threadIdx.x < kGroupRecords * TMAX) {   // c = w * silu(g) * u per (record, token)
      const int r = threadIdx.x / TMAX, t = threadIdx.x - r * TMAX;
      float c = 0.f;
      if (r < nvalid && t < T) {
        int j = -1;
        float w = 1.f;
        if (!shared) {
          const int d = (int)((unsigned)(rg.u0 + first + r) / (unsigned)I);
          j = s_meta.slot_j[d][t];
          if (j >= 0) w = s_w[t * k + j];
        }
        if (shared || j >= 0) {
          float g = 0.f, u = 0.f;
#pragma unroll
          for (int q = 0; q < kWarpsPerRecord; ++q) {
            g += s_gu[r][q][t][0];
            u += s_gu[r][q][t][1];
          }
          c = w * swiglu(g, u);
        }
      }
      s_c[r][t] = c;
    }
    consumers_sync();
    if (s_abort) break;
    // down columns: out[t][n] += c[r][t] * down_r[n] for this thread's 4-output chunks
#pragma unroll
    for (int ci = 0; ci < NCH; ++ci) {
      const int ch = threadIdx.x + ci * kConsumers;
      if (ch < H4) {
        for (int r = 0; r < nvalid; ++r) {
          const uint2 dv = *reinterpret_cast<const uint2*>(gbase + (size_t)r * rec_bytes + 4 * H + 8 * ch);
          const float d0 = bf16_lo(dv.x), d1 = bf16_hi(dv.x), d2 = bf16_lo(dv.y), d3 = bf16_hi(dv.y);
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            const float c = (t < T) ? s_c[r][t] : 0.f;
            if (c != 0.f) {
              acc[ci][t][0] = fmaf(c, d0, acc[ci][t][0]);
              acc[ci][t][1] = fmaf(c, d1, acc[ci][t][1]);
              acc[ci][t][2] = fmaf(c, d2, acc[ci][t][2]);
              acc[ci][t][3] = fmaf(c, d3, acc[ci][t][3]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) sm100::mbar_arrive(&empty_bar[sg]);
  }
  if (s_abort) {
    // let copies still in flight land before the CTA's shared memory goes away
    if (threadIdx.x == 0) {
      volatile int never = 0;
      for (int g2 = grp; g2 < ngroups && g2 < grp + NG; ++g2)
        sm100::mbar_wait(&full_bar[g2 % NG], (uint32_t)(g2 / NG) & 1u, a.err, &never, 20000000LL, false);
    }
    return;
  }

  // ---------------------------------------------------------------- exchange of partial outputs
#pragma unroll
  for (int ci = 0; ci < NCH; ++ci) {
    const int ch = threadIdx.x + ci * kConsumers;
    if (ch < H4) {
#pragma unroll
      for (int t = 0; t < TMAX; ++t)
        if (t < T)
          *reinterpret_cast<float4*>(a.partial + ((size_t)b * T + t) * H + 4 * ch) =
              make_float4(acc[ci][t][0], acc[ci][t][1], acc[ci][t][2], acc[ci][t][3]);
    }
  }
  consumers_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.ctr, 1ull);
    const unsigned long long target = tag * (unsigned long long)G;
    const long long t0 = clock64();
    while (ld_acquire_u64_g(a.ctr) < target) {
      if (clock64() - t0 > kSpinBudget) {
        set_error(a.err, kDevTimeout);
        s_abort = 1;
        break;
      }
    }
  }
  consumers_sync();
  if (s_abort) return;
  // This CTA's outputs: 4-output chunks [c0, c1) of the T x H/4 chunks. Every
  // (chunk, CTA partial) float4 is loaded at once into shared memory (the ring
  // is free now), then one warp per chunk adds the G partials in a fixed order.
  const int NC = T * H4;
  const int c0 = (int)((unsigned)b * (unsigned)NC / (unsigned)G);
  const int c1 = (int)((unsigned)(b + 1) * (unsigned)NC / (unsigned)G);
  const int npairs = (c1 - c0) * G;
  float4* stage = reinterpret_cast<float4*>(ring);   // [c1 - c0][G]
  for (int q0 = threadIdx.x; q0 < npairs; q0 += 8 * kConsumers) {
    uint4 v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int q = q0 + r * kConsumers;
      if (q < npairs) {
        const int cc = q / G, p = q - cc * G;
        const int cidx = c0 + cc;
        const int t = cidx / H4, ch = cidx - t * H4;
        v[r] = ldg_cg(a.partial + ((size_t)p * T + t) * H + 4 * ch);
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int q = q0 + r * kConsumers;
      if (q < npairs) stage[q] = make_float4(__uint_as_float(v[r].x), __uint_as_float(v[r].y),
                                             __uint_as_float(v[r].z), __uint_as_float(v[r].w));
    }
  }
  consumers_sync();
  for (int cc = warp; cc < c1 - c0; cc += kConsumerWarps) {
    float4 sacc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = lane; p < G; p += 32) {
      const float4 v = stage[cc * G + p];
      sacc.x += v.x; sacc.y += v.y; sacc.z += v.z; sacc.w += v.w;
    }
    for (int o = 16; o > 0; o >>= 1) {
      sacc.x += __shfl_xor_sync(0xFFFFFFFFu, sacc.x, o);
      sacc.y += __shfl_xor_sync(0xFFFFFFFFu, sacc.y, o);
      sacc.z += __shfl_xor_sync(0xFFFFFFFFu, sacc.z, o);
      sacc.w += __shfl_xor_sync(0xFFFFFFFFu, sacc.w, o);
    }
    if (lane == 0) {
      const int cidx = c0 + cc;
      const int t = cidx / H4, ch = cidx - t * H4;
      uint2 o2;
      o2.x = (uint32_t)f32_to_bf16_rne(sacc.x) | ((uint32_t)f32_to_bf16_rne(sacc.y) << 16);
      o2.y = (uint32_t)f32_to_bf16_rne(sacc.z) | ((uint32_t)f32_to_bf16_rne(sacc.w) << 16);
      *reinterpret_cast<uint2*>(a.out + (size_t)t * H + 4 * ch) = o2;
    }
  }
}

}  // namespace

// ===========================================================================
// Host side
// ===========================================================================
static int stream_ring_groups(const moe_layer* L, int T) {
  const int H = L->cfg.hidden;
  const size_t xb = ((size_t)T * H * 2 + 127) / 128 * 128;
  const size_t gb = (size_t)kGroupRecords * 6 * H;
  if (xb >= (size_t)kStreamSmemMax) return 0;
  return (int)std::min<size_t>((kStreamSmemMax - xb) / gb, kMaxRingGroups);
}

bool stream_supported(const moe_layer* L, int T) {
  const auto& c = L->cfg;
  if (c.weight_format != MOE_WEIGHTS_BF16 || !L->w_rec) return false;
  if (c.hidden > kMaxStreamH || T < 1 || T > kMaxDecodeT) return false;
  if ((c.num_experts + L->num_sms - 1) / L->num_sms > kMaxRouterRows) return false;
  const int ng = stream_ring_groups(L, T);
  if (ng < 2) return false;
  // the final exchange stages this CTA's (chunk, partial) pairs in the ring
  const size_t chunks = ((size_t)T * c.hidden / 4 + L->num_sms - 1) / L->num_sms;
  return chunks * L->num_sms * 16 <= (size_t)ng * kGroupRecords * 6 * c.hidden;
}

template <int TMAX>
static cudaError_t launch_stream_t(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb,
                                   cudaStream_t s) {
  const auto& c = L->cfg;
  StreamArgs a;
  a.x = x; a.T = T; a.H = c.hidden; a.E = c.num_experts; a.k = c.top_k; a.I = c.intermediate;
  a.Is = c.shared_intermediate;
  a.router_t = L->router_t; a.router_bias = L->router_bias; a.logit_bias = lb;
  a.rec = L->w_rec; a.rec_sh = L->ws_rec; a.rec_bytes = 6 * c.hidden;
  a.ring_groups = stream_ring_groups(L, T);
  a.x_bytes_al = (int)(((size_t)T * c.hidden * 2 + 127) / 128 * 128);
  a.words = L->dec.logit_words; a.partial = L->dec.partial; a.ctr = L->dec.sync_ctr + 2;
  a.idx = L->dec.idx; a.weights = L->dec.weights; a.meta = L->dec.meta;
  a.out = out; a.err = L->err; a.never_set = L->never_set;
  a.force_timeout = (c.flags & MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT) ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L->num_sms);
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = (size_t)a.x_bytes_al + (size_t)a.ring_groups * kGroupRecords * a.rec_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs co-resident: they wait on one another
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(L, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_decode_stream_kernel<TMAX>, a);
  prof_mark(L, s);
  return e;
}

cudaError_t stream_prepare(moe_layer* L) {
  (void)L;
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* f) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmemMax);
  };
  set((const void*)moe_decode_stream_kernel<1>);
  set((const void*)moe_decode_stream_kernel<2>);
  set((const void*)moe_decode_stream_kernel<4>);
  set((const void*)moe_decode_stream_kernel<8>);
  return e;
}

cudaError_t launch_stream(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb, cudaStream_t s) {
  if (T <= 1) return launch_stream_t<1>(L, x, out, T, lb, s);
  if (T <= 2) return launch_stream_t<2>(L, x, out, T, lb, s);
  if (T <= 4) return launch_stream_t<4>(L, x, out, T, lb, s);
  return launch_stream_t<8>(L, x, out, T, lb, s);
}

}  // namespace moe
