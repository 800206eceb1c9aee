// Record-streaming decode kernel of the MoE layer for MXFP4 routed experts
// (T <= MOE_DECODE_MAX_T): the same structure as the bf16 kernel in
// moe_stream.cu -- a producer warp bulk-copies per-feature records of the
// selected experts into a shared-memory ring, 16 consumer warps turn each
// record into its contribution to the output, one tagged exchange adds the
// CTAs' partial outputs -- with the expert weights decoded inside the dot
// products.
//
// "Three ways to speed up MoE inference on DGX Spark", section "Optimization
// 1": the routed experts are MXFP4 (e2m1 codes, one e8m0 scale per 32
// elements) and the decode path reads them in that form, a quarter of the
// bf16 bytes. "Optimizing on-device inference for Apple Silicon", section
// "Decode weights during matrix multiplication": the codes are decoded in
// registers as they are multiplied, never written back in a wider format.
//
// Records (repacked at create), per (expert e, intermediate feature i):
//   [ gate codes (H/2 B) | gate scales (H/32 B, padded to 16) |
//     up codes | up scales | down column codes (H/2 B) ] + 16 B padding
// Code byte j of a row holds elements 2j (low nibble) and 2j+1 (high); a scale
// covers 32 consecutive elements of its row. The down column of feature i
// holds W_down[e][n][i] for n = 0..H-1, two per byte (even n low). Its scales
// belong to (n, i / 32), i.e. to 32 consecutive features at once, so they are
// kept apart, one H-byte vector per (e, block of 32 features), and each ring
// group carries the one or two vectors its records need.
// The shared expert stays bf16 and uses the bf16 kernel's record format.
//
// Consumers (CUDA cores; per record the work is ~3H multiply-adds per token,
// far below what the copies deliver per SM, so no tensor-core tiling):
//   gate/up    16 / R warps per record of an R-record group, each over a slice
//              of H: codes -> f16 pairs (cvt.rn.f16x2.e2m1x2), multiplied with
//              an f16 copy of x (fma.rn.f32.f16: f16 products, fp32 sums), each
//              8-element word scaled by its block scale; warp sums to shared
//              memory, slices added in order, c = w * silu(g) * u per token.
//   down       thread q owns outputs n = 8q .. 8q+7 for every token and adds
//              c * code * scale over the group's records in record order.
// Readings: x is rounded to f16 for the MXFP4 products (exact for the normal
// f16 range |x| in [2^-14, 65504]; smaller values lose bits, larger overflow),
// the e2m1 values are exact in f16, and every sum is fp32.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_sm100.cuh"
#include "moe_stream_common.cuh"

namespace moe {

namespace {

using stream::consumers_sync;
using stream::cta_ranges;
using stream::kConsumers;
using stream::kConsumerWarps;
using stream::kMaxRingGroups;
using stream::kSpinBudget;
using stream::Ranges;
using stream::tagged;

constexpr int kMaxMx = 16;             // MXFP4 records per routed group: 16 (one warp each), or 8
                                       // (two warps each) when x leaves no room for two 16-record slots
constexpr int kShGroup = 2;            // bf16 shared-expert records per shared group (8 warps each)
constexpr int kMxMaxH = 4096;          // one 8-output chunk per consumer thread
constexpr int kParts = 8;              // most warps on one record (shared groups)

struct MxArgs {
  const uint16_t* x;           // bf16 [T][H]
  int T, H, E, k, I, Is;
  const float* router_t;       // fp32 [E][H]
  const float* router_bias;    // fp32 [E]
  const float* logit_bias;     // fp32 [T][E] or nullptr
  const uint8_t* rec;          // routed MXFP4 records [E][I] x mx_stride bytes
  const uint8_t* dsc;          // down scales [E][I / 32][H] bytes
  const uint8_t* rec_sh;       // shared-expert bf16 records [Is] x sh_stride bytes
  int mx_stride, sh_stride;    // bytes per record
  int sc_off;                  // padded bytes of one scale segment (pad16(H / 32))
  int mx_group;                // MXFP4 records per routed group (16 or 8)
  int slot_bytes;              // bytes of one ring slot group
  int ring_groups;             // slot groups in the ring
  int x_bytes_al;              // bytes of one x copy (T rows of H + 8 halves, 128-aligned)
  unsigned long long* words;   // [kMaxDecodeT][E] tagged logits
  unsigned long long* partial; // [G][H][TP] tagged partial outputs
  unsigned long long* ctr;     // calls completed x G (each CTA adds 1 when it leaves)
  int* idx;                    // [T][k]  diagnostics (CTA 0)
  float* weights;              // [T][k]
  DecodeMeta* meta;
  uint16_t* out;               // bf16 [T][H]
  int* err;
  const int* never_set;
  int force_timeout;
};

// Record offsets (bytes) of an MXFP4 record with scale segments of `so` bytes.
// (gate codes start at byte 0)
MOE_DEV int mx_gate_scales(int H) { return H / 2; }
MOE_DEV int mx_up_codes(int H, int so) { return H / 2 + so; }
MOE_DEV int mx_up_scales(int H, int so) { return H + so; }
MOE_DEV int mx_down_codes(int H, int so) { return H + 2 * so; }

// Unscaled dot of 8 e2m1 codes (one 32-bit word, element order) with 8 f16 of x.
MOE_DEV float dot8_e2m1(uint32_t codes, const uint4 xv) {
  float s = fma2_f16(e2m1x2_to_f16x2(codes & 0xFFu), xv.x, 0.f);
  s = fma2_f16(e2m1x2_to_f16x2((codes >> 8) & 0xFFu), xv.y, s);
  s = fma2_f16(e2m1x2_to_f16x2((codes >> 16) & 0xFFu), xv.z, s);
  return fma2_f16(e2m1x2_to_f16x2(codes >> 24), xv.w, s);
}

template <int TMAX>
__global__ void __launch_bounds__(stream::kThreads, 1) moe_decode_stream_mx_kernel(const MxArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                 // x [T][H + 8] bf16
  uint16_t* x16 = reinterpret_cast<uint16_t*>(smem + a.x_bytes_al); // x [T][H + 8] f16
  uint8_t* ring = smem + 2 * a.x_bytes_al;                          // ring_groups x slot_bytes

  __shared__ __align__(8) uint64_t full_bar[kMaxRingGroups];
  __shared__ __align__(8) uint64_t empty_bar[kMaxRingGroups];
  __shared__ __align__(8) uint64_t x_bar;
  __shared__ float s_rpart[kConsumerWarps][TMAX];                   // router partial sums
  __shared__ float s_gu[kMaxMx][kParts][TMAX][2];                   // gate/up slice sums
  // w * silu(g) * u per record and token, double-buffered by group parity: with
  // one warp per record a warp writes group k+1's values while others still
  // read group k's; group k+2 is written only after the barrier of group k+1.
  __shared__ float s_cb[2][kMaxMx][TMAX];
  __shared__ stream::RouteSmem rs;
  __shared__ unsigned long long s_tag;
  __shared__ int s_abort;

  const int T = a.T, H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
  const int XP = H + 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int NG = a.ring_groups;
  const int so = a.sc_off;
  const int mxs = a.mx_stride, shs = a.sh_stride;
  const int RGM = a.mx_group;
  const int sv_off = RGM * mxs;                      // scale vectors of a routed group, in its slot
  const int nblk = I / 32;
  const bool producer = (warp == kConsumerWarps);

  if (threadIdx.x == 0) {
    for (int g = 0; g < NG; ++g) {
      sm100::mbar_init(&full_bar[g], 1);
      sm100::mbar_init(&empty_bar[g], kConsumerWarps);
    }
    sm100::mbar_init(&x_bar, 1);
    sm100::fence_barrier_init();
    s_abort = 0;
    s_tag = stream::ld_relaxed_u64(a.ctr) / (unsigned long long)G + 1ull;   // see moe_stream_common.cuh
  }
  __syncthreads();
  const unsigned long long tag = s_tag;
  auto leave = [&]() { atomicAdd(a.ctr, 1ull); };   // once per CTA, on every exit path

  const Ranges rg0 = cta_ranges(b, G, Is, 0);
  const int ns = rg0.sh1 - rg0.sh0;
  const int nsg = (ns + kShGroup - 1) / kShGroup;   // shared (bf16) groups come first

  // (slot, block) of routed unit u: which down-scale vector it needs
  auto unit_blk = [&](int u, int& d, int& blk) {
    d = (int)((unsigned)u / (unsigned)I);
    blk = (u - d * I) / 32;
  };
  // Whole producer warp: lane 0 posts the group's byte count and issues its copies.
  auto issue_group = [&](int grp, int u0, int nr) {
    const int sg = grp % NG;
    uint8_t* base = ring + (size_t)sg * a.slot_bytes;
    if (lane == 0) {
      if (grp < nsg) {
        const int first = grp * kShGroup, n = min(kShGroup, ns - first);
        sm100::mbar_arrive_expect_tx(&full_bar[sg], (uint32_t)(n * shs));
        sm100::bulk_copy_g2s(base, a.rec_sh + (size_t)(rg0.sh0 + first) * shs, (uint32_t)(n * shs), &full_bar[sg]);
      } else {
        const int first = (grp - nsg) * RGM, n = min(RGM, nr - first);
        int d0, b0, dl, bl;
        unit_blk(u0 + first, d0, b0);
        unit_blk(u0 + first + n - 1, dl, bl);
        const bool two = (dl != d0 || bl != b0);
        sm100::mbar_arrive_expect_tx(&full_bar[sg], (uint32_t)(n * mxs + (two ? 2 : 1) * H));
        uint8_t* dst = base;
        unsigned u = (unsigned)(u0 + first);
        int left = n;
        while (left > 0) {
          const unsigned d = u / (unsigned)I, i = u - d * (unsigned)I;
          const int run = min(left, I - (int)i);
          sm100::bulk_copy_g2s(dst, a.rec + ((size_t)rs.meta.slot_expert[d] * I + i) * mxs, (uint32_t)(run * mxs),
                               &full_bar[sg]);
          dst += (size_t)run * mxs;
          u += run;
          left -= run;
        }
        sm100::bulk_copy_g2s(base + sv_off, a.dsc + ((size_t)rs.meta.slot_expert[d0] * nblk + b0) * H, (uint32_t)H,
                             &full_bar[sg]);
        if (two)
          sm100::bulk_copy_g2s(base + sv_off + H, a.dsc + ((size_t)rs.meta.slot_expert[dl] * nblk + bl) * H,
                               (uint32_t)H, &full_bar[sg]);
      }
    }
    __syncwarp();
  };
  int issued = 0;
  if (producer) {
    if (lane == 0) {
      sm100::mbar_arrive_expect_tx(&x_bar, (uint32_t)(T * H * 2));
      for (int t = 0; t < T; ++t)
        sm100::bulk_copy_g2s(xs + (size_t)t * XP, a.x + (size_t)t * H, (uint32_t)(H * 2), &x_bar);
      volatile int never = 0;   // shared records only after x (see moe_stream.cu)
      sm100::mbar_wait(&x_bar, 0, a.err, &never, kSpinBudget, false);
    }
    __syncwarp();
    for (; issued < nsg && issued < NG; ++issued) issue_group(issued, 0, 0);
  }

  // ---------------------------------------------------------------- consumers: router, f16 copy of x, routing
  if (!producer) {
    if (threadIdx.x == 0 && a.force_timeout && b == 0 && !bounded_wait_flag(a.never_set, 2000000LL))
      set_error(a.err, kDevTimeout);
    stream::router_publish<TMAX>(xs, XP, T, H, E, a.router_t, a.router_bias, a.logit_bias, a.words, tag, &x_bar,
                                 a.err, &s_abort, s_rpart);
    for (int q = threadIdx.x; q < T * H / 2; q += kConsumers) {   // bf16 pairs -> f16 pairs
      const int t = q / (H / 2), c = q - t * (H / 2);
      const uint32_t v = *reinterpret_cast<const uint32_t*>(xs + t * XP + 2 * c);
      const __half2 h = __floats2half2_rn(bf16_lo(v), bf16_hi(v));
      *reinterpret_cast<__half2*>(x16 + t * XP + 2 * c) = h;
    }
    stream::route_window(a.words, T, E, k, tag, rs, a.err, &s_abort);
  }
  __syncthreads();   // routing and the f16 x known to every warp
  if (s_abort) {
    if (threadIdx.x == 0) {   // let x and the shared-expert copies land first
      volatile int never = 0;
      sm100::mbar_wait(&x_bar, 0, a.err, &never, 20000000LL, false);
      for (int g2 = 0; g2 < nsg && g2 < NG; ++g2)
        sm100::mbar_wait(&full_bar[g2], 0, a.err, &never, 20000000LL, false);
      leave();
    }
    return;
  }
  const int D = rs.meta.num_slots;
  const Ranges rg = cta_ranges(b, G, Is, D * I);
  const int nr = rg.u1 - rg.u0;
  const int ngroups = nsg + (nr + RGM - 1) / RGM;

  if (b == 0 && !producer) {   // diagnostics copy of the routing
    for (int q = threadIdx.x; q < T * k; q += kConsumers) {
      a.idx[q] = rs.idx[q];
      a.weights[q] = rs.w[q];
    }
    const int* src = reinterpret_cast<const int*>(&rs.meta);
    int* dst = reinterpret_cast<int*>(a.meta);
    for (int q = threadIdx.x; q < (int)(sizeof(DecodeMeta) / 4); q += kConsumers) dst[q] = src[q];
  }

  if (producer) {   // routed groups as slots free up
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
    return;
  }

  // ---------------------------------------------------------------- consumers: groups
  const int Hw = H / 8;                  // 8-element words (codes) or chunks (bf16) per row
  const int q = threadIdx.x;             // this thread's outputs: n = 8q .. 8q+7
  const bool own = q < Hw;
  const int GS = mx_gate_scales(H), UC = mx_up_codes(H, so), US = mx_up_scales(H, so), DC = mx_down_codes(H, so);
  float acc[TMAX][8];
#pragma unroll
  for (int t = 0; t < TMAX; ++t)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[t][j] = 0.f;

  int grp = 0;
  for (; grp < ngroups; ++grp) {
    const int sg = grp % NG;
    const bool shared = grp < nsg;
    const int RG = shared ? kShGroup : RGM;
    const int first = shared ? grp * kShGroup : (grp - nsg) * RGM;
    const int nvalid = min(RG, (shared ? ns : nr) - first);
    const uint8_t* base = ring + (size_t)sg * a.slot_bytes;
    float (*s_c)[TMAX] = s_cb[grp & 1];
    sm100::mbar_wait(&full_bar[sg], (uint32_t)(grp / NG) & 1u, a.err, &s_abort, kSpinBudget);

    // gate/up: P warps per record, warp part p covers words [w0, w1) of both rows.
    // With one warp per record (P = 1) the warp's own sums are g and u, and its
    // lane 0 forms c right away; otherwise the parts meet in shared memory.
    const int P = kConsumerWarps / RG;
    {
      const int r = warp / P, p = warp - r * P;
      if (r < nvalid) {
        const int dd = shared ? 0 : (int)((unsigned)(rg.u0 + first + r) / (unsigned)I);
        const unsigned tmask = shared ? (1u << T) - 1u : rs.tmask[dd];
        const int w0 = p * Hw / P, w1 = (p + 1) * Hw / P;
        float ag[TMAX], au[TMAX];
#pragma unroll
        for (int t = 0; t < TMAX; ++t) ag[t] = au[t] = 0.f;
        if (shared) {
          const uint8_t* rec = base + (size_t)r * shs;
          for (int c = w0 + lane; c < w1; c += 32) {
            const uint4 gv = *reinterpret_cast<const uint4*>(rec + 16 * c);
            const uint4 uv = *reinterpret_cast<const uint4*>(rec + 2 * H + 16 * c);
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
              if (t < T && ((tmask >> t) & 1u)) {
                const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * XP + 8 * c);
                ag[t] = fma8_bf16(gv, xv, ag[t]);
                au[t] = fma8_bf16(uv, xv, au[t]);
              }
            }
          }
        } else {
          const uint8_t* rec = base + (size_t)r * mxs;
          for (int c = w0 + lane; c < w1; c += 32) {
            const uint32_t gw = *reinterpret_cast<const uint32_t*>(rec + 4 * c);
            const uint32_t uw = *reinterpret_cast<const uint32_t*>(rec + UC + 4 * c);
            const float gsc = e8m0_to_f32(rec[GS + c / 4]), usc = e8m0_to_f32(rec[US + c / 4]);
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
              if (t < T && ((tmask >> t) & 1u)) {
                const uint4 xv = *reinterpret_cast<const uint4*>(x16 + t * XP + 8 * c);
                ag[t] = fmaf(gsc, dot8_e2m1(gw, xv), ag[t]);
                au[t] = fmaf(usc, dot8_e2m1(uw, xv), au[t]);
              }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t < T && ((tmask >> t) & 1u)) {
            const float gs = warp_sum(ag[t]);
            const float us = warp_sum(au[t]);
            if (lane == 0) {
              if (P == 1) {   // routed record, whole row in this warp
                const int j = rs.meta.slot_j[dd][t];
                s_c[r][t] = rs.w[t * k + j] * swiglu(gs, us);
              } else {
                s_gu[r][p][t][0] = gs;
                s_gu[r][p][t][1] = us;
              }
            }
          } else if (P == 1 && lane == 0) {
            s_c[r][t] = 0.f;   // token t does not use this record's expert
          }
        }
      } else if (P == 1 && lane == 0) {
#pragma unroll
        for (int t = 0; t < TMAX; ++t) s_c[r][t] = 0.f;
      }
    }
    consumers_sync();
    if (P > 1) {
      if ((int)threadIdx.x < RG * TMAX) {   // c = w * silu(g) * u per (record, token)
        const int r = threadIdx.x / TMAX, t = threadIdx.x - r * TMAX;
        float c = 0.f;
        if (r < nvalid && t < T) {
          int j = -1;
          float w = 1.f;
          if (!shared) {
            const int dd = (int)((unsigned)(rg.u0 + first + r) / (unsigned)I);
            j = rs.meta.slot_j[dd][t];
            if (j >= 0) w = rs.w[t * k + j];
          }
          if (shared || j >= 0) {
            float g = 0.f, u = 0.f;
            for (int p = 0; p < P; ++p) {
              g += s_gu[r][p][t][0];
              u += s_gu[r][p][t][1];
            }
            c = w * swiglu(g, u);
          }
        }
        s_c[r][t] = c;
      }
      consumers_sync();
    }
    if (s_abort) break;
    // down: out[n][t] += c[r][t] * down_r[n] for this thread's 8 outputs, records in order
    if (own) {
      if (shared) {
        for (int r = 0; r < nvalid; ++r) {
          const uint4 dv = *reinterpret_cast<const uint4*>(base + (size_t)r * shs + 4 * H + 16 * q);
          const float v[8] = {bf16_lo(dv.x), bf16_hi(dv.x), bf16_lo(dv.y), bf16_hi(dv.y),
                              bf16_lo(dv.z), bf16_hi(dv.z), bf16_lo(dv.w), bf16_hi(dv.w)};
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            const float c = (t < T) ? s_c[r][t] : 0.f;
            if (c != 0.f) {
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[t][j] = fmaf(c, v[j], acc[t][j]);
            }
          }
        }
      } else {
        // Records [0, r1) use the group's first down-scale vector, [r1, nvalid)
        // the second: the group's features are consecutive, and a new vector
        // starts at the next multiple of 32 (slot ends are multiples of 32 too).
        const int i0 = (rg.u0 + first) - (int)((unsigned)(rg.u0 + first) / (unsigned)I) * I;
        const int r1 = min(nvalid, 32 - (i0 & 31));
        auto down_records = [&](int ra, int rb, const uint8_t* sv) {
          const uint2 sb = *reinterpret_cast<const uint2*>(sv + 8 * q);
          float f[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = e8m0_to_f32(((j < 4 ? sb.x : sb.y) >> (8 * (j & 3))) & 0xFFu);
          for (int r = ra; r < rb; ++r) {
            const uint32_t cw = *reinterpret_cast<const uint32_t*>(base + (size_t)r * mxs + DC + 4 * q);
            float v[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const uint32_t f2 = e2m1x2_to_f16x2((cw >> (8 * h)) & 0xFFu);
              const float2 ff = __half22float2(*reinterpret_cast<const __half2*>(&f2));
              v[2 * h] = ff.x * f[2 * h];
              v[2 * h + 1] = ff.y * f[2 * h + 1];
            }
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
              const float c = (t < T) ? s_c[r][t] : 0.f;
              if (c != 0.f) {
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[t][j] = fmaf(c, v[j], acc[t][j]);
              }
            }
          }
        };
        down_records(0, r1, base + sv_off);
        if (r1 < nvalid) down_records(r1, nvalid, base + sv_off + H);
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
      leave();
    }
    return;
  }

  // ---------------------------------------------------------------- exchange of partial outputs
  const int TP = T + (T & 1);
  if (own) {
#pragma unroll
    for (int t = 0; t < TMAX; t += 2) {
      if (t < T) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float v1 = (t + 1 < TMAX) ? acc[t + 1 < TMAX ? t + 1 : t][j] : 0.f;
          stream::st_relaxed_v2u64(a.partial + ((size_t)b * H + 8 * q + j) * TP + t, tagged(tag, acc[t][j]),
                                   tagged(tag, v1));
        }
      }
    }
  }
  consumers_sync();   // every warp is done reading the ring before it stages the exchange
  stream::collect_outputs(a.partial, reinterpret_cast<float*>(ring), tag, T, H, a.out, a.err, &s_abort);
  if (threadIdx.x == 0) leave();
}

}  // namespace

// ===========================================================================
// Host side
// ===========================================================================
static int mx_sc_off(int H) { return (H / 32 + 15) / 16 * 16; }
int stream_mx_record_stride(int H) { return 3 * H / 2 + 2 * mx_sc_off(H) + 16; }
static int mx_x_bytes(int T, int H) { return (int)(((size_t)T * (H + 8) * 2 + 127) / 128 * 128); }
static int mx_slot_bytes(int H, int rgm) {
  const size_t routed = (size_t)rgm * stream_mx_record_stride(H) + 2 * (size_t)H;
  const size_t shared = (size_t)kShGroup * stream_record_stride(H);
  return (int)((std::max(routed, shared) + 127) / 128 * 128);
}
// 16 MXFP4 records per routed group when two such slots fit beside the two x copies, else 8.
static int mx_group_records(int T, int H) {
  const size_t room = (size_t)stream::kSmemMax - 2 * (size_t)mx_x_bytes(T, H);
  return room >= 2 * (size_t)mx_slot_bytes(H, kMaxMx) ? kMaxMx : kMaxMx / 2;
}
static int mx_ring_groups(const moe_layer* L, int T) {
  const int H = L->cfg.hidden;
  const size_t xb = 2 * (size_t)mx_x_bytes(T, H);
  if (xb >= (size_t)stream::kSmemMax) return 0;
  return (int)std::min<size_t>((stream::kSmemMax - xb) / mx_slot_bytes(H, mx_group_records(T, H)), kMaxRingGroups);
}

bool stream_mx_supported(const moe_layer* L, int T) {
  const auto& c = L->cfg;
  if (c.weight_format != MOE_WEIGHTS_MXFP4 || !L->w_mx || !L->mx_dsc || !L->ws_rec) return false;
  if (c.hidden > kMxMaxH || c.hidden % 256 != 0 || T < 1 || T > kMaxDecodeT) return false;
  if ((c.num_experts + L->num_sms - 1) / L->num_sms > stream::kMaxRouterRows) return false;
  const int ng = mx_ring_groups(L, T);
  if (ng < 2) return false;
  return stream::collect_stage_bytes(L->num_sms, c.hidden, T) <=
         (size_t)ng * mx_slot_bytes(c.hidden, mx_group_records(T, c.hidden));
}

template <int TMAX>
static cudaError_t launch_stream_mx_t(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb,
                                      cudaStream_t s) {
  const auto& c = L->cfg;
  MxArgs a;
  a.x = x; a.T = T; a.H = c.hidden; a.E = c.num_experts; a.k = c.top_k; a.I = c.intermediate;
  a.Is = c.shared_intermediate;
  a.router_t = L->router_t; a.router_bias = L->router_bias; a.logit_bias = lb;
  a.rec = L->w_mx; a.dsc = L->mx_dsc; a.rec_sh = L->ws_rec;
  a.mx_stride = stream_mx_record_stride(c.hidden);
  a.sh_stride = stream_record_stride(c.hidden);
  a.sc_off = mx_sc_off(c.hidden);
  a.mx_group = mx_group_records(T, c.hidden);
  a.slot_bytes = mx_slot_bytes(c.hidden, a.mx_group);
  a.ring_groups = mx_ring_groups(L, T);
  a.x_bytes_al = mx_x_bytes(T, c.hidden);
  a.words = L->dec.logit_words; a.partial = L->dec.partial; a.ctr = L->dec.sync_ctr + 2;
  a.idx = L->dec.idx; a.weights = L->dec.weights; a.meta = L->dec.meta;
  a.out = out; a.err = L->err; a.never_set = L->never_set;
  a.force_timeout = (c.flags & MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT) ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L->num_sms);
  cfg.blockDim = dim3(stream::kThreads);
  cfg.dynamicSmemBytes = 2 * (size_t)a.x_bytes_al + (size_t)a.ring_groups * a.slot_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs co-resident: they wait on one another
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(L, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_decode_stream_mx_kernel<TMAX>, a);
  prof_mark(L, s);
  return e;
}

cudaError_t stream_mx_prepare(moe_layer* L) {
  (void)L;
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* f) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, stream::kSmemMax);
  };
  set((const void*)moe_decode_stream_mx_kernel<1>);
  set((const void*)moe_decode_stream_mx_kernel<2>);
  set((const void*)moe_decode_stream_mx_kernel<4>);
  set((const void*)moe_decode_stream_mx_kernel<8>);
  return e;
}

cudaError_t launch_stream_mx(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb, cudaStream_t s) {
  if (T <= 1) return launch_stream_mx_t<1>(L, x, out, T, lb, s);
  if (T <= 2) return launch_stream_mx_t<2>(L, x, out, T, lb, s);
  if (T <= 4) return launch_stream_mx_t<4>(L, x, out, T, lb, s);
  return launch_stream_mx_t<8>(L, x, out, T, lb, s);
}

}  // namespace moe
