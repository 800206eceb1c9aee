// Record-streaming decode kernel of the MoE layer for MXFP4 routed experts
// (T <= MOE_DECODE_MAX_T): the same structure as the bf16 kernel in
// moe_stream.cu -- a producer warp bulk-copies per-feature records of the
// selected experts into a shared-memory ring, 16 consumer warps turn each
// record into its contribution to the output, one exchange behind an arrival
// counter adds the CTAs' fp32 partial outputs -- with the expert weights
// decoded inside the dot products. The same kernel serves groupwise affine
// int4 routed experts (Q = INT4, below).
//
// "Three ways to speed up MoE inference on DGX Spark", section "Optimization
// 1": the routed experts are MXFP4 (e2m1 codes, one e8m0 scale per 32
// elements) and the decode path reads them in that form, a quarter of the
// bf16 bytes. "Optimizing on-device inference for Apple Silicon", section
// "Decode weights during matrix multiplication": the codes are decoded in
// registers as they are multiplied, never written back in a wider format.
//
// Records (repacked at create), per (expert e, intermediate feature i): gate
// and up codes, their e8m0 scales, and the down column's codes (layout in
// moe_stream_common.cuh, "MXFP4 records on the tensor cores"). The down
// column's scales belong to (n, i / 32), i.e. to 32 consecutive features at
// once, so they are kept apart, one H-byte vector per (e, block of 32
// features), and each ring group carries the one or two vectors it needs.
// The shared expert stays bf16 and uses the bf16 kernel's record format.
//
// Consumers (tensor cores, mma.sync with f16 fragments decoded from the codes
// by cvt.rn.f16x2.e2m1x2; e2m1 values are exact in f16):
//   gate/up    a group's 16 records are two 16-row tiles (gate rows, up rows
//              of 8 records); each warp covers 1/16 of H, one 32-element block
//              at a time: two k-steps into a fresh accumulator, then scaled by
//              the row's block scale; the 16 warp parts are added in order and
//              c = w * silu(g) * u is formed per (record, token).
//   down       K = the group's records: A = code[n][r] (f16), B = c[r][t] as
//              one f16 after a power-of-two shift that keeps the group's
//              largest |c| near 2^14 (relative error 2^-12, far inside the
//              MXFP4 output bounds); each 16-row tile's result is scaled by
//              the rows' down scales and added to the fp32 output tile.
// int4 (q * s + b, one bf16 (s, b) pair per 64 elements, "Optimizing on-device
// inference for Apple Silicon", section "Decode weights during matrix
// multiplication"): codes 0..15 become exact f16 integers (0x6400 | q is
// 1024 + q), each 64-element group's dot product is s * sum(q x) + b * sum(x)
// with sum(x) taken once per call, and c enters the down tiles as f16 hi + lo
// (~22 bits) to keep the bf16 output bounds; the down bias term uses the sum of
// c over a group's records, taken by the same MMA against an all-ones A.
// At batch 1 the layer is bound by HBM; decoding e2m1 on the CUDA cores costs
// several instructions per code byte, more than an SM's share of HBM leaves
// time for, while a tensor-core fragment needs one cvt per two codes.
// Readings: x is rounded to f16 for the 4-bit products (exact for the normal
// f16 range |x| in [2^-14, 65504]; smaller values lose bits; a larger one is
// reported as a device check failure, never rounded to infinity); every sum is
// fp32.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

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
constexpr int kShGroup = 4;            // bf16 shared-expert records per shared group (one MMA tile)
constexpr int kMaxMt = kMaxMx / 8;     // 16-row gate/up tiles per group
constexpr int kMxMaxH = kStreamMxMaxHidden;   // output tiles per warp kept in registers: H / 256
// Dynamic shared memory budget: the static part is at most 19,584 bytes and a
// block may hold 232,448 bytes in all; 207 KB keeps 16-record groups up to 7
// tokens at H = 2560.
constexpr int kMxSmemMax = 207 * 1024;
static_assert(kMxSmemMax + 19584 <= 232448, "static + dynamic shared memory of one block");
// Routed record formats of this kernel: MXFP4 (e2m1 codes, one e8m0 scale per
// 32 elements) and groupwise affine int4 (q * s + b, one bf16 (s, b) pair per
// 64 elements). The int4 instantiations also stage sum(x) per 32-element block
// (2,560 bytes of static shared memory), so their dynamic budget is 3 KB lower.
enum StreamQ { Q_MXFP4 = 0, Q_INT4 = 1 };
constexpr int kI4SmemMax = kMxSmemMax - 3 * 1024;
constexpr int kMaxXBlocks = kStreamMxMaxHidden / 32;
template <int Q> constexpr int smem_budget() { return Q == Q_INT4 ? kI4SmemMax : kMxSmemMax; }

struct MxArgs {
  const uint16_t* x;           // bf16 [T][H]
  int T, H, E, k, I, Is;
  const float* router_t;       // fp32 [E][H]
  const float* router_bias;    // fp32 [E]
  const float* logit_bias;     // fp32 [T][E] or nullptr
  const uint8_t* rec;          // routed MXFP4 records [E][I] x mx_stride bytes
  const uint8_t* dsc;          // down scale vectors: MXFP4 [E][I / 32][H] bytes, int4 [E][I / 64][H] (s, b) pairs
  const uint8_t* rec_sh;       // shared-expert bf16 records [Is] x sh_stride bytes
  int mx_stride, sh_stride;    // bytes per record
  int sc_off;                  // padded bytes of one scale segment (pad16(H / 32))
  int mx_group;                // MXFP4 records per routed group (16 or 8)
  int slot_bytes;              // bytes of one ring slot group
  int ring_groups;             // slot groups in the ring
  int x_bytes_al;              // bytes of one x copy (T rows of H + 8 halves, 128-aligned)
  int router_off;              // dynamic shared-memory offset for this CTA's router rows, or -1
                               // (the rows are then loaded from global memory by the consumers)
  unsigned long long* words;   // [kMaxDecodeT][E] tagged logits
  float* partial;              // [G][H][TP] per-CTA fp32 partial outputs
  unsigned long long* ctr;     // calls completed x G (each CTA adds 1 when it leaves)
  unsigned long long* arrivals;  // partial outputs stored x G (each CTA adds 1 per call)
  int* idx;                    // [T][k]  diagnostics (CTA 0)
  float* weights;              // [T][k]
  DecodeMeta* meta;
  uint16_t* out;               // bf16 [T][H]
  int* err;
  const int* never_set;
  int force_timeout;
};

// NT = H / 256: output tiles per warp, bf16 gate/up k-steps per warp (shared
// records) and twice the MXFP4 blocks per warp, fixed at compile time so that
// the tile loops are straight-line code.
template <int TMAX, int NT, int Q>
__global__ void __launch_bounds__(stream::kThreads, 1) moe_decode_stream_mx_kernel(const MxArgs a) {
  constexpr bool kI4 = Q == Q_INT4;
  constexpr int kVecFeat = kI4 ? 64 : 32;             // features sharing one down-scale vector
  const int vbytes = kI4 ? 4 * a.H : a.H;             // bytes of one down-scale vector
  extern __shared__ __align__(128) uint8_t smem[];
  // An error word left set by an earlier call means the layer's cross-CTA
  // counters and tagged words may be mid-generation: do nothing (outputs stay
  // undefined) until moe_layer_sync_status has read and cleared it. Every CTA
  // reads the same value: it was written before this launch began.
  if (*reinterpret_cast<const volatile int*>(a.err) != 0) return;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                 // x [T][H + 8] bf16
  uint16_t* x16 = reinterpret_cast<uint16_t*>(smem + a.x_bytes_al); // x [T][H + 8] f16
  uint8_t* ring = smem + 2 * a.x_bytes_al;                          // ring_groups x slot_bytes

  __shared__ __align__(8) uint64_t full_bar[kMaxRingGroups];
  __shared__ __align__(8) uint64_t empty_bar[kMaxRingGroups];
  __shared__ __align__(8) uint64_t x_bar;
  __shared__ float s_rpart[kConsumerWarps][TMAX];                   // router partial sums
  __shared__ __align__(16) float s_part[kConsumerWarps][kMaxMt][16][8];   // gate/up partial tiles
  __shared__ float s_cf[8][kMaxMx];                                 // c = w * silu(g) * u, [token][record]
  __shared__ unsigned s_cmax[2];                                    // largest |c| of a group (bits), by parity
  __shared__ float s_xsum[kI4 ? kMaxDecodeT * kMaxXBlocks : 1];     // int4: sum of x per (token, 32-block)
  __shared__ __align__(16) uint16_t s_zero[8];                      // a zero row for missing bf16 records
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
  const int nblk = I / kVecFeat;                      // down-scale vectors per expert
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
  if (threadIdx.x < 8) s_zero[threadIdx.x] = 0;
  __syncthreads();
  const unsigned long long tag = s_tag;
  auto leave = [&]() { atomicAdd(a.ctr, 1ull); };   // once per CTA, on every exit path

  const Ranges rg0 = cta_ranges(b, G, Is, 0);
  const int ns = rg0.sh1 - rg0.sh0;
  const int nsg = (ns + kShGroup - 1) / kShGroup;   // shared (bf16) groups come first

  // (slot, block) of routed unit u: which down-scale vector it needs
  auto unit_blk = [&](int u, int& d, int& blk) {
    d = (int)((unsigned)u / (unsigned)I);
    blk = (u - d * I) / kVecFeat;
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
        sm100::mbar_arrive_expect_tx(&full_bar[sg], (uint32_t)(n * mxs + (two ? 2 : 1) * vbytes));
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
        sm100::bulk_copy_g2s(base + sv_off, a.dsc + ((size_t)rs.meta.slot_expert[d0] * nblk + b0) * vbytes,
                             (uint32_t)vbytes, &full_bar[sg]);
        if (two)
          sm100::bulk_copy_g2s(base + sv_off + vbytes, a.dsc + ((size_t)rs.meta.slot_expert[dl] * nblk + bl) * vbytes,
                               (uint32_t)vbytes, &full_bar[sg]);
      }
    }
    __syncwarp();
  };
  int issued = 0;
  const int nr_rows = (E - b + G - 1) / G;             // router rows b, b + G, ... of this CTA
  const float* router_smem = a.router_off >= 0 ? reinterpret_cast<const float*>(smem + a.router_off) : nullptr;
  if (producer) {
    if (lane == 0) {
      const uint32_t rbytes = router_smem ? (uint32_t)(nr_rows * H * 4) : 0u;
      sm100::mbar_arrive_expect_tx(&x_bar, (uint32_t)(T * H * 2) + rbytes);
      for (int t = 0; t < T; ++t)
        sm100::bulk_copy_g2s(xs + (size_t)t * XP, a.x + (size_t)t * H, (uint32_t)(H * 2), &x_bar);
      for (int m = 0; router_smem && m < nr_rows; ++m)
        sm100::bulk_copy_g2s(smem + a.router_off + (size_t)m * H * 4, a.router_t + (size_t)(b + m * G) * H,
                             (uint32_t)(H * 4), &x_bar);
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
                                 a.err, &s_abort, s_rpart, router_smem);
    bool x_range = false;   // an |x| above the f16 range: reported, never rounded to infinity silently
    for (int q = threadIdx.x; q < T * H / 2; q += kConsumers) {   // bf16 pairs -> f16 pairs
      const int t = q / (H / 2), c = q - t * (H / 2);
      const uint32_t v = *reinterpret_cast<const uint32_t*>(xs + t * XP + 2 * c);
      x_range |= f16_overflows(bf16_lo(v)) || f16_overflows(bf16_hi(v));
      const __half2 h = __floats2half2_rn(bf16_lo(v), bf16_hi(v));
      *reinterpret_cast<__half2*>(x16 + t * XP + 2 * c) = h;
    }
    if (x_range) set_error(a.err, kDevCheck);
    if constexpr (kI4) {   // sum(x) of every 32-element block and token, fp32 in a fixed order
      for (int q = threadIdx.x; q < T * (H / 32); q += kConsumers) {
        const int t = q / (H / 32), blk = q - t * (H / 32);
        const uint32_t* xw = reinterpret_cast<const uint32_t*>(xs + t * XP + 32 * blk);
        float sm = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) sm += bf16_lo(xw[i]) + bf16_hi(xw[i]);
        s_xsum[t * kMaxXBlocks + blk] = sm;
      }
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
      stream::exchange_arrive(a.arrivals);
      leave();
    }
    return;
  }
  const int D = rs.meta.num_slots;
  Ranges rg = cta_ranges(b, G, Is, D * I);
  rg.u0 &= ~1;   // routed ranges start at even features: the down columns come in pairs of records
  rg.u1 &= ~1;   // (the same rounding on both sides of every boundary; D * I is even)
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
  const int gq = lane >> 2, cq = lane & 3;            // mma fragment coordinates
  const stream::MxLayout ly = stream::mx_layout(H, so);
  constexpr int nbw = NT / 2;                          // 32-element blocks per warp (gate/up)
  const uint32_t xs_u32 = sm100::smem_u32(xs);
  const uint32_t zero_u32 = sm100::smem_u32(s_zero);
  float acc[NT][4];   // output tiles w, w + 16, ... of warp w
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  // One group; the shared (bf16) and routed (MXFP4) groups run in two loops so
  // that each loop body holds one kind's code (the loop stays in the
  // instruction cache). Returns false when the CTA aborts.
  auto run_group = [&](auto kind, int grp) -> bool {
    constexpr bool shared = decltype(kind)::value;
    const int sg = grp % NG;
    const int RG = shared ? kShGroup : RGM;
    const int first = shared ? grp * kShGroup : (grp - nsg) * RGM;
    const int nvalid = min(RG, (shared ? ns : nr) - first);
    const uint8_t* base = ring + (size_t)sg * a.slot_bytes;
    unsigned* cmax = &s_cmax[grp & 1];
    if (threadIdx.x == 0) *cmax = 0u;   // group grp - 2's value was last read before this group's first barrier
    sm100::mbar_wait(&full_bar[sg], (uint32_t)(grp / NG) & 1u, a.err, &s_abort, kSpinBudget);

    // gate/up tiles (tile m: gate rows of records 8m..8m+7, then their up rows), this warp's part of K
    {
      float d[kMaxMt][4];
      if constexpr (shared) {
        stream::bf16_gu_tile<NT>(sm100::smem_u32(base), shs, nvalid, H, T, XP, xs_u32, zero_u32,
                                 warp * (H / kConsumerWarps), NT, d[0]);
      } else {
        if constexpr (kI4)
          stream::i4_gu_tiles<kMaxMt, nbw>(base, mxs, nvalid, (nvalid + 7) / 8, ly, T, XP, x16, s_xsum, kMaxXBlocks,
                                           warp * nbw, d);
        else
          stream::mx_gu_tiles<kMaxMt, nbw, TMAX == 1 ? 1 : nbw>(base, mxs, nvalid, (nvalid + 7) / 8, ly, T, XP, x16,
                                                                 warp * nbw, d);
      }
      const int nmt = shared ? 1 : (nvalid + 7) / 8;
#pragma unroll
      for (int m = 0; m < kMaxMt; ++m) {
        if (m < nmt) {
          *reinterpret_cast<float2*>(&s_part[warp][m][gq][2 * cq]) = make_float2(d[m][0], d[m][1]);
          *reinterpret_cast<float2*>(&s_part[warp][m][gq + 8][2 * cq]) = make_float2(d[m][2], d[m][3]);
        }
      }
    }
    consumers_sync();
    if ((int)threadIdx.x < 2 * kMaxMx * 8) {   // c = w * silu(g) * u per (record r, token t)
      // two lanes per (r, t): each adds half of the 16 warp partials, then they swap
      const int r = threadIdx.x >> 4, t = (threadIdx.x >> 1) & 7, hf = threadIdx.x & 1;
      const int m = r >> 3, rr = r & 7;
      float g = 0.f, u = 0.f;
      if (r < nvalid) {
#pragma unroll
        for (int q = 0; q < kConsumerWarps / 2; ++q) {
          g += s_part[hf * 8 + q][m][rr][t];
          u += s_part[hf * 8 + q][m][rr + 8][t];
        }
      }
      g += __shfl_xor_sync(0xFFFFFFFFu, g, 1);
      u += __shfl_xor_sync(0xFFFFFFFFu, u, 1);
      float c = 0.f;
      if (r < nvalid && t < T) {
        int j = -1;
        float w = 1.f;
        if (!shared) {
          const int dd = (int)((unsigned)(rg.u0 + first + r) / (unsigned)I);
          j = rs.meta.slot_j[dd][t];
          if (j >= 0) w = rs.w[t * k + j];
        }
        if (shared || j >= 0) c = w * swiglu(g, u);
      }
      if (hf == 0) {
        s_cf[t][r] = c;
        atomicMax(cmax, __float_as_uint(fabsf(c)));   // positive floats order like their bits
      }
    }
    consumers_sync();
    if (s_abort) return false;
    // down tiles: out[n][t] += sum_r down_r[n] * c[r][t]
    if constexpr (shared) {
      uint32_t bhi, blo;
      stream::bf16_hilo2(s_cf[gq][2 * cq], s_cf[gq][2 * cq + 1], bhi, blo);
      stream::bf16_down_tiles<NT>(sm100::smem_u32(base), shs, nvalid, H, NT, zero_u32, bhi, blo, acc);
    } else {
      // c' = c * 2^-e with the group's largest |c'| in [2^14, 2^15): far inside
      // the f16 range, and hi + lo keep ~22 significant bits of every c.
      const unsigned mb = *cmax;
      const int e = mb ? (int)((mb >> 23) & 0xFFu) - 127 - 14 : 0;
      const int ec = max(-120, min(120, e));
      const float down = __uint_as_float((uint32_t)(127 - ec) << 23), up = __uint_as_float((uint32_t)(127 + ec) << 23);
      // records [0, r1) use the group's first down-scale vector, [r1, nvalid)
      // the second: a new vector starts at the next multiple of 32 features
      const int i0 = (rg.u0 + first) - (int)((unsigned)(rg.u0 + first) / (unsigned)I) * I;
      const int r1 = min(nvalid, kVecFeat - (i0 & (kVecFeat - 1)));
      const float* cr = s_cf[gq];
      const int nv = r1 < nvalid ? 2 : 1;
      uint32_t bh[2][2], bl[2][2];
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const int lo_r = v ? r1 : 0, hi_r = v ? nvalid : r1;
        auto cv = [&](int r) { return (r >= lo_r && r < hi_r) ? cr[r] : 0.f; };
        if constexpr (kI4) {   // int4: c as f16 hi + lo (the bf16 output bounds)
          stream::f16_hilo2(cv(2 * cq), cv(2 * cq + 1), down, bh[v][0], bl[v][0]);
          stream::f16_hilo2(cv(2 * cq + 8), cv(2 * cq + 9), down, bh[v][1], bl[v][1]);
        } else {               // MXFP4: c as one f16 (relative error 2^-12, inside the MXFP4 bounds)
          const __half2 h0 = __floats2half2_rn(cv(2 * cq) * down, cv(2 * cq + 1) * down);
          const __half2 h1 = __floats2half2_rn(cv(2 * cq + 8) * down, cv(2 * cq + 9) * down);
          bh[v][0] = *reinterpret_cast<const uint32_t*>(&h0);
          bh[v][1] = *reinterpret_cast<const uint32_t*>(&h1);
          bl[v][0] = bl[v][1] = 0u;
        }
      }
      if constexpr (kI4) {
        float csum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};   // sum of c over each vector's records, tokens 2cq, 2cq + 1
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          if (v < nv) {
            float s0, s1;
            stream::colsum_f16(bh[v], bl[v], s0, s1);
            csum[v][0] = s0 * up;
            csum[v][1] = s1 * up;
          }
        }
        stream::i4_down_tiles<NT>(base, mxs, nvalid, ly, nv, reinterpret_cast<const uint32_t*>(base + sv_off),
                                  reinterpret_cast<const uint32_t*>(base + sv_off + vbytes), up, bh, bl, csum, acc);
      } else {
        stream::mx_down_tiles<NT>(base, mxs, nvalid, ly, nv, base + sv_off, base + sv_off + H, up, bh, acc);
      }
    }
    __syncwarp();
    if (lane == 0) sm100::mbar_arrive(&empty_bar[sg]);
    return true;
  };
  int grp = 0;
  for (; grp < nsg; ++grp)
    if (!run_group(std::true_type{}, grp)) break;
  if (!s_abort)
    for (; grp < ngroups; ++grp)
      if (!run_group(std::false_type{}, grp)) break;
  if (s_abort) {
    // let copies still in flight land before the CTA's shared memory goes away
    if (threadIdx.x == 0) {
      volatile int never = 0;
      for (int g2 = grp; g2 < ngroups && g2 < grp + NG; ++g2)
        sm100::mbar_wait(&full_bar[g2 % NG], (uint32_t)(g2 / NG) & 1u, a.err, &never, 20000000LL, false);
      stream::exchange_arrive(a.arrivals);
      leave();
    }
    return;
  }

  // ---------------------------------------------------------------- exchange of partial outputs
#pragma unroll
  for (int j = 0; j < NT; ++j)
    stream::publish_tile_f32<TMAX == 1>(a.partial, b, H, T, 16 * (warp + kConsumerWarps * j), acc[j]);
  stream::collect_outputs_f32(a.partial, reinterpret_cast<float*>(ring), a.arrivals, tag * (unsigned long long)G, T, H,
                              a.out, a.err, &s_abort);
  if (threadIdx.x == 0) leave();
}

}  // namespace

// ===========================================================================
// Host side
// ===========================================================================
// Bytes of one scale segment of a record: MXFP4 one e8m0 byte per 32 elements,
// int4 one 4-byte (s, b) pair per 64 elements; padded to 16.
static int q_sc_off(int Q, int H) { return (Q == Q_INT4 ? H / 16 : H / 32 + 15) / 16 * 16; }
static int q_record_stride(int Q, int H) { return 3 * H / 2 + 2 * q_sc_off(Q, H) + 16; }
int stream_mx_record_stride(int H) { return q_record_stride(Q_MXFP4, H); }
int stream_i4_record_stride(int H) { return q_record_stride(Q_INT4, H); }
static int q_vec_bytes(int Q, int H) { return Q == Q_INT4 ? 4 * H : H; }
static int q_budget(int Q) { return Q == Q_INT4 ? kI4SmemMax : kMxSmemMax; }
static int mx_x_bytes(int T, int H) { return (int)(((size_t)T * (H + 8) * 2 + 127) / 128 * 128); }
static int mx_slot_bytes(int Q, int H, int rgm) {
  const size_t routed = (size_t)rgm * q_record_stride(Q, H) + 2 * (size_t)q_vec_bytes(Q, H);
  const size_t shared = (size_t)kShGroup * stream_record_stride(H);
  return (int)((std::max(routed, shared) + 127) / 128 * 128);
}
// 16 records per routed group when two such slots fit beside the two x copies, else 8.
static int mx_group_records(int Q, int T, int H) {
  const size_t room = (size_t)q_budget(Q) - 2 * (size_t)mx_x_bytes(T, H);
  return room >= 2 * (size_t)mx_slot_bytes(Q, H, kMaxMx) ? kMaxMx : kMaxMx / 2;
}
static int mx_ring_groups(const moe_layer* L, int Q, int T) {
  const int H = L->cfg.hidden;
  const size_t xb = 2 * (size_t)mx_x_bytes(T, H);
  if (xb >= (size_t)q_budget(Q)) return 0;
  return (int)std::min<size_t>((q_budget(Q) - xb) / mx_slot_bytes(Q, H, mx_group_records(Q, T, H)), kMaxRingGroups);
}
static int layer_q(const moe_layer* L) { return L->cfg.weight_format == MOE_WEIGHTS_INT4 ? Q_INT4 : Q_MXFP4; }

bool stream_mx_supported(const moe_layer* L, int T) {
  const auto& c = L->cfg;
  if (c.weight_format != MOE_WEIGHTS_MXFP4 && c.weight_format != MOE_WEIGHTS_INT4) return false;
  if (!L->w_mx || !L->mx_dsc || !L->ws_rec) return false;
  const int Q = layer_q(L);
  // 16 warps x whole 32-element blocks of H in the gate/up tiles
  if (c.hidden > kMxMaxH || c.hidden % 512 != 0 || T < 1 || T > kMaxDecodeT) return false;
  if (Q == Q_INT4 && c.intermediate % 64 != 0) return false;
  if ((c.num_experts + L->num_sms - 1) / L->num_sms > stream::kMaxRouterRows) return false;
  const int ng = mx_ring_groups(L, Q, T);
  if (ng < 2) return false;
  return stream::collect_f32_fits(L->num_sms, c.hidden, T,
                                  (size_t)ng * mx_slot_bytes(Q, c.hidden, mx_group_records(Q, T, c.hidden)));
}

template <int TMAX, int NT, int Q>
static cudaError_t launch_stream_mx_t(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb,
                                      cudaStream_t s) {
  const auto& c = L->cfg;
  MxArgs a;
  a.x = x; a.T = T; a.H = c.hidden; a.E = c.num_experts; a.k = c.top_k; a.I = c.intermediate;
  a.Is = c.shared_intermediate;
  a.router_t = L->router_t; a.router_bias = L->router_bias; a.logit_bias = lb;
  a.rec = L->w_mx; a.dsc = L->mx_dsc; a.rec_sh = L->ws_rec;
  a.mx_stride = q_record_stride(Q, c.hidden);
  a.sh_stride = stream_record_stride(c.hidden);
  a.sc_off = q_sc_off(Q, c.hidden);
  a.mx_group = mx_group_records(Q, T, c.hidden);
  a.slot_bytes = mx_slot_bytes(Q, c.hidden, a.mx_group);
  a.ring_groups = mx_ring_groups(L, Q, T);
  a.x_bytes_al = mx_x_bytes(T, c.hidden);
  {
    // This CTA's router rows go by bulk copy into the shared memory behind the
    // ring when it has room, else the consumers load them from global memory.
    const size_t rbytes = (size_t)((c.num_experts + L->num_sms - 1) / L->num_sms) * c.hidden * 4;
    const size_t ring_end = 2 * (size_t)a.x_bytes_al + (size_t)a.ring_groups * a.slot_bytes;
    a.router_off = ring_end + rbytes <= (size_t)q_budget(Q) ? (int)ring_end : -1;
  }
  a.words = L->dec.logit_words; a.partial = reinterpret_cast<float*>(L->dec.partial);
  a.ctr = L->dec.sync_ctr + 2; a.arrivals = L->dec.sync_ctr + 3;
  a.idx = L->dec.idx; a.weights = L->dec.weights; a.meta = L->dec.meta;
  a.out = out; a.err = L->err; a.never_set = L->never_set;
  a.force_timeout = (c.flags & MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT) ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L->num_sms);
  cfg.blockDim = dim3(stream::kThreads);
  cfg.dynamicSmemBytes = 2 * (size_t)a.x_bytes_al + (size_t)a.ring_groups * a.slot_bytes;
  if (a.router_off >= 0)
    cfg.dynamicSmemBytes = (size_t)a.router_off +
                           (size_t)((c.num_experts + L->num_sms - 1) / L->num_sms) * c.hidden * 4;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs co-resident: they wait on one another
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(L, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_decode_stream_mx_kernel<TMAX, NT, Q>, a);
  prof_mark(L, s);
  return e;
}

template <int NT, int Q, typename F>
static void set_all(F& set) {
  set((const void*)moe_decode_stream_mx_kernel<1, NT, Q>, q_budget(Q));
  set((const void*)moe_decode_stream_mx_kernel<2, NT, Q>, q_budget(Q));
  set((const void*)moe_decode_stream_mx_kernel<4, NT, Q>, q_budget(Q));
  set((const void*)moe_decode_stream_mx_kernel<8, NT, Q>, q_budget(Q));
}

cudaError_t stream_mx_prepare(moe_layer* L) {
  (void)L;
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* f, int bytes) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  };
  set_all<2, Q_MXFP4>(set);
  set_all<4, Q_MXFP4>(set);
  set_all<6, Q_MXFP4>(set);
  set_all<8, Q_MXFP4>(set);
  set_all<10, Q_MXFP4>(set);
  set_all<2, Q_INT4>(set);
  set_all<4, Q_INT4>(set);
  set_all<6, Q_INT4>(set);
  set_all<8, Q_INT4>(set);
  set_all<10, Q_INT4>(set);
  return e;
}

template <int NT, int Q>
static cudaError_t launch_stream_mx_nt(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb,
                                       cudaStream_t s) {
  if (T <= 1) return launch_stream_mx_t<1, NT, Q>(L, x, out, T, lb, s);
  if (T <= 2) return launch_stream_mx_t<2, NT, Q>(L, x, out, T, lb, s);
  if (T <= 4) return launch_stream_mx_t<4, NT, Q>(L, x, out, T, lb, s);
  return launch_stream_mx_t<8, NT, Q>(L, x, out, T, lb, s);
}

template <int Q>
static cudaError_t launch_stream_q(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb,
                                   cudaStream_t s) {
  switch (L->cfg.hidden / 256) {   // H % 512 == 0, H <= 2560 (stream_mx_supported)
    case 2: return launch_stream_mx_nt<2, Q>(L, x, out, T, lb, s);
    case 4: return launch_stream_mx_nt<4, Q>(L, x, out, T, lb, s);
    case 6: return launch_stream_mx_nt<6, Q>(L, x, out, T, lb, s);
    case 8: return launch_stream_mx_nt<8, Q>(L, x, out, T, lb, s);
    default: return launch_stream_mx_nt<10, Q>(L, x, out, T, lb, s);
  }
}

cudaError_t launch_stream_mx(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb, cudaStream_t s) {
  return layer_q(L) == Q_INT4 ? launch_stream_q<Q_INT4>(L, x, out, T, lb, s) : launch_stream_q<Q_MXFP4>(L, x, out, T, lb, s);
}

}  // namespace moe
