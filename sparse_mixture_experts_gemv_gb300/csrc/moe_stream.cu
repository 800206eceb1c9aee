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
//              routing is known) its routed records into a ring of slot groups in
//              shared memory (full/empty mbarriers). Consecutive features of one
//              expert are adjacent in HBM, so a group of records is one or two
//              contiguous copies.
//   router     the router rows are split evenly over the CTAs (1-2 rows each at
//              E = 256), copied into shared memory with x, and every logit is
//              computed by the same fp32 sequence, so equal rows give bitwise
//              equal logits wherever they land. Each is published as a 64-bit
//              word {call tag, value} by warps that never poll; readers poll
//              until every word carries the current call's tag (no separate
//              barrier).
//   top-k      every CTA derives the routing from the published logits
//              (identical inputs and arithmetic on every CTA).
//   groups     up to 8 records per group. The gate/up dot products of the group
//              are one 16-row x T-token tile: each warp multiplies its 1/16 of H
//              on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 out, rows
//              read with ldmatrix straight from the bulk-copied records), the 16
//              partial tiles are added in warp order, and c = w * silu(g) * u is
//              formed per (record, token). The down projection is a second tile
//              product: out[n][t] += sum_r down_r[n] * c[r][t] (m16n8k8, c split
//              exactly enough into two bf16 terms hi + lo), each warp owning
//              fixed 16-row tiles of the output in registers across all groups.
//              At batch 1 the layer is bound by HBM; the tensor cores are used
//              here only because they do these small products in far fewer
//              instructions than scalar FMAs, which keeps the consumers ahead of
//              the copies.
//   exchange   each CTA stores its fp32 partial outputs [H][T], fences, and adds
//              one to an arrival counter; one thread per CTA waits (bounded)
//              until the counter reaches this call's target, the CTA pulls its
//              slice of outputs from every CTA into shared memory, adds the
//              parts in a fixed CTA order (deterministic) and writes bf16.
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_sm100.cuh"
#include "moe_stream_common.cuh"

namespace moe {

namespace {

using stream::kConsumerWarps;
using stream::kConsumers;
using stream::kMaxRingGroups;
using stream::kMaxRouterRows;
using stream::kSpinBudget;
constexpr int kStreamThreads = stream::kThreads;
// Dynamic shared memory budget: the kernel's static part is at most 11,136 bytes
// (TMAX = 8), and a block may hold 232,448 bytes in all. 216 KB keeps two
// 8-record ring groups beside x up to 5 tokens at H = 2048 (6 and more take
// three 4-record groups).
constexpr int kStreamSmemMax = 216 * 1024;
static_assert(kStreamSmemMax + 11136 <= 232448, "static + dynamic shared memory of one block");
constexpr int kMaxGroupRecords = 8;                 // records per ring group (one 16-row MMA tile)
constexpr int kMaxStreamH = kStreamMaxHidden;       // output tiles per warp kept in registers: H / 256
constexpr int kMaxTiles = kMaxStreamH / 256;
constexpr int kMaxKSteps = kMaxStreamH / 16 / 16;    // 16-wide k-steps per warp in the gate/up tile
constexpr int kRecPad = 16;                         // bytes after each record (bank spread for ldmatrix)

struct StreamArgs {
  const uint16_t* x;           // bf16 [T][H]
  int T, H, E, k, I, Is;
  const float* router_t;       // fp32 [E][H]
  const float* router_bias;    // fp32 [E]
  const float* logit_bias;     // fp32 [T][E] or nullptr
  const uint8_t* rec;          // routed records [E][I] x rec_stride bytes
  const uint8_t* rec_sh;       // shared-expert records [Is] x rec_stride bytes
  int rec_stride;              // 6 * H + kRecPad
  int group_records;           // records per ring group (8, or 4 when x is large)
  int ring_groups;             // slot groups in the ring
  int x_bytes_al;              // bytes of the x region (T rows of H + 8 bf16, 128-aligned)
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

using stream::ld_relaxed_u64;
using stream::mma_16816;
using stream::tagged;
using stream::consumers_sync;
using stream::Ranges;
using stream::cta_ranges;

template <int TMAX>
__global__ void __launch_bounds__(kStreamThreads, 1) moe_decode_stream_kernel(const StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  // An error word left set by an earlier call means the layer's cross-CTA
  // counters and tagged words may be mid-generation: do nothing (outputs stay
  // undefined) until moe_layer_sync_status has read and cleared it. Every CTA
  // reads the same value: it was written before this launch began.
  if (*reinterpret_cast<const volatile int*>(a.err) != 0) return;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);   // x [T][H + 8] bf16 (row pitch spreads banks)
  uint8_t* ring = smem + a.x_bytes_al;                // ring_groups x group_records records

  __shared__ __align__(8) uint64_t full_bar[kMaxRingGroups];
  __shared__ __align__(8) uint64_t empty_bar[kMaxRingGroups];
  __shared__ __align__(8) uint64_t x_bar;
  __shared__ float s_rpart[kConsumerWarps][TMAX];                 // router partial sums
  __shared__ __align__(16) float s_part[kConsumerWarps][16][8];   // gate/up partial tiles [warp][row][token]
  __shared__ __align__(16) uint16_t s_chi[8][8], s_clo[8][8];     // c = w * h as bf16 hi + lo, [token][record]
  __shared__ __align__(16) uint16_t s_zero[8];                    // a zero row for missing records
  __shared__ stream::RouteSmem rs;
  __shared__ unsigned long long s_tag;
  __shared__ int s_abort;

  const int T = a.T, H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
  const int XP = H + 8;                               // x row pitch (elements)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int NG = a.ring_groups, RG = a.group_records;
  const int stride = a.rec_stride;
  const bool producer = (warp == kConsumerWarps);

  if (threadIdx.x == 0) {
    for (int g = 0; g < NG; ++g) {
      sm100::mbar_init(&full_bar[g], 1);
      sm100::mbar_init(&empty_bar[g], kConsumerWarps);
    }
    sm100::mbar_init(&x_bar, 1);
    sm100::fence_barrier_init();
    s_abort = 0;
    // Every CTA adds 1 to ctr when it leaves, so at the start of a call
    // ctr / G = calls completed. No CTA of this call leaves before it has read
    // every CTA's partial outputs, which each CTA publishes after reading ctr.
    s_tag = ld_relaxed_u64(a.ctr) / (unsigned long long)G + 1ull;
  }
  if (threadIdx.x < 8) s_zero[threadIdx.x] = 0;
  __syncthreads();
  const unsigned long long tag = s_tag;
  // Every exit path of every CTA calls this exactly once (thread 0), after the
  // CTA has read everything of this call that other CTAs publish.
  auto leave = [&]() { atomicAdd(a.ctr, 1ull); };

  const Ranges rg0 = cta_ranges(b, G, Is, 0);   // shared range does not depend on routing
  const int ns = rg0.sh1 - rg0.sh0;
  // A CTA's records are its ns shared-expert records, then its routed records,
  // cut into groups of RG: groups [0, ns / RG) are all shared and go out before
  // routing; a group that starts in the shared part and ends in the routed part
  // ("mixed") has its shared records copied before routing and the rest after.
  const int nfull_sh = ns / RG;                 // all-shared groups
  const int gmix = (ns % RG) ? nfull_sh : -1;   // the mixed group, if any

  // ---------------------------------------------------------------- producer: x + shared records
  // Lane 0 of the producer warp posts a group's byte count and copies each
  // contiguous run of records (routed records may cross from one expert's last
  // feature to the next slot's first).
  auto copy_shared = [&](uint8_t* dst, int p0, int cnt, uint64_t* bar) {
    sm100::bulk_copy_g2s(dst, a.rec_sh + (size_t)(rg0.sh0 + p0) * stride, (uint32_t)(cnt * stride), bar);
  };
  auto copy_routed = [&](uint8_t* dst, int u, int cnt, uint64_t* bar) {
    while (cnt > 0) {
      const unsigned d = (unsigned)u / (unsigned)I, i = (unsigned)u - d * (unsigned)I;
      const int run = min(cnt, I - (int)i);
      sm100::bulk_copy_g2s(dst, a.rec + ((size_t)rs.meta.slot_expert[d] * I + i) * stride, (uint32_t)(run * stride),
                           bar);
      dst += (size_t)run * stride;
      u += run;
      cnt -= run;
    }
  };
  // part: 0 = all of the group, 1 = its shared records only (before routing), 2 = the rest
  auto issue_group = [&](int grp, int part, int u0, int nr) {
    const int sg = grp % NG;
    uint8_t* dst = ring + (size_t)sg * RG * stride;
    if (lane == 0) {
      const int p0 = grp * RG;
      const int p1 = part == 1 ? min(ns, p0 + RG) : min(ns + nr, p0 + RG);
      const int sh_n = max(0, min(ns, p1) - p0);
      const int rt_n = part == 1 ? 0 : (p1 - p0) - sh_n;
      if (part == 1) {
        if (grp == gmix) sm100::mbar_expect_tx(&full_bar[sg], (uint32_t)(sh_n * stride));
        else sm100::mbar_arrive_expect_tx(&full_bar[sg], (uint32_t)(sh_n * stride));
        copy_shared(dst, p0, sh_n, &full_bar[sg]);
      } else if (part == 2) {
        sm100::mbar_arrive_expect_tx(&full_bar[sg], (uint32_t)(rt_n * stride));
        copy_routed(dst + (size_t)sh_n * stride, u0 + max(0, p0 - ns), rt_n, &full_bar[sg]);
      } else {
        sm100::mbar_arrive_expect_tx(&full_bar[sg], (uint32_t)((sh_n + rt_n) * stride));
        if (sh_n > 0) copy_shared(dst, p0, sh_n, &full_bar[sg]);
        copy_routed(dst + (size_t)sh_n * stride, u0 + max(0, p0 - ns), rt_n, &full_bar[sg]);
      }
    }
    __syncwarp();
  };
  const int npre = min(NG, nfull_sh + (gmix >= 0 ? 1 : 0));   // groups whose shared records go out before routing
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
    }
    // The shared-expert records go out once x has landed: issued at kernel
    // start, their copies would queue ahead of x, the router rows and the
    // router's logit exchange, all of which are on the critical path.
    if (lane == 0) {
      volatile int never = 0;
      sm100::mbar_wait(&x_bar, 0, a.err, &never, kSpinBudget, false);
    }
    __syncwarp();
    for (int g = 0; g < npre; ++g) issue_group(g, 1, 0, 0);
  }

  // ---------------------------------------------------------------- consumers: router logits, routing
  if (!producer) {
    if (threadIdx.x == 0 && a.force_timeout && b == 0 && !bounded_wait_flag(a.never_set, 2000000LL))
      set_error(a.err, kDevTimeout);
    stream::router_publish<TMAX>(xs, XP, T, H, E, a.router_t, a.router_bias, a.logit_bias, a.words, tag, &x_bar,
                                 a.err, &s_abort, s_rpart, router_smem);
    stream::route_window(a.words, T, E, k, tag, rs, a.err, &s_abort);
  }
  __syncthreads();   // routing known to every warp, producer included
  if (s_abort) {
    // nothing routed was issued; let x and the shared-expert copies land first
    // (the mixed group's phase still needs its arrival)
    if (threadIdx.x == 0) {
      volatile int never = 0;
      sm100::mbar_wait(&x_bar, 0, a.err, &never, 20000000LL, false);
      for (int g2 = 0; g2 < npre; ++g2) {
        if (g2 == gmix) sm100::mbar_arrive(&full_bar[g2]);
        sm100::mbar_wait(&full_bar[g2], 0, a.err, &never, 20000000LL, false);
      }
      stream::exchange_arrive(a.arrivals);
      leave();
    }
    return;
  }

  const int D = rs.meta.num_slots;
  const int U = D * I;
  const Ranges rg = cta_ranges(b, G, Is, U);
  const int nr = rg.u1 - rg.u0;
  const int ngroups = (ns + nr + RG - 1) / RG;

  if (b == 0 && !producer) {   // diagnostics copy of the routing
    for (int q = threadIdx.x; q < T * k; q += kConsumers) {
      a.idx[q] = rs.idx[q];
      a.weights[q] = rs.w[q];
    }
    const int* src = reinterpret_cast<const int*>(&rs.meta);
    int* dst = reinterpret_cast<int*>(a.meta);
    for (int q = threadIdx.x; q < (int)(sizeof(DecodeMeta) / 4); q += kConsumers) dst[q] = src[q];
  }

  // ---------------------------------------------------------------- producer: routed records
  if (producer) {
    if (gmix >= 0 && gmix < npre) issue_group(gmix, 2, rg.u0, nr);   // the mixed group's routed records
    for (int issued = npre; issued < ngroups; ++issued) {
      bool go = !s_abort;
      if (go && issued >= NG && lane == 0) {
        const int sg = issued % NG;
        const uint32_t par = (uint32_t)((issued / NG) - 1) & 1u;
        go = sm100::mbar_wait(&empty_bar[sg], par, a.err, &s_abort, kSpinBudget);
      }
      if (!__shfl_sync(0xFFFFFFFFu, go, 0)) break;
      issue_group(issued, 0, rg.u0, nr);
    }
    return;   // the consumers outlive every copy issued here (they wait for each)
  }

  // ---------------------------------------------------------------- consumers: groups
  const int gq = lane >> 2, cq = lane & 3;       // mma fragment coordinates (row group, column pair)
  const int ntile = H / 256;                      // 16-row output tiles per warp (warp w: tiles w, w + 16, ...)
  const int kslice = H / kConsumerWarps;          // this warp's share of H in the gate/up products
  const int k0w = warp * kslice;
  float acc[kMaxTiles][4];
#pragma unroll
  for (int j = 0; j < kMaxTiles; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const uint32_t xs_u32 = sm100::smem_u32(xs);
  const uint32_t zero_u32 = sm100::smem_u32(s_zero);

  int grp = 0;
  for (; grp < ngroups; ++grp) {
    const int sg = grp % NG;
    const int first = grp * RG;                    // position of the group's first record in the CTA's list
    const int nvalid = min(RG, ns + nr - first);
    const uint32_t gbase = sm100::smem_u32(ring + (size_t)sg * RG * stride);
    sm100::mbar_wait(&full_bar[sg], (uint32_t)(grp / NG) & 1u, a.err, &s_abort, kSpinBudget);

    // gate/up: tile rows 0-7 = gate rows of records 0-7, rows 8-15 = their up rows;
    // this warp covers K = [k0w, k0w + kslice)
    {
      float d[4];
      stream::bf16_gu_tile<kMaxKSteps>(gbase, stride, nvalid, H, T, XP, xs_u32, zero_u32, k0w, kslice / 16, d);
      *reinterpret_cast<float2*>(&s_part[warp][gq][2 * cq]) = make_float2(d[0], d[1]);
      *reinterpret_cast<float2*>(&s_part[warp][gq + 8][2 * cq]) = make_float2(d[2], d[3]);
    }
    consumers_sync();
    if ((int)threadIdx.x < 128) {   // c = w * silu(g) * u per (record r, token t), as bf16 hi + lo
      // two lanes per (r, t): each adds half of the 16 warp partials, then they swap
      const int r = threadIdx.x >> 4, t = (threadIdx.x >> 1) & 7, hf = threadIdx.x & 1;
      float g = 0.f, u = 0.f;
#pragma unroll
      for (int q = 0; q < kConsumerWarps / 2; ++q) {
        g += s_part[hf * 8 + q][r][t];
        u += s_part[hf * 8 + q][r + 8][t];
      }
      g += __shfl_xor_sync(0xFFFFFFFFu, g, 1);
      u += __shfl_xor_sync(0xFFFFFFFFu, u, 1);
      float c = 0.f;
      if (r < nvalid && t < T) {
        const bool shared = first + r < ns;
        int j = -1;
        float w = 1.f;
        if (!shared) {
          const int dd = (int)((unsigned)(rg.u0 + first + r - ns) / (unsigned)I);
          j = rs.meta.slot_j[dd][t];
          if (j >= 0) w = rs.w[t * k + j];
        }
        if (shared || j >= 0) c = w * swiglu(g, u);
      }
      if (hf == 0) {
        const uint16_t hi = f32_to_bf16_rne(c);
        s_chi[t][r] = hi;
        s_clo[t][r] = f32_to_bf16_rne(c - __uint_as_float((uint32_t)hi << 16));
      }
    }
    consumers_sync();
    if (s_abort) break;
    // down: out[n][t] += sum_r down_r[n] * c[r][t] for this warp's output tiles
    stream::bf16_down_tiles<kMaxTiles>(gbase, stride, nvalid, H, ntile, zero_u32,
                                       *reinterpret_cast<const uint32_t*>(&s_chi[gq][2 * cq]),
                                       *reinterpret_cast<const uint32_t*>(&s_clo[gq][2 * cq]), acc);
    __syncwarp();
    if (lane == 0) sm100::mbar_arrive(&empty_bar[sg]);
  }
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
  for (int j = 0; j < kMaxTiles; ++j)
    if (j < ntile) stream::publish_tile_f32(a.partial, b, H, T, 16 * (warp + kConsumerWarps * j), acc[j]);
  stream::collect_outputs_f32(a.partial, reinterpret_cast<float*>(ring), a.arrivals, tag * (unsigned long long)G, T, H,
                              a.out, a.err, &s_abort);
  if (threadIdx.x == 0) leave();
}

}  // namespace

// ===========================================================================
// Host side
// ===========================================================================
static int stream_x_bytes(int T, int H) { return (int)(((size_t)T * (H + 8) * 2 + 127) / 128 * 128); }
int stream_record_stride(int H) { return 6 * H + kRecPad; }
// 8 records per group when two such groups fit beside x, else 4.
static int stream_group_records(int T, int H) {
  const size_t room = (size_t)kStreamSmemMax - (size_t)stream_x_bytes(T, H);
  return room >= (size_t)2 * kMaxGroupRecords * stream_record_stride(H) ? kMaxGroupRecords : kMaxGroupRecords / 2;
}

static int stream_ring_groups(const moe_layer* L, int T) {
  const int H = L->cfg.hidden;
  const size_t xb = (size_t)stream_x_bytes(T, H);
  const size_t gb = (size_t)stream_group_records(T, H) * (6 * H + kRecPad);
  if (xb >= (size_t)kStreamSmemMax) return 0;
  return (int)std::min<size_t>((kStreamSmemMax - xb) / gb, kMaxRingGroups);
}

bool stream_supported(const moe_layer* L, int T) {
  const auto& c = L->cfg;
  if (c.weight_format != MOE_WEIGHTS_BF16 || !L->w_rec) return false;
  if (c.hidden > kMaxStreamH || c.hidden % 256 != 0 || T < 1 || T > kMaxDecodeT) return false;
  if ((c.num_experts + L->num_sms - 1) / L->num_sms > kMaxRouterRows) return false;
  const int ng = stream_ring_groups(L, T);
  if (ng < 2) return false;
  // the final exchange stages G x (rows of this CTA) x TP fp32 values in the ring
  return stream::collect_f32_fits(L->num_sms, c.hidden, T,
                                  (size_t)ng * stream_group_records(T, c.hidden) * stream_record_stride(c.hidden));
}

template <int TMAX>
static cudaError_t launch_stream_t(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb,
                                   cudaStream_t s) {
  const auto& c = L->cfg;
  StreamArgs a;
  a.x = x; a.T = T; a.H = c.hidden; a.E = c.num_experts; a.k = c.top_k; a.I = c.intermediate;
  a.Is = c.shared_intermediate;
  a.router_t = L->router_t; a.router_bias = L->router_bias; a.logit_bias = lb;
  a.rec = L->w_rec; a.rec_sh = L->ws_rec; a.rec_stride = stream_record_stride(c.hidden);
  a.group_records = stream_group_records(T, c.hidden);
  a.ring_groups = stream_ring_groups(L, T);
  a.x_bytes_al = stream_x_bytes(T, c.hidden);
  {
    // This CTA's router rows go by bulk copy into the shared memory behind the
    // ring when it has room, else the consumers load them from global memory.
    // (Copying them into a ring slot that no shared-expert record uses before
    // routing was measured too: slower at T = 4 on GB300, 54.4 vs 53.7 us.)
    const int G = L->num_sms;
    const size_t rbytes = (size_t)((c.num_experts + G - 1) / G) * c.hidden * 4;
    const size_t ring_end = (size_t)a.x_bytes_al + (size_t)a.ring_groups * a.group_records * a.rec_stride;
    a.router_off = ring_end + rbytes <= (size_t)kStreamSmemMax ? (int)ring_end : -1;
  }
  a.words = L->dec.logit_words; a.partial = reinterpret_cast<float*>(L->dec.partial);
  a.ctr = L->dec.sync_ctr + 2; a.arrivals = L->dec.sync_ctr + 3;
  a.idx = L->dec.idx; a.weights = L->dec.weights; a.meta = L->dec.meta;
  a.out = out; a.err = L->err; a.never_set = L->never_set;
  a.force_timeout = (c.flags & MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT) ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L->num_sms);
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = (size_t)a.x_bytes_al + (size_t)a.ring_groups * a.group_records * a.rec_stride;
  if (a.router_off >= 0)
    cfg.dynamicSmemBytes = std::max(cfg.dynamicSmemBytes,
                                    (size_t)a.router_off + (size_t)((c.num_experts + L->num_sms - 1) / L->num_sms) *
                                                               c.hidden * 4);
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
