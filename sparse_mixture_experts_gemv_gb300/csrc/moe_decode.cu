// Weight-streaming (GEMV) path of the MoE layer for small token windows
// (T <= MOE_DECODE_MAX_T: batch-1 decode and speculative verify windows).
//
// "Optimizing on-device inference for Apple Silicon", section "Decode: reduce
// bytes moved per token": at batch 1 the layer is bound by how many weight bytes
// it reads, so every kernel here streams each needed weight byte exactly once
// with 16-byte coalesced loads and keeps the arithmetic in registers. Section
// "Overlap independent work": the shared expert does not depend on routing, so
// its gate/up projection runs in the same kernel as the router. Section "Reduce
// intermediate and state traffic": the gated gate/up projection is one kernel
// and the down projection is fused with the routing weight and the shared
// expert. "Three ways to speed up MoE inference on DGX Spark", section
// "Optimization 3": a 4-token verify window touches up to 32 experts, so the
// window's distinct experts are read once each, for all tokens that chose them.
//
// One cooperative kernel, one CTA per SM, three phases separated by two
// bounded grid-wide synchronisations (monotonic arrival counters; the last CTA
// to arrive releases the next generation, so the kernel is also safe to replay
// from a CUDA graph):
//   phase 1  fp32 router logits + shared-expert gate/up (SwiGLU); the last CTA
//            to arrive does top-k, the renormalised softmax weights and the
//            window's distinct-expert list.
//   phase 2  one pass over the gate/up rows of each distinct expert for all
//            tokens that chose it; each warp keeps its next units on their way
//            from HBM to L2, and each CTA prefetches the down rows it needs in
//            phase 3.
//   phase 3  down rows of every distinct expert and of the shared expert,
//            weighted by the routing weights, summed in a fixed order, bf16 out.
// Latency, not arithmetic, sets the time of a batch-1 layer: warps issue their
// weight loads in batches of 16 x 16 bytes per lane before using any of them,
// and kernel boundaries are replaced by the two in-kernel synchronisations.
// The kernel is templated on the routed weight format: bf16, MXFP4 (e2m1 codes
// with e8m0 scales per 32) and groupwise affine int4 (q * s + b per 64, summed
// as s * sum(q x) + b * sum(x)). The record-streaming kernels serve bf16 and
// MXFP4 layers within their limits; this one serves the rest.
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_sm100.cuh"
#include <cuda_fp16.h>

namespace moe {

struct FmtBF16 {};
struct FmtMXFP4 {};
struct FmtInt4 {};   // groupwise affine int4: q * s + b, one (s, b) bf16 pair per 64 elements

constexpr int kGemvThreads = 512;
constexpr int kLookahead = 2;  // extra rounds of gate/up units each warp keeps on their way to L2

__device__ __forceinline__ float e8m0_scale(uint32_t s) { return ldexpf(1.0f, (int)s - 127); }

// Sum of 8 bf16 weights (one 16-byte chunk) times 8 bf16 activations.
__device__ __forceinline__ float dot8_bf16(const uint4 w, const uint4 x) {
  float a = bf16_lo(w.x) * bf16_lo(x.x);
  a = fmaf(bf16_hi(w.x), bf16_hi(x.x), a);
  a = fmaf(bf16_lo(w.y), bf16_lo(x.y), a);
  a = fmaf(bf16_hi(w.y), bf16_hi(x.y), a);
  a = fmaf(bf16_lo(w.z), bf16_lo(x.z), a);
  a = fmaf(bf16_hi(w.z), bf16_hi(x.z), a);
  a = fmaf(bf16_lo(w.w), bf16_lo(x.w), a);
  a = fmaf(bf16_hi(w.w), bf16_hi(x.w), a);
  return a;
}

// Sum of 8 bf16 weights times 8 fp32 activations (two float4).
__device__ __forceinline__ float dot8_bf16_f32(const uint4 w, const float4 a, const float4 b) {
  float s = bf16_lo(w.x) * a.x;
  s = fmaf(bf16_hi(w.x), a.y, s);
  s = fmaf(bf16_lo(w.y), a.z, s);
  s = fmaf(bf16_hi(w.y), a.w, s);
  s = fmaf(bf16_lo(w.z), b.x, s);
  s = fmaf(bf16_hi(w.z), b.y, s);
  s = fmaf(bf16_lo(w.w), b.z, s);
  s = fmaf(bf16_hi(w.w), b.w, s);
  return s;
}

// Unscaled sum of 32 e2m1 codes (16 bytes) times 32 f16 activations at xs (shared, 16-byte aligned).
__device__ __forceinline__ float dot32_e2m1_f16(const uint4 c, const uint16_t* xs) {
  const uint4* xv = reinterpret_cast<const uint4*>(xs);
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {       // 8 codes per 32-bit word, 8 activations per uint4
    const uint4 x = xv[q];
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) s = fma2_f16(e2m1x2_to_f16x2(cw[q] >> (8 * b)), xw[b], s);
  }
  return s;
}

// Two unsigned 4-bit codes of one byte (element 2i in the low nibble) -> f16x2,
// exact: 0x6400 | q is the f16 1024 + q, and 1024 is subtracted in f16.
__device__ __forceinline__ uint32_t u4x2_to_f16x2(uint32_t byte) {
  const uint32_t w = 0x64006400u | (byte & 0x0Fu) | ((byte & 0xF0u) << 12);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0x64006400u));
  return r;
}

// Unscaled sum of 32 int4 codes (16 bytes) times 32 f16 activations at xs.
__device__ __forceinline__ float dot32_u4_f16(const uint4 c, const uint16_t* xs) {
  const uint4* xv = reinterpret_cast<const uint4*>(xs);
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 x = xv[q];
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) s = fma2_f16(u4x2_to_f16x2(cw[q] >> (8 * b)), xw[b], s);
  }
  return s;
}

// ===========================================================================
// Shared pieces
// ===========================================================================
// Copy the window's routing metadata into shared memory in one round trip.
__device__ __forceinline__ void load_meta(const DecodeMeta* m, DecodeMeta* s_meta) {
  const int* src = reinterpret_cast<const int*>(m);
  int* dst = reinterpret_cast<int*>(s_meta);
  constexpr int kWords = (int)(sizeof(DecodeMeta) / 4);
  for (int q = threadIdx.x; q < kWords; q += blockDim.x) dst[q] = ldg_cg_s32(src + q);
}

// One batch of a gate/up row pair: 8 chunks of 16 bytes per row per lane.
__device__ __forceinline__ void gu_load_bf16(const uint8_t* grec, const uint8_t* urec, int b0, int nch,
                                             uint4 (&v)[16], int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int c = b0 + lane + 32 * q;
    if (c < nch) {
      v[q] = ldg_stream(grec + 16 * c);
      v[8 + q] = ldg_stream(urec + 16 * c);
    }
  }
}

template <int TMAX>
__device__ __forceinline__ void gu_fma_bf16(const uint4 (&v)[16], int b0, int nch, const uint16_t* xs, int T,
                                            int H, float (&ag)[TMAX], float (&au)[TMAX], int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int c = b0 + lane + 32 * q;
    if (c < nch) {
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const uint4 xx = *reinterpret_cast<const uint4*>(xs + t * H + 8 * c);
          ag[t] = fma8_bf16(v[q], xx, ag[t]);
          au[t] = fma8_bf16(v[8 + q], xx, au[t]);
        }
      }
    }
  }
}

// MXFP4 row pair: each 16-byte chunk holds 32 codes = one scale block; the
// scale bytes follow the codes in the row record.
__device__ __forceinline__ void gu_load_mx(const uint8_t* grec, const uint8_t* urec, int H, int b0, int nch,
                                           uint4 (&v)[16], uint32_t (&sc)[16], int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int c = b0 + lane + 32 * q;
    if (c < nch) {
      v[q] = ldg_stream(grec + 16 * c);
      v[8 + q] = ldg_stream(urec + 16 * c);
      sc[q] = __ldg(grec + H / 2 + c);
      sc[8 + q] = __ldg(urec + H / 2 + c);
    }
  }
}

template <int TMAX>
__device__ __forceinline__ void gu_fma_mx(const uint4 (&v)[16], const uint32_t (&sc)[16], int b0, int nch,
                                          const uint16_t* xs, int T, int H, float (&ag)[TMAX], float (&au)[TMAX],
                                          int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int c = b0 + lane + 32 * q;
    if (c < nch) {
      const float sg = e8m0_scale(sc[q]), su = e8m0_scale(sc[8 + q]);
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const uint16_t* xp = xs + t * H + 32 * c;   // f16 activations
          ag[t] = fmaf(dot32_e2m1_f16(v[q], xp), sg, ag[t]);
          au[t] = fmaf(dot32_e2m1_f16(v[8 + q], xp), su, au[t]);
        }
      }
    }
  }
}

// Int4 row pair: each 16-byte chunk holds 32 codes = half a 64-element group;
// the (scale, bias) pairs follow the codes in the row record.
__device__ __forceinline__ void gu_load_i4(const uint8_t* grec, const uint8_t* urec, int H, int b0, int nch,
                                           uint4 (&v)[16], uint32_t (&par)[16], int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int c = b0 + lane + 32 * q;
    if (c < nch) {
      v[q] = ldg_stream(grec + 16 * c);
      v[8 + q] = ldg_stream(urec + 16 * c);
      par[q] = __ldg(reinterpret_cast<const uint32_t*>(grec + H / 2 + 4 * (c >> 1)));
      par[8 + q] = __ldg(reinterpret_cast<const uint32_t*>(urec + H / 2 + 4 * (c >> 1)));
    }
  }
}

// sum over a chunk of (q s + b) x = s * sum(q x) + b * sum(x); sum(x) of every
// 32-element chunk of every token is staged in xsum [T][H / 32].
template <int TMAX>
__device__ __forceinline__ void gu_fma_i4(const uint4 (&v)[16], const uint32_t (&par)[16], int b0, int nch,
                                          const uint16_t* xs, const float* xsum, int T, int H, float (&ag)[TMAX],
                                          float (&au)[TMAX], int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int c = b0 + lane + 32 * q;
    if (c < nch) {
      const float sg = bf16_lo(par[q]), bg = bf16_hi(par[q]);
      const float su = bf16_lo(par[8 + q]), bu = bf16_hi(par[8 + q]);
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const uint16_t* xp = xs + t * H + 32 * c;   // f16 activations
          const float xsm = xsum[t * nch + c];
          ag[t] = fmaf(bg, xsm, fmaf(sg, dot32_u4_f16(v[q], xp), ag[t]));
          au[t] = fmaf(bu, xsm, fmaf(su, dot32_u4_f16(v[8 + q], xp), au[t]));
        }
      }
    }
  }
}

// ===========================================================================
// The fused decode kernel: one cooperative launch, one CTA per SM.
// ===========================================================================
struct FusedArgs {
  const uint16_t* x;           // bf16 [T][H]
  int T, H, E, k, I, Is;
  const float* router_t;       // fp32 [E][H]
  const float* router_bias;    // fp32 [E]
  const float* logit_bias;     // fp32 [T][E] or nullptr
  const uint16_t* ws_gu;       // bf16 [Is][2][H]
  const uint16_t* ws_down;     // bf16 [H][Is]
  const uint8_t* w_gu;         // routed gate/up records [E][I][2][rb_gu]
  int64_t rb_gu;
  const uint8_t* w_down;       // routed down records [E][H][rb_down]
  int64_t rb_down;
  // shared-memory plan (bytes): region 1 holds x in phases 1-2 and h in phase 3;
  // then this CTA's shared-expert down rows; then `slots_cap` slots of routed down rows
  int smem_r1, smem_sh, slot_stride, slots_cap, rows_max;
  float* logits;               // [T][E]
  float* h;                    // [T*k][I]
  float* h_shared;             // [T][Is]
  int* idx;                    // [T][k]     (written by CTA 0, diagnostics)
  float* weights;              // [T][k]     (written by CTA 0, diagnostics)
  DecodeMeta* meta;            //            (written by CTA 0, diagnostics)
  unsigned long long* sync_ctr;   // [2] monotonic arrival counters
  uint16_t* out;               // bf16 [T][H]
  int* err;
  const int* never_set;
  int force_timeout;
};

MOE_DEV unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide arrival (one thread per CTA): the counter only grows, so the call's
// generation is the old value / gridDim.x and the barrier opens once the
// counter reaches (generation + 1) * gridDim.x.
MOE_DEV unsigned long long grid_arrive(unsigned long long* ctr) {
  __threadfence();
  return atomicAdd(ctr, 1ull) / gridDim.x;
}
// Bounded wait (one thread per CTA) until every CTA of generation `gen` arrived.
MOE_DEV bool grid_wait(const unsigned long long* ctr, unsigned long long gen, int* err) {
  const unsigned long long target = (gen + 1) * gridDim.x;
  const long long t0 = clock64();
  while (ld_acquire_u64(ctr) < target) {
    if (clock64() - t0 > 4000000000LL) {  // ~2 s: something is wrong, do not hang the GPU
      set_error(err, kDevTimeout);
      return false;
    }
  }
  return true;
}

template <int TMAX, class Fmt>
__global__ void __launch_bounds__(kGemvThreads, 1)
moe_decode_fused_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  // An error word left set by an earlier call means the layer's cross-CTA
  // counters and tagged words may be mid-generation: do nothing (outputs stay
  // undefined) until moe_layer_sync_status has read and cleared it. Every CTA
  // reads the same value: it was written before this launch began.
  if (*reinterpret_cast<const volatile int*>(a.err) != 0) return;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);   // phases 1-2: x [T][H] bf16
  uint8_t* s_shrows = smem + a.smem_r1;               // shared-expert down rows [n0, n1) x Is bf16
  uint8_t* s_rows = s_shrows + a.smem_sh;             // routed down rows, slot d at d * slot_stride
  __shared__ DecodeMeta s_meta;
  __shared__ float s_w[kMaxDecodeT * kMaxTopK];
  __shared__ int s_idx[kMaxDecodeT * kMaxTopK];
  __shared__ int s_slot_of[kMaxDecodeT * kMaxTopK];
  __shared__ int s_router_done;
  __shared__ int s_abort;
  __shared__ unsigned long long s_gen;
  __shared__ __align__(8) uint64_t bar_sh, bar_rt;
  __shared__ float s_rpart[4 * 4 * kMaxDecodeT];   // router-row quarter partials [row][quarter][t]
  __shared__ int s_rcnt[4];

  const int T = a.T, H = a.H, E = a.E, I = a.I, Is = a.Is, k = a.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int nw = kGemvThreads / 32;
  const int G = gridDim.x, b = blockIdx.x;
  const int n0 = (int)((int64_t)b * H / G), n1 = (int)((int64_t)(b + 1) * H / G);  // phase-3 rows
  const int nrows = n1 - n0;
  const int nr = (E - b + G - 1) / G;               // router rows b, b + G, ... of this CTA
  const int sh0 = (int)((int64_t)b * Is / G), sh1 = (int)((int64_t)(b + 1) * Is / G);
  constexpr bool kMx = std::is_same<Fmt, FmtMXFP4>::value;
  constexpr bool kI4 = std::is_same<Fmt, FmtInt4>::value;
  uint16_t* xs16 = xs + (size_t)T * H;                // MXFP4 / int4 layers: x as f16 for the code products
  float* xsum = reinterpret_cast<float*>(xs16 + (size_t)T * H);  // int4: sum of x per 32 elements [T][H/32]

  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar_sh, 1);
    sm100::mbar_init(&bar_rt, 1);
    sm100::fence_barrier_init();
    s_router_done = 0;
    s_abort = 0;
    for (int r = 0; r < 4; ++r) s_rcnt[r] = 0;
    if (nr == 0) s_gen = grid_arrive(&a.sync_ctr[0]);  // no router rows: arrive at once
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (a.force_timeout && b == 0 && !bounded_wait_flag(a.never_set, 2000000LL)) set_error(a.err, kDevTimeout);
    // shared-expert down rows of phase 3 do not depend on routing: copy them now
    const uint32_t bytes = (uint32_t)(nrows * Is * 2);
    sm100::mbar_arrive_expect_tx(&bar_sh, bytes);
    if (bytes) sm100::bulk_copy_g2s(s_shrows, a.ws_down + (int64_t)n0 * Is, bytes, &bar_sh);
  }

  // ------------------------------------------------ phase 1: router + shared gate/up
  // Items: (router row r of this CTA, quarter of H) for r < nr, then this CTA's
  // shared-expert units. The last quarter to finish a row adds the four partial
  // sums in order and writes the logit.
  const int nri = 4 * nr;
  const int nch_r = H / 4;                      // 16-byte chunks (4 floats) of a router row
  uint4 v[16];
  {
    const int slot = warp;   // first item of this warp: loads issued before x arrives
    if (slot < nri) {
      const float* row = a.router_t + (size_t)(b + (slot >> 2) * G) * H;
      const int qlo = (slot & 3) * nch_r / 4, qhi = ((slot & 3) + 1) * nch_r / 4;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int c = qlo + lane + 32 * q;
        if (c < qhi) v[q] = ldg_stream(row + 4 * c);
      }
    } else if (slot - nri < sh1 - sh0) {
      const uint8_t* grec = reinterpret_cast<const uint8_t*>(a.ws_gu + (size_t)(sh0 + slot - nri) * 2 * H);
      gu_load_bf16(grec, grec + 2 * H, 0, H / 8, v, lane);
    }
  }
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = threadIdx.x; i < T * H / 8; i += blockDim.x) {
      const uint4 v8 = src[i];
      dst[i] = v8;
      if (kMx || kI4) {  // exact for |x| >= 2^-14 (bf16 has fewer significand bits than f16)
        const uint32_t w4[4] = {v8.x, v8.y, v8.z, v8.w};
        uint32_t h4[4];
        bool x_range = false;   // |x| above the f16 range: reported, never rounded to infinity silently
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          x_range |= f16_overflows(bf16_lo(w4[q])) || f16_overflows(bf16_hi(w4[q]));
          const __half2 hh = __floats2half2_rn(bf16_lo(w4[q]), bf16_hi(w4[q]));
          h4[q] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        if (x_range) set_error(a.err, kDevCheck);
        reinterpret_cast<uint4*>(xs16)[i] = make_uint4(h4[0], h4[1], h4[2], h4[3]);
      }
    }
  }
  __syncthreads();
  if (kI4) {  // fixed-order fp32 sums of the bf16 x values, 32 at a time
    for (int q = threadIdx.x; q < T * (H / 32); q += blockDim.x) {
      const uint32_t* xw = reinterpret_cast<const uint32_t*>(xs) + 16 * q;
      float sm = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) sm += bf16_lo(xw[i]) + bf16_hi(xw[i]);
      xsum[q] = sm;
    }
    __syncthreads();
  }
  for (int slot = warp; slot < nri + (sh1 - sh0); slot += nw) {
    const bool preloaded = slot == warp;
    if (slot < nri) {
      const int rl = slot >> 2, qt = slot & 3;
      const int u = b + rl * G;
      const float* row = a.router_t + (size_t)u * H;
      const int qlo = qt * nch_r / 4, qhi = (qt + 1) * nch_r / 4;
      float acc[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
      for (int b0 = qlo; b0 < qhi; b0 += 32 * 16) {
        if (!(preloaded && b0 == qlo)) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int c = b0 + lane + 32 * q;
            if (c < qhi) v[q] = ldg_stream(row + 4 * c);
          }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int c = b0 + lane + 32 * q;
          if (c < qhi) {
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
              if (t < T) {
                const uint2 xx = *reinterpret_cast<const uint2*>(xs + t * H + 4 * c);
                float sacc = acc[t];
                sacc = fmaf(__uint_as_float(v[q].x), bf16_lo(xx.x), sacc);
                sacc = fmaf(__uint_as_float(v[q].y), bf16_hi(xx.x), sacc);
                sacc = fmaf(__uint_as_float(v[q].z), bf16_lo(xx.y), sacc);
                sacc = fmaf(__uint_as_float(v[q].w), bf16_hi(xx.y), sacc);
                acc[t] = sacc;
              }
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const float sum = warp_sum(acc[t]);
          if (lane == t) s_rpart[(rl * 4 + qt) * kMaxDecodeT + t] = sum;
        }
      }
      __threadfence_block();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = (atomicAdd(&s_rcnt[rl], 1) == 3);
      last = __shfl_sync(0xFFFFFFFFu, last, 0);
      if (last) {  // all four quarters of row u are in: logit = ordered sum + biases
        __threadfence_block();
        if (lane < T) {
          const volatile float* pp = s_rpart + rl * 4 * kMaxDecodeT + lane;
          float sl = pp[0];
          sl += pp[kMaxDecodeT];
          sl += pp[2 * kMaxDecodeT];
          sl += pp[3 * kMaxDecodeT];
          sl += a.router_bias[u];
          if (a.logit_bias) sl += a.logit_bias[(size_t)lane * E + u];
          a.logits[(size_t)lane * E + u] = sl;
        }
        __threadfence();
        __syncwarp();
        // the warp completing this CTA's last router row arrives for the whole CTA
        if (lane == 0 && atomicAdd(&s_router_done, 1) == nr - 1) s_gen = grid_arrive(&a.sync_ctr[0]);
      }
    } else {
      const int i = sh0 + slot - nri;
      const uint8_t* grec = reinterpret_cast<const uint8_t*>(a.ws_gu + (size_t)i * 2 * H);
      const uint8_t* urec = grec + 2 * H;
      const int nch = H / 8;
      float ag[TMAX], au[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) ag[t] = au[t] = 0.f;
      for (int b0 = 0; b0 < nch; b0 += 32 * 8) {
        if (!(preloaded && b0 == 0)) gu_load_bf16(grec, urec, b0, nch, v, lane);
        gu_fma_bf16<TMAX>(v, b0, nch, xs, T, H, ag, au, lane);
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const float gs = warp_sum(ag[t]);
          const float us = warp_sum(au[t]);
          if (lane == t) a.h_shared[(size_t)t * Is + i] = swiglu(gs, us);
        }
      }
    }
  }

  // ------------------------------------------------ sync A: all router logits written
  __syncthreads();
  if (threadIdx.x == 0 && !grid_wait(&a.sync_ctr[0], s_gen, a.err)) s_abort = 1;
  __syncthreads();
  if (s_abort) return;

  // Every CTA derives the routing itself from the logits (identical inputs,
  // identical arithmetic): top-k, renormalised weights, distinct experts.
  if (warp < T) {
    const int t = warp;
    if (E <= 256) warp_topk<1>(a.logits + (size_t)t * E, E, k, lane, s_idx + t * k, s_w + t * k);
    else warp_topk<2>(a.logits + (size_t)t * E, E, k, lane, s_idx + t * k, s_w + t * k);
    __syncwarp();
    if (b == 0 && lane < k) {
      a.idx[t * k + lane] = s_idx[t * k + lane];
      a.weights[t * k + lane] = s_w[t * k + lane];
    }
  }
  __syncthreads();
  if (warp == 0 && T == 1) {  // one token: its k experts are the slots, in order
    for (int q = lane; q < k * kMaxDecodeT; q += 32) s_meta.slot_j[q / kMaxDecodeT][q % kMaxDecodeT] = -1;
    __syncwarp();
    if (lane < k) {
      s_meta.slot_expert[lane] = s_idx[lane];
      s_meta.slot_j[lane][0] = (signed char)lane;
    }
    if (lane == 0) s_meta.num_slots = k;
  } else if (warp == 0) {
    const int n = T * k;
    bool first[2] = {false, false};
    int firstpos[2] = {0, 0};
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int aidx = lane + 32 * h2;
      if (aidx < n) {
        const int e = s_idx[aidx];
        int q = 0;
        while (s_idx[q] != e) ++q;
        first[h2] = (q == aidx);
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
    __syncwarp();
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int aidx = lane + 32 * h2;
      if (aidx < n) {
        const int slot = s_slot_of[firstpos[h2]];
        if (first[h2]) s_meta.slot_expert[slot] = s_idx[aidx];
        s_meta.slot_j[slot][aidx / k] = (signed char)(aidx % k);
      }
    }
    if (lane == 0) s_meta.num_slots = D;
  }
  __syncthreads();
  const int D = s_meta.num_slots;
  if (b == 0) {  // diagnostics copy of the window's routing metadata
    const int* src = reinterpret_cast<const int*>(&s_meta);
    int* dst = reinterpret_cast<int*>(a.meta);
    for (int q = threadIdx.x; q < (int)(sizeof(DecodeMeta) / 4); q += blockDim.x) dst[q] = src[q];
  }

  // ------------------------------------------------ phase 2: routed gate/up
  const int d_smem = D < a.slots_cap ? D : a.slots_cap;  // slots whose down rows go to shared memory
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)(nrows * a.rb_down);
    sm100::mbar_arrive_expect_tx(&bar_rt, bytes * d_smem);
    if (bytes)
      for (int d = 0; d < d_smem; ++d)
        sm100::bulk_copy_g2s(s_rows + (size_t)d * a.slot_stride,
                             a.w_down + ((int64_t)s_meta.slot_expert[d] * H + n0) * a.rb_down, bytes, &bar_rt);
  }
  if (threadIdx.x == 32 && nrows > 0) {  // the remaining slots' down rows: HBM -> L2
    for (int d = d_smem; d < D; ++d)
      prefetch_l2_bulk(a.w_down + ((int64_t)s_meta.slot_expert[d] * H + n0) * a.rb_down,
                       (uint32_t)(nrows * a.rb_down));
  }
  const int64_t U = (int64_t)D * I;
  const int64_t u0 = U * b / G, u1 = U * (b + 1) / G;
  const int64_t unit_bytes = 2 * a.rb_gu;
  if (lane == 0) {  // this warp's next rounds of units: HBM -> L2
    for (int r = 0; r <= kLookahead; ++r) {
      const int64_t u = u0 + warp + (int64_t)nw * r;
      if (u < u1)
        prefetch_l2_bulk(a.w_gu + ((int64_t)s_meta.slot_expert[u / I] * I + u % I) * unit_bytes, (uint32_t)unit_bytes);
    }
  }
  for (int64_t u = u0 + warp; u < u1; u += nw) {
    const int64_t ua = u + (int64_t)nw * (kLookahead + 1);
    if (lane == 0 && ua < u1)
      prefetch_l2_bulk(a.w_gu + ((int64_t)s_meta.slot_expert[ua / I] * I + ua % I) * unit_bytes, (uint32_t)unit_bytes);
    const int d = (int)(u / I), i = (int)(u % I);
    const uint8_t* grec = a.w_gu + ((int64_t)s_meta.slot_expert[d] * I + i) * unit_bytes;
    const uint8_t* urec = grec + a.rb_gu;
    float ag[TMAX], au[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) ag[t] = au[t] = 0.f;
    if constexpr (std::is_same<Fmt, FmtBF16>::value) {
      const int nch = H / 8;
      for (int b0 = 0; b0 < nch; b0 += 32 * 8) {
        gu_load_bf16(grec, urec, b0, nch, v, lane);
        gu_fma_bf16<TMAX>(v, b0, nch, xs, T, H, ag, au, lane);
      }
    } else if constexpr (std::is_same<Fmt, FmtMXFP4>::value) {
      const int nch = H / 32;
      uint32_t sc[16];
      for (int b0 = 0; b0 < nch; b0 += 32 * 8) {
        gu_load_mx(grec, urec, H, b0, nch, v, sc, lane);
        gu_fma_mx<TMAX>(v, sc, b0, nch, xs16, T, H, ag, au, lane);
      }
    } else {
      const int nch = H / 32;
      uint32_t par[16];
      for (int b0 = 0; b0 < nch; b0 += 32 * 8) {
        gu_load_i4(grec, urec, H, b0, nch, v, par, lane);
        gu_fma_i4<TMAX>(v, par, b0, nch, xs16, xsum, T, H, ag, au, lane);
      }
    }
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const float gsum = warp_sum(ag[t]);
        const float usum = warp_sum(au[t]);
        const int j = s_meta.slot_j[d][t];
        if (lane == t && j >= 0) a.h[((int64_t)t * k + j) * I + i] = swiglu(gsum, usum);
      }
    }
  }

  // ------------------------------------------------ sync B: all SwiGLU outputs written
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long gen = grid_arrive(&a.sync_ctr[1]);
    if (!grid_wait(&a.sync_ctr[1], gen, a.err)) s_abort = 1;
    // down rows copied to shared memory during phase 2
    if (!s_abort) {
      volatile int never = 0;
      if (!sm100::mbar_wait(&bar_sh, 0, a.err, &never, 4000000000LL, false) ||
          !sm100::mbar_wait(&bar_rt, 0, a.err, &never, 4000000000LL, false))
        s_abort = 1;
    }
  }
  __syncthreads();
  if (s_abort) return;

  // ------------------------------------------------ phase 3: down + combine
  // Work items (expert slot, block of RB output rows) are spread over all warps
  // (slot D is the shared expert, weight 1); an item dots each of its rows with
  // the slot's SwiGLU outputs, read once per item. Per-warp partial sums meet in
  // shared memory and are added in warp order (deterministic).
  // SwiGLU outputs as 16-bit in shared memory: bf16 for bf16 weights, f16 for
  // MXFP4 weights (the e2m1 values are exact in f16); the shared expert is bf16.
  uint16_t* hs16 = reinterpret_cast<uint16_t*>(smem);          // [T*k][I]
  uint16_t* hss16 = hs16 + (size_t)T * k * I;                  // [T][Is]
  float* s_part = reinterpret_cast<float*>(s_rows + (size_t)a.slots_cap * a.slot_stride);  // [nw][rows_max][T]
  {
    const int n4 = T * k * I / 4;
    bool h_range = false;   // an f16 SwiGLU output above the f16 range: reported, never silently infinite
    for (int q = threadIdx.x; q < n4; q += blockDim.x) {
      const uint4 f = ldg_cg(reinterpret_cast<const uint4*>(a.h) + q);
      uint2 o;
      if (kMx || kI4) {
        h_range |= f16_overflows(__uint_as_float(f.x)) || f16_overflows(__uint_as_float(f.y)) ||
                   f16_overflows(__uint_as_float(f.z)) || f16_overflows(__uint_as_float(f.w));
        const __half2 p0 = __floats2half2_rn(__uint_as_float(f.x), __uint_as_float(f.y));
        const __half2 p1 = __floats2half2_rn(__uint_as_float(f.z), __uint_as_float(f.w));
        o.x = *reinterpret_cast<const uint32_t*>(&p0);
        o.y = *reinterpret_cast<const uint32_t*>(&p1);
      } else {
        o.x = (uint32_t)f32_to_bf16_rne(__uint_as_float(f.x)) | ((uint32_t)f32_to_bf16_rne(__uint_as_float(f.y)) << 16);
        o.y = (uint32_t)f32_to_bf16_rne(__uint_as_float(f.z)) | ((uint32_t)f32_to_bf16_rne(__uint_as_float(f.w)) << 16);
      }
      reinterpret_cast<uint2*>(hs16)[q] = o;
    }
    if (h_range) set_error(a.err, kDevCheck);
    const int s4 = T * Is / 4;
    for (int q = threadIdx.x; q < s4; q += blockDim.x) {
      const uint4 f = ldg_cg(reinterpret_cast<const uint4*>(a.h_shared) + q);
      uint2 o;
      o.x = (uint32_t)f32_to_bf16_rne(__uint_as_float(f.x)) | ((uint32_t)f32_to_bf16_rne(__uint_as_float(f.y)) << 16);
      o.y = (uint32_t)f32_to_bf16_rne(__uint_as_float(f.z)) | ((uint32_t)f32_to_bf16_rne(__uint_as_float(f.w)) << 16);
      reinterpret_cast<uint2*>(hss16)[q] = o;
    }
    for (int q = threadIdx.x; q < nw * a.rows_max * T; q += blockDim.x) s_part[q] = 0.f;
  }
  __syncthreads();
  constexpr int RB = TMAX <= 2 ? 8 : (TMAX <= 4 ? 4 : 2);   // rows per item
  const int npass = (nrows + RB - 1) / RB;
  const int nslots = D + (Is > 0 ? 1 : 0);
  for (int item = warp; item < nslots * npass; item += nw) {
    const int sd = item / npass, r0 = (item - sd * npass) * RB;
    const bool shared = (sd == D);
    const bool mx = !shared && kMx;
    const bool i4 = !shared && kI4;
    const int K = shared ? Is : I;
    const int nsub = K / 8;                    // 8-element sub-chunks of a row
    const bool in_smem = shared || sd < d_smem;
    const uint8_t* rows_base;
    int64_t rstride;
    if (shared) { rows_base = s_shrows; rstride = (int64_t)Is * 2; }
    else if (in_smem) { rows_base = s_rows + (size_t)sd * a.slot_stride; rstride = a.rb_down; }
    else { rows_base = a.w_down + ((int64_t)s_meta.slot_expert[sd] * H + n0) * a.rb_down; rstride = a.rb_down; }
    float wt[TMAX];
    const uint16_t* hrow[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      wt[t] = 0.f;
      hrow[t] = nullptr;
      if (t < T) {
        if (shared) { wt[t] = 1.f; hrow[t] = hss16 + (size_t)t * Is; }
        else {
          const int j = s_meta.slot_j[sd][t];
          if (j >= 0) { wt[t] = s_w[t * k + j]; hrow[t] = hs16 + ((size_t)t * k + j) * I; }
        }
      }
    }
    float acc[RB][TMAX];
#pragma unroll
    for (int rr = 0; rr < RB; ++rr)
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[rr][t] = 0.f;
    for (int c = lane; c < nsub; c += 32) {
      uint4 hv[TMAX];
      float hsum[TMAX];   // int4: sum of the 8 f16 SwiGLU outputs of this sub-chunk
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        hsum[t] = 0.f;
        if (hrow[t]) {
          hv[t] = *reinterpret_cast<const uint4*>(hrow[t] + 8 * c);
          if (i4) {
            float sm = 0.f;
            sm = fma2_f16(0x3C003C00u, hv[t].x, sm);   // 1.0 x each pair
            sm = fma2_f16(0x3C003C00u, hv[t].y, sm);
            sm = fma2_f16(0x3C003C00u, hv[t].z, sm);
            sm = fma2_f16(0x3C003C00u, hv[t].w, sm);
            hsum[t] = sm;
          }
        }
      }
      uint4 wv[RB];
      uint32_t sb[RB];
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) {  // issue the row loads of this item together
        if (r0 + rr < nrows) {
          const uint8_t* rec = rows_base + (r0 + rr) * rstride;
          if (i4) {   // 8 codes; the (scale, bias) pair of group c / 8
            wv[rr].x = in_smem ? *reinterpret_cast<const uint32_t*>(rec + 4 * c)
                               : __ldg(reinterpret_cast<const uint32_t*>(rec + 4 * c));
            sb[rr] = in_smem ? *reinterpret_cast<const uint32_t*>(rec + I / 2 + 4 * (c >> 3))
                             : __ldg(reinterpret_cast<const uint32_t*>(rec + I / 2 + 4 * (c >> 3)));
          } else if (!mx) {
            wv[rr] = in_smem ? *reinterpret_cast<const uint4*>(rec + 16 * c) : ldg_stream(rec + 16 * c);
          } else {
            wv[rr].x = in_smem ? *reinterpret_cast<const uint32_t*>(rec + 4 * c)
                               : __ldg(reinterpret_cast<const uint32_t*>(rec + 4 * c));
            sb[rr] = in_smem ? rec[I / 2 + c / 4] : __ldg(rec + I / 2 + c / 4);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) {
        if (r0 + rr < nrows) {
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (hrow[t]) {
              if (i4) {
                float sdot = 0.f;
                sdot = fma2_f16(u4x2_to_f16x2(wv[rr].x), hv[t].x, sdot);
                sdot = fma2_f16(u4x2_to_f16x2(wv[rr].x >> 8), hv[t].y, sdot);
                sdot = fma2_f16(u4x2_to_f16x2(wv[rr].x >> 16), hv[t].z, sdot);
                sdot = fma2_f16(u4x2_to_f16x2(wv[rr].x >> 24), hv[t].w, sdot);
                acc[rr][t] = fmaf(bf16_hi(sb[rr]), hsum[t], fmaf(bf16_lo(sb[rr]), sdot, acc[rr][t]));
              } else if (!mx) {
                acc[rr][t] = fma8_bf16(wv[rr], hv[t], acc[rr][t]);
              } else {  // one scale per 32 elements: constant over these 8
                float sdot = 0.f;
                sdot = fma2_f16(e2m1x2_to_f16x2(wv[rr].x), hv[t].x, sdot);
                sdot = fma2_f16(e2m1x2_to_f16x2(wv[rr].x >> 8), hv[t].y, sdot);
                sdot = fma2_f16(e2m1x2_to_f16x2(wv[rr].x >> 16), hv[t].z, sdot);
                sdot = fma2_f16(e2m1x2_to_f16x2(wv[rr].x >> 24), hv[t].w, sdot);
                acc[rr][t] = fmaf(e8m0_scale(sb[rr]), sdot, acc[rr][t]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (hrow[t] && r0 + rr < nrows) {   // warp-uniform conditions
          const float sum = warp_sum(acc[rr][t]);
          if (lane == 0) s_part[((size_t)warp * a.rows_max + r0 + rr) * T + t] += wt[t] * sum;
        }
      }
    }
  }
  __syncthreads();
  for (int q = threadIdx.x; q < nrows * T; q += blockDim.x) {
    const int r = q / T, t = q - r * T;
    float sum = 0.f;
    for (int w = 0; w < nw; ++w) sum += s_part[((size_t)w * a.rows_max + r) * T + t];
    a.out[(size_t)t * H + n0 + r] = f32_to_bf16_rne(sum);
  }
}

// ===========================================================================
// Host launcher
// ===========================================================================
size_t decode_smem_bytes_down(const moe_layer* L, int T) {
  const auto& c = L->cfg;
  return (size_t)T * ((size_t)c.top_k * c.intermediate + c.shared_intermediate) * sizeof(float);
}

constexpr int kFusedSmemMax = 216 * 1024;  // dynamic shared memory budget of the fused kernel

static size_t align16(size_t v) { return (v + 15) / 16 * 16; }

template <int TMAX, class Fmt>
static cudaError_t launch_fused_t(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* logit_bias,
                                  cudaStream_t s) {
  const auto& c = L->cfg;
  FusedArgs a;
  a.x = x; a.T = T; a.H = c.hidden; a.E = c.num_experts; a.k = c.top_k; a.I = c.intermediate;
  a.Is = c.shared_intermediate;
  a.router_t = L->router_t; a.router_bias = L->router_bias; a.logit_bias = logit_bias;
  a.ws_gu = L->ws_gu; a.ws_down = L->ws_down;
  a.w_gu = L->w_gu; a.rb_gu = L->row_bytes.gu; a.w_down = L->w_down; a.rb_down = L->row_bytes.down;
  const int rows_max = (c.hidden + L->num_sms - 1) / L->num_sms;
  constexpr bool kI4 = std::is_same<Fmt, FmtInt4>::value;
  const size_t xb = (size_t)T * c.hidden * sizeof(uint16_t) * (std::is_same<Fmt, FmtMXFP4>::value || kI4 ? 2 : 1) +
                    (kI4 ? (size_t)T * (c.hidden / 32) * sizeof(float) : 0);
  const size_t hb = decode_smem_bytes_down(L, T);
  a.smem_r1 = (int)align16(xb > hb ? xb : hb);
  a.smem_sh = (int)align16((size_t)rows_max * c.shared_intermediate * 2);
  a.slot_stride = (int)((size_t)rows_max * L->row_bytes.down);
  a.rows_max = rows_max;
  const size_t part_bytes = (size_t)(kGemvThreads / 32) * rows_max * T * sizeof(float);
  long left = (long)kFusedSmemMax - a.smem_r1 - a.smem_sh - (long)part_bytes;
  int cap = left > 0 ? (int)(left / a.slot_stride) : 0;
  if (cap > T * c.top_k) cap = T * c.top_k;
  a.slots_cap = cap;
  a.logits = L->dec.logits; a.h = L->dec.h; a.h_shared = L->dec.h_shared;
  a.idx = L->dec.idx; a.weights = L->dec.weights; a.meta = L->dec.meta;
  a.sync_ctr = L->dec.sync_ctr;
  a.out = out; a.err = L->err; a.never_set = L->never_set;
  a.force_timeout = (c.flags & MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT) ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L->num_sms);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = (size_t)a.smem_r1 + a.smem_sh + (size_t)cap * a.slot_stride + part_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs co-resident: they wait on one another
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(L, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_decode_fused_kernel<TMAX, Fmt>, a);
  prof_mark(L, s);
  return e;
}

template <class Fmt>
static cudaError_t set_attrs_fmt() {
  cudaError_t e = cudaSuccess;
  auto set = [&](const void* f) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemMax);
  };
  set((const void*)moe_decode_fused_kernel<1, Fmt>);
  set((const void*)moe_decode_fused_kernel<2, Fmt>);
  set((const void*)moe_decode_fused_kernel<4, Fmt>);
  set((const void*)moe_decode_fused_kernel<8, Fmt>);
  return e;
}

cudaError_t decode_prepare(moe_layer* L) {
  cudaError_t e = set_attrs_fmt<FmtBF16>();
  if (e == cudaSuccess) e = set_attrs_fmt<FmtMXFP4>();
  if (e == cudaSuccess) e = set_attrs_fmt<FmtInt4>();
  return e;
}

template <class Fmt>
static cudaError_t launch_decode_fmt(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* lb,
                                     cudaStream_t s) {
  if (T <= 1) return launch_fused_t<1, Fmt>(L, x, out, T, lb, s);
  if (T <= 2) return launch_fused_t<2, Fmt>(L, x, out, T, lb, s);
  if (T <= 4) return launch_fused_t<4, Fmt>(L, x, out, T, lb, s);
  return launch_fused_t<8, Fmt>(L, x, out, T, lb, s);
}

cudaError_t launch_decode(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* logit_bias,
                          cudaStream_t s) {
  if (stream_supported(L, T)) return launch_stream(L, x, out, T, logit_bias, s);
  if (stream_mx_supported(L, T)) return launch_stream_mx(L, x, out, T, logit_bias, s);
  // a layer that keeps only the feature records has no rows for this kernel:
  // the grouped path serves any T
  if (!L->w_gu || !L->ws_gu) return launch_grouped(L, x, out, T, logit_bias, s);
  if (L->cfg.weight_format == MOE_WEIGHTS_MXFP4) return launch_decode_fmt<FmtMXFP4>(L, x, out, T, logit_bias, s);
  if (L->cfg.weight_format == MOE_WEIGHTS_INT4) return launch_decode_fmt<FmtInt4>(L, x, out, T, logit_bias, s);
  return launch_decode_fmt<FmtBF16>(L, x, out, T, logit_bias, s);
}

}  // namespace moe
