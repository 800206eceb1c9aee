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
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

struct FmtBF16 {};
struct FmtMXFP4 {};

constexpr int kGemvThreads = 512;
constexpr int kLookahead = 2;  // extra rounds of gate/up units each warp keeps on their way to L2

// e2m1 code values (OCP MX FP4 element): sign, 2 exponent bits (bias 1), 1 mantissa bit.
__device__ __forceinline__ void fill_e2m1_lut(float* lut) {
  if (threadIdx.x < 16) {
    const int c = threadIdx.x;
    const int e = (c >> 1) & 3, m = c & 1;
    float mag = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
    lut[c] = (c & 8) ? -mag : mag;
  }
}

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

// Sum of 32 e2m1 codes (16 bytes, even element in the low nibble) times 32 bf16
// activations starting at xs (shared memory, 16-byte aligned); unscaled.
__device__ __forceinline__ float dot32_e2m1_bf16(const uint4 c, const uint16_t* xs, const float* lut) {
  const uint4* xv = reinterpret_cast<const uint4*>(xs);
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {       // 8 codes per 32-bit word, 8 activations per uint4
    const uint4 x = xv[q];
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) {     // one byte = elements 2b (low nibble), 2b+1 (high nibble)
      const uint32_t byte = (cw[q] >> (8 * b)) & 0xFFu;
      s = fmaf(lut[byte & 15u], bf16_lo(xw[b]), s);
      s = fmaf(lut[byte >> 4], bf16_hi(xw[b]), s);
    }
  }
  return s;
}

__device__ __forceinline__ float dot32_e2m1_f32(const uint4 c, const float* hs, const float* lut) {
  const float4* hv = reinterpret_cast<const float4*>(hs);
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 a = hv[2 * q], b = hv[2 * q + 1];
    const float h8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
      const uint32_t byte = (cw[q] >> (8 * bb)) & 0xFFu;
      s = fmaf(lut[byte & 15u], h8[2 * bb], s);
      s = fmaf(lut[byte >> 4], h8[2 * bb + 1], s);
    }
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
          ag[t] += dot8_bf16(v[q], xx);
          au[t] += dot8_bf16(v[8 + q], xx);
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
                                          const float* lut, int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int c = b0 + lane + 32 * q;
    if (c < nch) {
      const float sg = e8m0_scale(sc[q]), su = e8m0_scale(sc[8 + q]);
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const uint16_t* xp = xs + t * H + 32 * c;
          ag[t] = fmaf(dot32_e2m1_bf16(v[q], xp, lut), sg, ag[t]);
          au[t] = fmaf(dot32_e2m1_bf16(v[8 + q], xp, lut), su, au[t]);
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
  int64_t down_prefetch_limit; // prefetch the routed down rows during phase 2 if they total <= this
  float* logits;               // [T][E]
  float* h;                    // [T*k][I]
  float* h_shared;             // [T][Is]
  int* idx;                    // [T][k]
  float* weights;              // [T][k]
  DecodeMeta* meta;
  unsigned long long* sync_ctr;   // [2] monotonic arrival counters
  unsigned long long* sync_flag;  // [2] generation released by the last arrival
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
MOE_DEV void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// Grid-wide arrival of this CTA (thread 0 only). Returns the generation of this
// call and whether this CTA is the last to arrive.
MOE_DEV unsigned long long grid_arrive(unsigned long long* ctr, bool* last) {
  __threadfence();
  const unsigned long long t = atomicAdd(ctr, 1ull);
  *last = (t % gridDim.x) == gridDim.x - 1;
  return t / gridDim.x;
}
// Wait (thread 0 only, bounded) until generation `gen` has been released.
MOE_DEV bool grid_wait(const unsigned long long* flag, unsigned long long gen, int* err) {
  const long long t0 = clock64();
  while ((long long)(ld_acquire_u64(flag) - (gen + 1)) < 0) {
    if (clock64() - t0 > 4000000000LL) {  // ~2 s: something is wrong, do not hang the GPU
      set_error(err, kDevTimeout);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

template <int TMAX, class Fmt>
__global__ void __launch_bounds__(kGemvThreads, 1)
moe_decode_fused_kernel(const FusedArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);  // phases 1-2: x [T][H] bf16
  float* hs = reinterpret_cast<float*>(smem);        // phase 3:   h [T*k][I] fp32, then h_shared [T][Is]
  __shared__ float lut[16];
  __shared__ DecodeMeta s_meta;
  __shared__ float s_w[kMaxDecodeT * kMaxTopK];
  __shared__ int s_idx[kMaxDecodeT * kMaxTopK];
  __shared__ int s_slot_of[kMaxDecodeT * kMaxTopK];
  __shared__ int s_last;                 // this CTA arrived last at sync A
  __shared__ int s_abort;                // a grid-wide wait ran out: leave
  __shared__ unsigned long long s_gen;   // generation of sync A in this call

  const int T = a.T, H = a.H, E = a.E, I = a.I, Is = a.Is, k = a.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int nw = kGemvThreads / 32;
  const int G = gridDim.x, b = blockIdx.x;
  const int n0 = (int)((int64_t)b * H / G), n1 = (int)((int64_t)(b + 1) * H / G);  // phase-3 rows
  if constexpr (std::is_same<Fmt, FmtMXFP4>::value) fill_e2m1_lut(lut);

  if (threadIdx.x == 0) {
    if (a.force_timeout && b == 0 && !bounded_wait_flag(a.never_set, 2000000LL)) set_error(a.err, kDevTimeout);
    // shared-expert down rows of phase 3: start HBM -> L2 now
    if (Is > 0 && n1 > n0) prefetch_l2_bulk(a.ws_down + (int64_t)n0 * Is, (uint32_t)((n1 - n0) * Is * 2));
  }

  // ------------------------------------------------ phase 1: router + shared gate/up
  // CTA b: router rows r = b, b + G, ... (one per warp from warp 0 up) and the
  // shared-expert units [sh0, sh1) on the following warps.
  const int nr = (E - b + G - 1) / G;
  const int sh0 = (int)((int64_t)b * Is / G), sh1 = (int)((int64_t)(b + 1) * Is / G);
  uint4 v[16];
  {
    const int slot = warp;   // first assignment of this warp (loads issued before x arrives)
    if (slot < nr) {
      const float* row = a.router_t + (size_t)(b + slot * G) * H;
      const int nch = H / 4;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int c = lane + 32 * q;
        if (c < nch) v[q] = ldg_stream(row + 4 * c);
      }
    } else if (slot - nr < sh1 - sh0) {
      const uint8_t* grec = reinterpret_cast<const uint8_t*>(a.ws_gu + (size_t)(sh0 + slot - nr) * 2 * H);
      gu_load_bf16(grec, grec + 2 * H, 0, H / 8, v, lane);
    }
  }
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = threadIdx.x; i < T * H / 8; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  for (int slot = warp; slot < nr + (sh1 - sh0); slot += nw) {
    const bool preloaded = slot == warp;
    if (slot < nr) {
      const int u = b + slot * G;
      const float* row = a.router_t + (size_t)u * H;
      const int nch = H / 4;
      float acc[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
      for (int b0 = 0; b0 < nch; b0 += 32 * 16) {
        if (!(preloaded && b0 == 0)) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int c = b0 + lane + 32 * q;
            if (c < nch) v[q] = ldg_stream(row + 4 * c);
          }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int c = b0 + lane + 32 * q;
          if (c < nch) {
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
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          float s = warp_sum(acc[t]);
          if (lane == t) {
            s += a.router_bias[u];
            if (a.logit_bias) s += a.logit_bias[(size_t)t * E + u];
            a.logits[(size_t)t * E + u] = s;
          }
        }
      }
    } else {
      const int i = sh0 + slot - nr;
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

  // ------------------------------------------------ sync A: routing
  __syncthreads();
  if (threadIdx.x == 0) {
    bool last;
    s_gen = grid_arrive(&a.sync_ctr[0], &last);
    s_last = last ? 1 : 0;
    s_abort = 0;
  }
  __syncthreads();
  const unsigned long long genA = s_gen;
  if (s_last) {
    // Last CTA: top-k over the complete logits, weights, distinct-expert list.
    __threadfence();
    if (warp < T) {
      const int t = warp;
      constexpr int kPer = kMaxExperts / 32;
      uint32_t key[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int e = lane + 32 * j;
        key[j] = (e < E) ? f32_order_key(ldg_cg_f32(a.logits + (size_t)t * E + e)) : 0u;
      }
      float sel_v[kMaxTopK];
      int sel_e[kMaxTopK];
#pragma unroll
      for (int r = 0; r < kMaxTopK; ++r) {
        if (r < k) {
          uint32_t lk = 0u;
          int lj = 0;
#pragma unroll
          for (int j = 0; j < kPer; ++j)
            if (key[j] > lk) { lk = key[j]; lj = j; }
          const uint32_t gmax = __reduce_max_sync(0xFFFFFFFFu, lk);
          const uint32_t cand = (lk == gmax) ? (uint32_t)(lane + 32 * lj) : 0xFFFFFFFFu;
          const uint32_t gidx = __reduce_min_sync(0xFFFFFFFFu, cand);
          if (lane == (int)(gidx & 31u)) {
#pragma unroll
            for (int j = 0; j < kPer; ++j)
              if (j == (int)(gidx >> 5)) key[j] = 0u;
          }
          sel_v[r] = f32_from_order_key(gmax);
          sel_e[r] = (int)gidx;
        }
      }
      float ex[kMaxTopK], sum = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxTopK; ++r)
        if (r < k) { ex[r] = expf(sel_v[r] - sel_v[0]); sum += ex[r]; }
#pragma unroll
      for (int r = 0; r < kMaxTopK; ++r) {
        if (r < k && lane == r) {
          a.idx[t * k + r] = sel_e[r];
          a.weights[t * k + r] = ex[r] / sum;
          s_idx[t * k + r] = sel_e[r];
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
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
      for (int q = lane; q < D * kMaxDecodeT; q += 32) a.meta->slot_j[q / kMaxDecodeT][q % kMaxDecodeT] = -1;
      __syncwarp();
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int aidx = lane + 32 * h2;
        if (aidx < n) {
          const int slot = s_slot_of[firstpos[h2]];
          if (first[h2]) a.meta->slot_expert[slot] = s_idx[aidx];
          a.meta->slot_j[slot][aidx / k] = (signed char)(aidx % k);
        }
      }
      if (lane == 0) a.meta->num_slots = D;
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        st_release_u64(&a.sync_flag[0], genA + 1);
      }
    }
  }
  if (threadIdx.x == 0 && !grid_wait(&a.sync_flag[0], genA, a.err)) s_abort = 1;
  __syncthreads();
  if (s_abort) return;

  // ------------------------------------------------ phase 2: routed gate/up
  load_meta(a.meta, &s_meta);
  __syncthreads();
  const int D = s_meta.num_slots;
  const int64_t U = (int64_t)D * I;
  const int64_t u0 = U * b / G, u1 = U * (b + 1) / G;
  const int64_t unit_bytes = 2 * a.rb_gu;
  auto unit_ptr = [&](int64_t u) {
    const int d = (int)(u / I), i = (int)(u % I);
    return a.w_gu + ((int64_t)s_meta.slot_expert[d] * I + i) * unit_bytes;
  };
  if (lane == 0) {  // this warp's next rounds of units: HBM -> L2
    for (int r = 0; r <= kLookahead; ++r) {
      const int64_t u = u0 + warp + (int64_t)nw * r;
      if (u < u1) prefetch_l2_bulk(unit_ptr(u), (uint32_t)unit_bytes);
    }
  }
  if (threadIdx.x == 32 && (int64_t)D * H * a.rb_down <= a.down_prefetch_limit && n1 > n0) {
    for (int d = 0; d < D; ++d)  // phase-3 down rows of this CTA
      prefetch_l2_bulk(a.w_down + ((int64_t)s_meta.slot_expert[d] * H + n0) * a.rb_down,
                       (uint32_t)((n1 - n0) * a.rb_down));
  }
  for (int64_t u = u0 + warp; u < u1; u += nw) {
    if (lane == 0 && u + (int64_t)nw * (kLookahead + 1) < u1)
      prefetch_l2_bulk(unit_ptr(u + (int64_t)nw * (kLookahead + 1)), (uint32_t)unit_bytes);
    const int d = (int)(u / I), i = (int)(u % I);
    const uint8_t* grec = unit_ptr(u);
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
    } else {
      const int nch = H / 32;
      uint32_t sc[16];
      for (int b0 = 0; b0 < nch; b0 += 32 * 8) {
        gu_load_mx(grec, urec, H, b0, nch, v, sc, lane);
        gu_fma_mx<TMAX>(v, sc, b0, nch, xs, T, H, ag, au, lut, lane);
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
    bool last;
    const unsigned long long gen = grid_arrive(&a.sync_ctr[1], &last);
    if (last) st_release_u64(&a.sync_flag[1], gen + 1);
    if (!grid_wait(&a.sync_flag[1], gen, a.err)) s_abort = 1;
  }
  __syncthreads();
  if (s_abort) return;

  // ------------------------------------------------ phase 3: down + combine
  float* hss = hs + (size_t)T * k * I;
  for (int q = threadIdx.x; q < T * k; q += blockDim.x) s_w[q] = ldg_cg_f32(a.weights + q);
  {
    const int n16 = T * k * I / 4;
    for (int q = threadIdx.x; q < n16; q += blockDim.x)
      reinterpret_cast<uint4*>(hs)[q] = ldg_cg(reinterpret_cast<const uint4*>(a.h) + q);
    const int s16 = T * Is / 4;
    for (int q = threadIdx.x; q < s16; q += blockDim.x)
      reinterpret_cast<uint4*>(hss)[q] = ldg_cg(reinterpret_cast<const uint4*>(a.h_shared) + q);
  }
  __syncthreads();
  const bool bf = std::is_same<Fmt, FmtBF16>::value;
  const int nch = bf ? I / 8 : I / 32;
  const int F = D * nch;
  for (int n = n0 + warp; n < n1; n += nw) {
    float acc[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
    const uint16_t* srow = a.ws_down + (size_t)n * Is;
    const int snch = Is / 8;
    uint4 sv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = lane + 32 * q;
      if (c < snch) sv[q] = ldg_stream(srow + 8 * c);
    }
    for (int f0 = 0; f0 < F; f0 += 32 * 16) {
      uint32_t sc[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int f = f0 + lane + 32 * q;
        if (f < F) {
          const int d = f / nch, c = f - d * nch;
          const uint8_t* rec = a.w_down + ((int64_t)s_meta.slot_expert[d] * H + n) * a.rb_down;
          v[q] = ldg_stream(rec + 16 * c);
          if (!bf) sc[q] = __ldg(rec + I / 2 + c);
        }
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int f = f0 + lane + 32 * q;
        if (f < F) {
          const int d = f / nch, c = f - d * nch;
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (t < T) {
              const int j = s_meta.slot_j[d][t];
              if (j >= 0) {
                if (bf) {
                  const float* hp = hs + ((size_t)t * k + j) * I + 8 * c;
                  acc[t] = fmaf(s_w[t * k + j],
                                dot8_bf16_f32(v[q], *reinterpret_cast<const float4*>(hp),
                                              *reinterpret_cast<const float4*>(hp + 4)),
                                acc[t]);
                } else {
                  const float* hp = hs + ((size_t)t * k + j) * I + 32 * c;
                  acc[t] = fmaf(s_w[t * k + j] * e8m0_scale(sc[q]), dot32_e2m1_f32(v[q], hp, lut), acc[t]);
                }
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = lane + 32 * q;
      if (c < snch) {
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t < T) {
            const float* hp = hss + (size_t)t * Is + 8 * c;
            acc[t] += dot8_bf16_f32(sv[q], *reinterpret_cast<const float4*>(hp),
                                    *reinterpret_cast<const float4*>(hp + 4));
          }
        }
      }
    }
    for (int c = lane + 128; c < snch; c += 32) {  // shared rows longer than 128 chunks
      const uint4 wv = ldg_stream(srow + 8 * c);
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const float* hp = hss + (size_t)t * Is + 8 * c;
          acc[t] += dot8_bf16_f32(wv, *reinterpret_cast<const float4*>(hp), *reinterpret_cast<const float4*>(hp + 4));
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const float s = warp_sum(acc[t]);
        if (lane == t) a.out[(size_t)t * H + n] = f32_to_bf16_rne(s);
      }
    }
  }
}

// ===========================================================================
// Host launcher
// ===========================================================================
size_t decode_smem_bytes_down(const moe_layer* L, int T) {
  const auto& c = L->cfg;
  return (size_t)T * ((size_t)c.top_k * c.intermediate + c.shared_intermediate) * sizeof(float);
}

static size_t fused_smem_bytes(const moe_layer* L, int T) {
  const size_t xb = (size_t)T * L->cfg.hidden * sizeof(uint16_t);
  const size_t hb = decode_smem_bytes_down(L, T);
  return xb > hb ? xb : hb;
}

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
  a.down_prefetch_limit = 40ll << 20;
  a.logits = L->dec.logits; a.h = L->dec.h; a.h_shared = L->dec.h_shared;
  a.idx = L->dec.idx; a.weights = L->dec.weights; a.meta = L->dec.meta;
  a.sync_ctr = L->dec.sync_ctr; a.sync_flag = L->dec.sync_flag;
  a.out = out; a.err = L->err; a.never_set = L->never_set;
  a.force_timeout = (c.flags & MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT) ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L->num_sms);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = fused_smem_bytes(L, T);
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
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 210 * 1024);
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
  if (L->cfg.weight_format == MOE_WEIGHTS_MXFP4) return launch_decode_fmt<FmtMXFP4>(L, x, out, T, logit_bias, s);
  return launch_decode_fmt<FmtBF16>(L, x, out, T, logit_bias, s);
}

}  // namespace moe
