// Device helpers shared by the MoE layer kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

namespace moe {

// ---------------------------------------------------------------------------
// Device error word codes (mirrors moe_status_t values).
// ---------------------------------------------------------------------------
enum : int { kDevOk = 0, kDevTimeout = 5, kDevCheck = 6 };

MOE_DEV void set_error(int* err, int code) { atomicCAS(err, 0, code); }

// ---------------------------------------------------------------------------
// bf16 <-> fp32 (bit level; bf16 is the top half of an fp32).
// ---------------------------------------------------------------------------
MOE_DEV float bf16_lo(uint32_t two) { return __uint_as_float(two << 16); }
MOE_DEV float bf16_hi(uint32_t two) { return __uint_as_float(two & 0xFFFF0000u); }

// fp32 -> bf16 with round-to-nearest-even (finite inputs).
MOE_DEV uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// SwiGLU gate: silu(g) * u with silu(g) = g / (1 + exp(-g)).
MOE_DEV float swiglu(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Order-preserving map of an fp32 to uint32 (larger float -> larger key).
MOE_DEV uint32_t f32_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MOE_DEV float f32_from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// acc + sum of 8 bf16 weights times 8 bf16 activations, with the mixed-precision
// FMA (bf16 inputs, fp32 accumulate; the bf16 product is exact in fp32).
MOE_DEV float fma8_bf16(const uint4 w, const uint4 x, float acc) {
  asm("{\n .reg .b16 w0, w1, w2, w3, w4, w5, w6, w7, x0, x1, x2, x3, x4, x5, x6, x7;\n"
      " mov.b32 {w0, w1}, %1;\n mov.b32 {w2, w3}, %2;\n mov.b32 {w4, w5}, %3;\n mov.b32 {w6, w7}, %4;\n"
      " mov.b32 {x0, x1}, %5;\n mov.b32 {x2, x3}, %6;\n mov.b32 {x4, x5}, %7;\n mov.b32 {x6, x7}, %8;\n"
      " fma.rn.f32.bf16 %0, w0, x0, %0;\n fma.rn.f32.bf16 %0, w1, x1, %0;\n"
      " fma.rn.f32.bf16 %0, w2, x2, %0;\n fma.rn.f32.bf16 %0, w3, x3, %0;\n"
      " fma.rn.f32.bf16 %0, w4, x4, %0;\n fma.rn.f32.bf16 %0, w5, x5, %0;\n"
      " fma.rn.f32.bf16 %0, w6, x6, %0;\n fma.rn.f32.bf16 %0, w7, x7, %0;\n}"
      : "+f"(acc)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w));
  return acc;
}

// Two e2m1 codes of one byte -> f16x2 (element 2i, the low nibble, in the low half).
MOE_DEV uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(r) : "r"(byte));
  return r;
}

// acc + sum over two f16 pairs: (w.lo * x.lo + w.hi * x.hi), fp32 accumulate.
MOE_DEV float fma2_f16(uint32_t w, uint32_t x, float acc) {
  asm("{\n .reg .b16 w0, w1, x0, x1;\n mov.b32 {w0, w1}, %1;\n mov.b32 {x0, x1}, %2;\n"
      " fma.rn.f32.f16 %0, w0, x0, %0;\n fma.rn.f32.f16 %0, w1, x1, %0;\n}"
      : "+f"(acc) : "r"(w), "r"(x));
  return acc;
}

// True when a finite fp32 value lies outside the f16 range (its f16 rounding
// would be infinite). Infinite or NaN inputs are not flagged: they propagate as
// they would through fp32 arithmetic.
MOE_DEV bool f16_overflows(float v) { return fabsf(v) > 65504.0f && fabsf(v) < __int_as_float(0x7F800000); }

// e8m0 scale byte -> 2^(s - 127) as fp32 (s = 255, NaN, is never stored).
MOE_DEV float e8m0_to_f32(uint32_t s) { return __uint_as_float(s ? (s << 23) : 0x00400000u); }

// ---------------------------------------------------------------------------
// Global loads.
// ---------------------------------------------------------------------------
// Streaming 16-byte load of read-only weights: not kept in L1.
MOE_DEV uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// L2-coherent 16-byte load (data written by an earlier kernel of the same layer call).
MOE_DEV uint4 ldg_cg(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
MOE_DEV float ldg_cg_f32(const float* p) {
  float r;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}
MOE_DEV int ldg_cg_s32(const int* p) {
  int r;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// Fire-and-forget prefetch of `bytes` (multiple of 16) starting at a 16-byte
// aligned global address into L2, issued in pieces of at most 32 KB.
MOE_DEV void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  const char* c = static_cast<const char*>(p);
  while (bytes > 0) {
    const uint32_t n = bytes < 32768u ? bytes : 32768u;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(c), "r"(n) : "memory");
    c += n;
    bytes -= n;
  }
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.
// ---------------------------------------------------------------------------
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------------------
// Warp reductions.
// ---------------------------------------------------------------------------
MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Bounded spin on a device flag: returns true when *flag != 0 within `max_ns`.
MOE_DEV bool bounded_wait_flag(const volatile int* flag, long long max_ns) {
  long long t0 = (long long)clock64();
  // clock64 counts SM cycles; 2.1 GHz upper bound keeps the budget conservative.
  const long long budget = max_ns * 2;
  while (*flag == 0) {
    if ((long long)clock64() - t0 > budget) return false;
    __nanosleep(256);
  }
  return true;
}

// ===========================================================================
// Top-k of one token's logits by one warp.
// ===========================================================================
// Lane l holds the logits of experts l, l + 32, ... as order-preserving keys
// (8 G of them, 0 for experts >= E). Each of k rounds (a rolled loop: this code
// runs once per call and is mostly fetched cold, so it is kept small) takes
// every lane's largest remaining key (the lower expert on equal keys), the
// warp maximum of those (redux), the lowest expert index among equal maxima
// (second redux), and removes the winner from its lane. Writes the k experts in
// descending order (exact ties to the lower index) and their softmax weights
// renormalised over the k.
template <int G>
MOE_DEV void warp_topk_keys(uint32_t (&key)[G][8], int (&jj)[G][8], int k, int lane, int* out_e, float* out_w) {
  (void)jj;
  float v0 = 0.f, sum = 0.f, my_ex = 0.f;
  int my_e = 0;
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    uint32_t bk = 0u;
    int bq = 0;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (key[g][q] > bk) { bk = key[g][q]; bq = 8 * g + q; }   // strict: the lower local index wins a tie
    const uint32_t gmax = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t cand = (bk == gmax) ? (uint32_t)(lane + 32 * bq) : 0xFFFFFFFFu;
    const uint32_t gidx = __reduce_min_sync(0xFFFFFFFFu, cand);
    if (lane == (int)(gidx & 31u)) {   // remove the winner
      const int wq = (int)(gidx >> 5);
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (8 * g + q == wq) key[g][q] = 0u;
    }
    const float val = f32_from_order_key(gmax);
    if (r == 0) v0 = val;
    const float ex = expf(val - v0);   // renormalised softmax over the k selected logits, summed in round order
    sum += ex;
    if (lane == r) { my_ex = ex; my_e = (int)gidx; }
  }
  if (lane < k) {
    out_e[lane] = my_e;
    out_w[lane] = my_ex / sum;
  }
}

template <int G>
MOE_DEV void warp_topk(const float* logits, int E, int k, int lane, int* out_e, float* out_w) {
  uint32_t key[G][8];
  int jj[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane + 32 * (8 * g + q);
      key[g][q] = (e < E) ? f32_order_key(ldg_cg_f32(logits + e)) : 0u;
    }
  warp_topk_keys<G>(key, jj, k, lane, out_e, out_w);
}

}  // namespace moe
