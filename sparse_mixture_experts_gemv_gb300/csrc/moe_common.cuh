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

}  // namespace moe
