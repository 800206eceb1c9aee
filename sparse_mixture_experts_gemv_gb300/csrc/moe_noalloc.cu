// Routing (router logits + top-k + renormalised weights) that allocates no
// device memory, for callers that cannot call cudaMalloc: code inside a host
// framework that owns all device memory through its own pool and forbids raw
// allocations, or real-time paths that must not allocate (nor risk an
// allocation failure) once they are running. The caller passes every input and
// output buffer; the only scratch
// memory (the fp32 router logits between the two kernels) is the file-scope
// device array below, which every GPU that loads this library holds until the
// process exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <mutex>

#include "moe_common.cuh"
#include "moe_layer.h"

namespace moe {
namespace {

constexpr int kNoAllocMaxT = MOE_NOALLOC_MAX_TOKENS;
constexpr int kNoAllocMaxE = MOE_NOALLOC_MAX_EXPERTS;
constexpr int kNoAllocMaxK = 8;

// Router logits [T][E] of the current call. Shared by every call of this entry
// point on the device; overwritten in full by each call before it is read.
static __device__ __align__(256) float g_noalloc_logits[kNoAllocMaxT * kNoAllocMaxE];

// Device address of g_noalloc_logits per device (host code cannot use the
// symbol's name as a device address), with the unique id of the context it was
// looked up in: after a device reset the module is loaded again, possibly at
// another address, so a new context makes the next call look the address up
// again instead of launching with a stale one.
constexpr int kMaxDevices = 64;
struct ScratchAddr {
  float* ptr;
  unsigned long long ctx_id;   // 0: unknown (look up again on every call)
};
ScratchAddr g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Driver entry points through the runtime, so that the library does not link
// libcuda directly (it still loads on machines without a driver).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (!get_current || !get_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return 0;
    get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_context_id();
  if (g_scratch[dev].ptr == nullptr || id == 0 || g_scratch[dev].ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_logits);   // also makes the device's context current
    if (e != cudaSuccess) return e;
    g_scratch[dev].ptr = static_cast<float*>(p);
    g_scratch[dev].ctx_id = current_context_id();
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

// logits[t][e] = x[t] . W_r[:, e] + bias[e] + logit_bias[t][e]; one warp per expert row
// of router_t [E][H] (fp32, expert-major).
__global__ void __launch_bounds__(256)
noalloc_router_kernel(const uint16_t* __restrict__ x, const float* __restrict__ router_t,
                      const float* __restrict__ bias, const float* __restrict__ logit_bias, int T, int H, int E,
                      float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= E) return;
  const float* row = router_t + (size_t)e * H;
  float acc[kNoAllocMaxT];
#pragma unroll
  for (int t = 0; t < kNoAllocMaxT; ++t) acc[t] = 0.f;
  for (int c = lane; c < H / 4; c += 32) {  // 4 weights (16 bytes) per step
    const float4 w = *reinterpret_cast<const float4*>(row + 4 * c);
#pragma unroll
    for (int t = 0; t < kNoAllocMaxT; ++t) {
      if (t < T) {
        const uint2 xx = *reinterpret_cast<const uint2*>(x + (size_t)t * H + 4 * c);
        float s = acc[t];
        s = fmaf(w.x, bf16_lo(xx.x), s);
        s = fmaf(w.y, bf16_hi(xx.x), s);
        s = fmaf(w.z, bf16_lo(xx.y), s);
        s = fmaf(w.w, bf16_hi(xx.y), s);
        acc[t] = s;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kNoAllocMaxT; ++t) {
    if (t < T) {
      float s = warp_sum(acc[t]);
      if (lane == 0) {
        if (bias) s += bias[e];
        if (logit_bias) s += logit_bias[(size_t)t * E + e];
        logits[(size_t)t * E + e] = s;
      }
    }
  }
}

// Top-k per token (one warp per token): exact ties go to the lower expert
// index; weights are the softmax over the k selected logits.
__global__ void __launch_bounds__(kNoAllocMaxT * 32)
noalloc_topk_kernel(const float* __restrict__ logits, int T, int E, int k, int* __restrict__ idx,
                    float* __restrict__ weights) {
  const int lane = threadIdx.x & 31, t = threadIdx.x >> 5;
  if (t >= T) return;
  constexpr int kPer = kNoAllocMaxE / 32;
  uint32_t key[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = lane + 32 * j;
    key[j] = (e < E) ? f32_order_key(logits[(size_t)t * E + e]) : 0u;
  }
  float v0 = 0.f, sum = 0.f, my_ex = 0.f;
  int my_e = 0;
  for (int r = 0; r < k; ++r) {
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
    const float val = f32_from_order_key(gmax);
    if (r == 0) v0 = val;
    const float ex = expf(val - v0);
    sum += ex;
    if (lane == r) { my_ex = ex; my_e = (int)gidx; }
  }
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    weights[(size_t)t * k + lane] = my_ex / sum;
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_topk_noalloc(const void* x_dev, const float* router_t_dev,
                                               const float* router_bias_dev, const float* logit_bias_dev, int32_t T,
                                               int32_t H, int32_t E, int32_t k, int32_t* idx_dev,
                                               float* weights_dev, void* stream) {
  if (!x_dev || !router_t_dev || !idx_dev || !weights_dev) return MOE_ERR_INVALID_ARG;
  if (T < 1 || H < 4 || H % 4 != 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)x_dev & 7) || ((uintptr_t)router_t_dev & 15)) return MOE_ERR_INVALID_ARG;
  // Sizes beyond the fixed scratch array (T * E router logits) are refused.
  if (T > moe::kNoAllocMaxT || E > moe::kNoAllocMaxE || k > moe::kNoAllocMaxK) return MOE_ERR_UNSUPPORTED;
  float* logits = nullptr;
  cudaError_t e = moe::scratch_for_current_device(&logits);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  moe::noalloc_router_kernel<<<(E + 7) / 8, 256, 0, s>>>((const uint16_t*)x_dev, router_t_dev, router_bias_dev,
                                                         logit_bias_dev, T, H, E, logits);
  e = cudaGetLastError();
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  moe::noalloc_topk_kernel<<<1, moe::kNoAllocMaxT * 32, 0, s>>>(logits, T, E, k, idx_dev, weights_dev);
  e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
