// Online-FP8 output projection (LM head): logits = x W^T with W quantized to
// FP8 E4M3 when the head is created.
//
// "Three ways to speed up MoE inference on DGX Spark", section "Optimization 2":
// the bf16 head (hidden 2,560 -> 157,184 vocabulary entries) is read in full for
// every decoded token; quantizing it to FP8 when it is built halves the bytes the
// GEMV reads. Here one fp32 scale per output row (row amax / 448) and E4M3 codes
// with round-to-nearest-even and saturation; the activations stay bf16.
//
// The GEMV is bound by HBM bandwidth (1 byte of weight per multiply-add and
// token): each warp streams two rows with 16-byte loads that bypass L1, turns
// each pair of codes into an f16 pair with cvt.rn.f16x2.e4m3x2 (exact), and
// multiplies it by the f16 copy of x in shared memory with fp32-accumulating
// FMAs (the f16 x f16 product is exact in fp32); the warp's partial sums are
// added by shuffles and scaled by the row's fp32 scale.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include "moe_common.cuh"
#include "moe_internal.h"

struct moe_lmhead {
  int hidden, vocab, device, num_sms;
  uint8_t* codes;   // E4M3 [V][H]
  float* scales;    // fp32 [V]
};

namespace moe {
namespace {

constexpr int kThreads = 256;

MOE_DEV uint32_t e4m3x2_to_f16x2(uint32_t two) {   // low byte -> low half
  uint32_t r;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(r) : "r"(two));
  return r;
}
MOE_DEV uint32_t f32x2_to_e4m3x2(float lo, float hi) {  // RNE, saturating; lo -> low byte
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
MOE_DEV uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One warp per row: amax, scale = amax / 448 (IEEE division), codes of w / scale.
__global__ void __launch_bounds__(kThreads) lmhead_quantize_kernel(const uint16_t* __restrict__ w, int V, int H,
                                                                   uint8_t* __restrict__ codes,
                                                                   float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < V; row += nw) {
    const uint32_t* wr = reinterpret_cast<const uint32_t*>(w + (size_t)row * H);
    float amax = 0.f;
    for (int i = lane; i < H / 2; i += 32) {
      const uint32_t v = wr[i];
      amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(v)), fabsf(bf16_hi(v))));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = amax > 0.f ? amax / 448.f : 1.f;
    uint16_t* cr = reinterpret_cast<uint16_t*>(codes + (size_t)row * H);
    for (int i = lane; i < H / 2; i += 32) {
      const uint32_t v = wr[i];
      cr[i] = (uint16_t)f32x2_to_e4m3x2(bf16_lo(v) / s, bf16_hi(v) / s);
    }
    if (lane == 0) scales[row] = s;
  }
}

// logits[t][v] for T tokens; two rows per warp, grid-stride over row pairs.
template <int T>
__global__ void __launch_bounds__(kThreads, 4) lmhead_gemv_kernel(const uint8_t* __restrict__ codes,
                                                                  const float* __restrict__ scales,
                                                                  const uint16_t* __restrict__ x, float* __restrict__ out,
                                                                  int V, int H) {
  extern __shared__ uint32_t xs[];   // [T][H / 2] f16 pairs
  const int hp = H / 2;
  for (int i = threadIdx.x; i < T * hp; i += blockDim.x) {
    const uint32_t v = reinterpret_cast<const uint32_t*>(x)[i];
    xs[i] = f32x2_to_f16x2(bf16_lo(v), bf16_hi(v));
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), nw = gridDim.x * (blockDim.x >> 5);
  const int nch = H / 16;   // 16-byte chunks of a row
  for (int r0 = 2 * gw; r0 < V; r0 += 2 * nw) {
    const bool two = r0 + 1 < V;
    const uint8_t* p0 = codes + (size_t)r0 * H;
    const uint8_t* p1 = two ? p0 + H : p0;
    float a0[T], a1[T];
#pragma unroll
    for (int t = 0; t < T; ++t) { a0[t] = 0.f; a1[t] = 0.f; }
#pragma unroll 2
    for (int c = lane; c < nch; c += 32) {
      const uint4 w0 = ldg_stream(p0 + 16 * c), w1 = ldg_stream(p1 + 16 * c);
      const uint32_t c0[4] = {w0.x, w0.y, w0.z, w0.w}, c1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const uint4 xa = *reinterpret_cast<const uint4*>(xs + t * hp + 8 * c);
        const uint4 xb = *reinterpret_cast<const uint4*>(xs + t * hp + 8 * c + 4);
        const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {   // word k: codes 4k..4k+3 = x pairs 2k, 2k + 1
          a0[t] = fma2_f16(e4m3x2_to_f16x2(c0[k]), xw[2 * k], a0[t]);
          a0[t] = fma2_f16(e4m3x2_to_f16x2(c0[k] >> 16), xw[2 * k + 1], a0[t]);
          a1[t] = fma2_f16(e4m3x2_to_f16x2(c1[k]), xw[2 * k], a1[t]);
          a1[t] = fma2_f16(e4m3x2_to_f16x2(c1[k] >> 16), xw[2 * k + 1], a1[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        a0[t] += __shfl_xor_sync(0xFFFFFFFFu, a0[t], o);
        a1[t] += __shfl_xor_sync(0xFFFFFFFFu, a1[t], o);
      }
    }
    if (lane == 0) {
      const float s0 = scales[r0];
#pragma unroll
      for (int t = 0; t < T; ++t) out[(size_t)t * V + r0] = a0[t] * s0;
      if (two) {
        const float s1 = scales[r0 + 1];
#pragma unroll
        for (int t = 0; t < T; ++t) out[(size_t)t * V + r0 + 1] = a1[t] * s1;
      }
    }
  }
}

template <int T>
cudaError_t allow_smem_t(int hidden) {
  return cudaFuncSetAttribute(lmhead_gemv_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, T * hidden * 2);
}

template <int T>
cudaError_t launch_gemv_t(const moe_lmhead* h, const uint16_t* x, float* out, cudaStream_t s) {
  const size_t smem = (size_t)T * h->hidden * 2;
  lmhead_gemv_kernel<T><<<h->num_sms * 4, kThreads, smem, s>>>(h->codes, h->scales, x, out, h->vocab, h->hidden);
  return cudaGetLastError();
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status_t moe_lmhead_create(int32_t hidden, int32_t vocab, const void* w_dev, moe_lmhead_t** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!w_dev || hidden <= 0 || vocab <= 0) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)w_dev & 15)) return MOE_ERR_INVALID_ARG;
  if (hidden % 256 != 0 || hidden > MOE_LMHEAD_MAX_HIDDEN) return MOE_ERR_UNSUPPORTED;
  moe_lmhead* h = new (std::nothrow) moe_lmhead();
  if (!h) return MOE_ERR_OOM;
  memset(h, 0, sizeof(*h));
  h->hidden = hidden;
  h->vocab = vocab;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess) e = cudaMalloc((void**)&h->codes, (size_t)vocab * hidden);
  if (e == cudaSuccess) e = cudaMalloc((void**)&h->scales, sizeof(float) * (size_t)vocab);
  if (e == cudaSuccess) {
    moe::lmhead_quantize_kernel<<<h->num_sms * 8, moe::kThreads>>>((const uint16_t*)w_dev, vocab, hidden, h->codes,
                                                                     h->scales);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = moe::allow_smem_t<1>(hidden);
  if (e == cudaSuccess) e = moe::allow_smem_t<2>(hidden);
  if (e == cudaSuccess) e = moe::allow_smem_t<3>(hidden);
  if (e == cudaSuccess) e = moe::allow_smem_t<4>(hidden);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    const moe_status_t st = e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : moe::record_cuda_failure(e, "moe_lmhead_create");
    moe_lmhead_destroy(h);
    return st;
  }
  *out = h;
  return MOE_OK;
}

void moe_lmhead_destroy(moe_lmhead_t* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  if (h->codes) cudaFree(h->codes);
  if (h->scales) cudaFree(h->scales);
  delete h;
}

moe_status_t moe_lmhead_forward(moe_lmhead_t* h, const void* x_dev, float* logits_dev, int32_t T, void* stream) {
  if (!h || T < 0 || T > MOE_LMHEAD_MAX_T) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_dev || !logits_dev || ((uintptr_t)x_dev & 15) || ((uintptr_t)logits_dev & 3)) return MOE_ERR_INVALID_ARG;
  const uintptr_t xa = (uintptr_t)x_dev, oa = (uintptr_t)logits_dev;
  const size_t xb = (size_t)T * h->hidden * 2, ob = (size_t)T * h->vocab * 4;
  if (xa < oa + ob && oa < xa + xb) return MOE_ERR_INVALID_ARG;  // overlap
  cudaStream_t s = (cudaStream_t)stream;
  const uint16_t* x = (const uint16_t*)x_dev;
  cudaError_t e;
  switch (T) {
    case 1: e = moe::launch_gemv_t<1>(h, x, logits_dev, s); break;
    case 2: e = moe::launch_gemv_t<2>(h, x, logits_dev, s); break;
    case 3: e = moe::launch_gemv_t<3>(h, x, logits_dev, s); break;
    default: e = moe::launch_gemv_t<4>(h, x, logits_dev, s); break;
  }
  return e == cudaSuccess ? MOE_OK : moe::record_cuda_failure(e, "moe_lmhead_forward");
}

moe_status_t moe_lmhead_get_weights(moe_lmhead_t* h, void* codes_dev, float* scales_dev, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (codes_dev) e = cudaMemcpyAsync(codes_dev, h->codes, (size_t)h->vocab * h->hidden, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && scales_dev)
    e = cudaMemcpyAsync(scales_dev, h->scales, sizeof(float) * h->vocab, cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? MOE_OK : moe::record_cuda_failure(e, "moe_lmhead_get_weights");
}

}  // extern "C"
