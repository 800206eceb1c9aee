// C ABI of the MoE layer: argument checks, weight repacking, workspace, path
// selection and diagnostics. The forward pass itself is in moe_decode.cu
// (weight-streaming path) and moe_grouped.cu (grouped tensor-core path).
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace {

thread_local char g_cuda_error[256] = "";

moe_status_t cuda_fail(cudaError_t e, const char* what) {
  snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
  return MOE_ERR_CUDA;
}

}  // namespace

namespace moe {
moe_status_t record_cuda_failure(cudaError_t e, const char* what) { return cuda_fail(e, what); }
}  // namespace moe

namespace {

#define MOE_CUDA(call)                                           \
  do {                                                           \
    cudaError_t e_ = (call);                                     \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);          \
  } while (0)

int64_t pad32(int64_t v) { return (v + 31) / 32 * 32; }

// Every device allocation of a layer goes through here so that a failed create
// frees exactly what it got.
struct Allocs {
  std::vector<void*> ptrs;
  int64_t bytes_total = 0;   // every byte this layer allocated on the device
  moe_status_t get(void** p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      *p = nullptr;
      return MOE_ERR_OOM;
    }
    ptrs.push_back(*p);
    bytes_total += (int64_t)bytes;
    return MOE_OK;
  }
  void free_all() {
    for (void* p : ptrs) cudaFree(p);
    ptrs.clear();
  }
};

struct LayerOwner {
  moe_layer L;
  Allocs allocs;
};

__global__ void transpose_f32_kernel(const float* __restrict__ in, float* __restrict__ out, int rows, int cols) {
  // in [rows][cols] -> out [cols][rows]
  __shared__ float tile[32][33];
  const int c = blockIdx.x * 32 + threadIdx.x;
  for (int r0 = 0; r0 < 32; r0 += 8) {
    const int r = blockIdx.y * 32 + threadIdx.y + r0;
    if (r < rows && c < cols) tile[threadIdx.y + r0][threadIdx.x] = in[(size_t)r * cols + c];
  }
  __syncthreads();
  const int orow = blockIdx.x * 32 + threadIdx.y;  // output row = input column
  const int ocol = blockIdx.y * 32 + threadIdx.x;
  for (int r0 = 0; r0 < 32; r0 += 8) {
    if (orow + r0 < cols && ocol < rows) out[(size_t)(orow + r0) * rows + ocol] = tile[threadIdx.x][threadIdx.y + r0];
  }
}

// W = hi + mid + lo exactly, each term bf16 (8 significant bits each cover the
// 24-bit fp32 significand; every step is an exact fp32 subtraction).
__global__ void split3_bf16_kernel(const float* __restrict__ w, uint16_t* __restrict__ out, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = w[i];
    const uint16_t hi = moe::f32_to_bf16_rne(v);
    const float r1 = v - __uint_as_float((uint32_t)hi << 16);
    const uint16_t mid = moe::f32_to_bf16_rne(r1);
    const float r2 = r1 - __uint_as_float((uint32_t)mid << 16);
    const uint16_t lo = moe::f32_to_bf16_rne(r2);
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = lo;
  }
}

// down [E][H][I] -> the down column of each record: element n of the third
// H-row of record (e, i) (records `stride` bytes apart) = down[e][n][i].
__global__ void down_to_columns_kernel(const uint16_t* __restrict__ down, uint8_t* __restrict__ rec, int H, int I,
                                       int stride) {
  __shared__ uint16_t tile[32][33];
  const size_t e = blockIdx.z;
  const int i = blockIdx.x * 32 + threadIdx.x;
  for (int r0 = 0; r0 < 32; r0 += 8) {
    const int n = blockIdx.y * 32 + threadIdx.y + r0;
    if (n < H && i < I) tile[threadIdx.y + r0][threadIdx.x] = down[(e * H + n) * I + i];
  }
  __syncthreads();
  const int n = blockIdx.y * 32 + threadIdx.x;
  for (int r0 = 0; r0 < 32; r0 += 8) {
    const int io = blockIdx.x * 32 + threadIdx.y + r0;
    if (io < I && n < H)
      reinterpret_cast<uint16_t*>(rec + (e * I + io) * (size_t)stride + 4 * (size_t)H)[n] = tile[threadIdx.x][threadIdx.y + r0];
  }
}

// MXFP4 down codes [E][H][I/2] (element (n, i) in nibble i & 1 of byte i / 2 of
// row n) -> the down columns of each pair of records (features 2p, 2p + 1) in
// 16-row tiles. Byte i / 2 of row n already holds both features' codes for
// that row (feature 2p in the low nibble), which is the code pair one lane of
// an m16n8k16 A fragment needs (k = 2c, 2c + 1). For tile t (rows 16t ..
// 16t + 15) and g < 8, bytes 2g and 2g + 1 of the tile's 16 are rows 16t + g
// and 16t + g + 8; the first H / 32 tiles of the pair sit in record 2p's column,
// the rest in record 2p + 1's (each record keeps H / 2 bytes).
// One block: 64 features (32 pairs) x 64 rows.
__global__ void mx_down_to_columns_kernel(const uint8_t* __restrict__ down, uint8_t* __restrict__ rec, int H, int I,
                                          int stride, int col_off) {
  __shared__ uint8_t tile[64][32];            // [row n][pair]
  const size_t e = blockIdx.z;
  const int i0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
  const int t = threadIdx.x;
  {
    const int n = t >> 2, part = t & 3;
    *reinterpret_cast<uint2*>(&tile[n][8 * part]) =
        *reinterpret_cast<const uint2*>(down + (e * H + n0 + n) * (size_t)(I / 2) + i0 / 2 + 8 * part);
  }
  __syncthreads();
  {
    const int pl = t >> 3, part = (t >> 1) & 3, h = t & 1;   // pair, 16-row tile of the block, half of its bytes
    const int tile_abs = n0 / 16 + part, half_tiles = H / 32;
    const int sel = tile_abs >= half_tiles ? 1 : 0;
    uint8_t o[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {               // g = 4h + q: rows 16 part + g and 16 part + g + 8
      o[2 * q] = tile[16 * part + 4 * h + q][pl];
      o[2 * q + 1] = tile[16 * part + 4 * h + q + 8][pl];
    }
    uint8_t* dst = rec + (e * I + i0 + 2 * pl + sel) * (size_t)stride + col_off +
                   16 * (tile_abs - sel * half_tiles) + 8 * h;
    *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(o);
  }
}

// MXFP4 gate or up codes [rows][H/2] -> the records, each 16-byte block (32
// elements) shuffled for the tensor-core fragments: stored byte 4c + m = source
// byte c + 4m.
__global__ void mx_shuffle_codes_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ rec, size_t rows, int H,
                                        int stride, int dst_off) {
  const int nb = H / 32;
  const size_t total = rows * nb;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < total; q += (size_t)gridDim.x * blockDim.x) {
    const size_t row = q / nb, blk = q % nb;
    const uint4 v = *reinterpret_cast<const uint4*>(src + row * (size_t)(H / 2) + 16 * blk);
    const uint8_t* in = reinterpret_cast<const uint8_t*>(&v);
    uint8_t o[16];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int m = 0; m < 4; ++m) o[4 * c + m] = in[c + 4 * m];
    *reinterpret_cast<uint4*>(rec + row * (size_t)stride + dst_off + 16 * blk) = *reinterpret_cast<const uint4*>(o);
  }
}

// MXFP4 down scales [E][H][I/32] -> [E][I/32][H] (one vector per 32 features).
__global__ void mx_down_scales_kernel(const uint8_t* __restrict__ ds, uint8_t* __restrict__ out, int E, int H,
                                      int nblk) {
  const size_t total = (size_t)E * nblk * H;
  for (size_t o = blockIdx.x * (size_t)blockDim.x + threadIdx.x; o < total; o += (size_t)gridDim.x * blockDim.x) {
    const size_t n = o % H, eb = o / H, blk = eb % nblk, e = eb / nblk;
    out[o] = ds[(e * H + n) * nblk + blk];
  }
}

// Groupwise affine int4 down (scale, bias) pairs [E][H][I/64] -> one vector of H
// pairs per (expert, 64 features): out[e][blk][n] = scale | bias << 16.
__global__ void i4_down_vectors_kernel(const uint16_t* __restrict__ scales, const uint16_t* __restrict__ biases,
                                       uint32_t* __restrict__ out, int E, int H, int nblk) {
  const size_t total = (size_t)E * nblk * H;
  for (size_t o = blockIdx.x * (size_t)blockDim.x + threadIdx.x; o < total; o += (size_t)gridDim.x * blockDim.x) {
    const size_t n = o % H, eb = o / H, blk = eb % nblk, e = eb / nblk;
    const size_t q = (e * H + n) * nblk + blk;
    out[o] = (uint32_t)scales[q] | ((uint32_t)biases[q] << 16);
  }
}

// Groupwise affine int4: the (scale, bias) bf16 pair of group g of each row goes
// to bytes [off + 4g, off + 4g + 4) of the row's record (scale first).
__global__ void i4_group_params_kernel(const uint16_t* __restrict__ scales, const uint16_t* __restrict__ biases,
                                       uint8_t* __restrict__ rec, size_t rows, int ngroups, int64_t rb, int64_t off) {
  const size_t total = rows * ngroups;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < total; q += (size_t)gridDim.x * blockDim.x) {
    const size_t row = q / ngroups, g = q % ngroups;
    *reinterpret_cast<uint32_t*>(rec + row * rb + off + 4 * g) = (uint32_t)scales[q] | ((uint32_t)biases[q] << 16);
  }
}

moe_status_t validate(const moe_layer_config_t* c, const moe_layer_weights_t* w) {
  if (!c || !w) return MOE_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->num_experts <= 0 || c->top_k <= 0 || c->intermediate <= 0 ||
      c->shared_intermediate < 0 || c->max_tokens <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->num_experts) return MOE_ERR_INVALID_ARG;
  if (c->weight_format != MOE_WEIGHTS_BF16 && c->weight_format != MOE_WEIGHTS_MXFP4 &&
      c->weight_format != MOE_WEIGHTS_INT4)
    return MOE_ERR_INVALID_ARG;
  if (c->flags & ~(uint32_t)(MOE_FLAG_FORCE_GROUPED | MOE_FLAG_ONE_WEIGHT_COPY | MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT))
    return MOE_ERR_INVALID_ARG;
  if (c->hidden % 256 != 0 || c->hidden > 8192) return MOE_ERR_UNSUPPORTED;
  if (c->intermediate % 128 != 0 || c->intermediate > 4096) return MOE_ERR_UNSUPPORTED;
  if (c->shared_intermediate % 128 != 0 || c->shared_intermediate > 4096) return MOE_ERR_UNSUPPORTED;
  if (c->num_experts > moe::kMaxExperts || c->top_k > moe::kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (c->max_tokens > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  if (!w->router_dev || !w->gate_dev || !w->up_dev || !w->down_dev) return MOE_ERR_INVALID_ARG;
  if (c->shared_intermediate > 0 && (!w->shared_gate_dev || !w->shared_up_dev || !w->shared_down_dev))
    return MOE_ERR_INVALID_ARG;
  if (c->weight_format != MOE_WEIGHTS_BF16 &&
      (!w->gate_scales_dev || !w->up_scales_dev || !w->down_scales_dev))
    return MOE_ERR_INVALID_ARG;
  if (c->weight_format == MOE_WEIGHTS_INT4 &&
      (!w->gate_biases_dev || !w->up_biases_dev || !w->down_biases_dev))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t alloc_workspace(LayerOwner* o) {
  moe_layer& L = o->L;
  const auto& c = L.cfg;
  const int T8 = moe::kMaxDecodeT;
  moe_status_t st;
#define GET(ptr, bytes) \
  if ((st = o->allocs.get((void**)&(ptr), (bytes))) != MOE_OK) return st
  GET(L.dec.logits, sizeof(float) * T8 * c.num_experts);
  GET(L.dec.idx, sizeof(int) * T8 * c.top_k);
  GET(L.dec.weights, sizeof(float) * T8 * c.top_k);
  GET(L.dec.meta, sizeof(moe::DecodeMeta));
  GET(L.dec.h, sizeof(float) * (size_t)T8 * c.top_k * c.intermediate);
  GET(L.dec.h_shared, sizeof(float) * (size_t)T8 * std::max(c.shared_intermediate, 1));
  GET(L.dec.sync_ctr, sizeof(unsigned long long) * 4);
  GET(L.dec.logit_words, sizeof(unsigned long long) * T8 * c.num_experts);
  GET(L.dec.partial, sizeof(unsigned long long) * (size_t)L.num_sms * T8 * c.hidden);
  GET(L.err, sizeof(int) * 4);
  GET(L.never_set, sizeof(int));
  GET(L.x_stage, sizeof(uint16_t) * (size_t)c.max_tokens * c.hidden);
  GET(L.out_stage, sizeof(uint16_t) * (size_t)c.max_tokens * c.hidden);
  GET(L.bias_stage, sizeof(float) * (size_t)c.max_tokens * c.num_experts);
#undef GET
  cudaMemset(L.dec.sync_ctr, 0, sizeof(unsigned long long) * 4);
  cudaMemset(L.dec.logit_words, 0, sizeof(unsigned long long) * T8 * c.num_experts);
  cudaMemset(L.dec.partial, 0, sizeof(unsigned long long) * (size_t)L.num_sms * T8 * c.hidden);
  cudaMemset(L.err, 0, sizeof(int) * 4);
  cudaMemset(L.never_set, 0, sizeof(int));
  cudaMemset(L.dec.meta, 0, sizeof(moe::DecodeMeta));
  L.mem_workspace_bytes += o->allocs.bytes_total;   // the layer's first allocations
  return MOE_OK;
}

moe_status_t repack(LayerOwner* o, const moe_layer_weights_t* w) {
  moe_layer& L = o->L;
  const auto& c = L.cfg;
  const int64_t H = c.hidden, E = c.num_experts, I = c.intermediate, Is = c.shared_intermediate;
  const int64_t mem0 = o->allocs.bytes_total;
  moe_status_t st;
#define GET(ptr, bytes) \
  if ((st = o->allocs.get((void**)&(ptr), (bytes))) != MOE_OK) return st

  // Router: transpose to one contiguous fp32 row per expert, plus the exact
  // three-term bf16 split used by the grouped path's tensor-core router.
  GET(L.router_t, sizeof(float) * H * E);
  GET(L.router_bias, sizeof(float) * E);
  GET(L.router_split, sizeof(uint16_t) * 3 * H * E);
  {
    dim3 block(32, 8), grid((unsigned)((E + 31) / 32), (unsigned)((H + 31) / 32));
    transpose_f32_kernel<<<grid, block>>>(w->router_dev, L.router_t, (int)H, (int)E);
    MOE_CUDA(cudaGetLastError());
    split3_bf16_kernel<<<256, 256>>>(L.router_t, L.router_split, (size_t)H * E);
    MOE_CUDA(cudaGetLastError());
  }
  if (w->router_bias_dev)
    MOE_CUDA(cudaMemcpy(L.router_bias, w->router_bias_dev, sizeof(float) * E, cudaMemcpyDeviceToDevice));
  else
    MOE_CUDA(cudaMemset(L.router_bias, 0, sizeof(float) * E));

  // With MOE_FLAG_ONE_WEIGHT_COPY, bf16 layers the record-streaming kernel
  // serves keep one copy of the expert weights: the feature records below,
  // which the grouped GEMMs then read too (gate/up rows K-major, down columns
  // MN-major). Otherwise the row layouts of the three-phase decode kernel and
  // the grouped GEMMs are kept as well (the grouped down GEMM is faster on them).
  const bool records_only = (c.flags & MOE_FLAG_ONE_WEIGHT_COPY) && c.weight_format == MOE_WEIGHTS_BF16 &&
                            H <= moe::kStreamMaxHidden;
  L.row_bytes.gu = c.weight_format == MOE_WEIGHTS_BF16 ? H * 2 : 0;
  L.row_bytes.down = c.weight_format == MOE_WEIGHTS_BF16 ? I * 2 : 0;

  // Routed experts: gate row i and up row i adjacent ([E][I][2][row]).
  if (records_only) {
    // no row layouts
  } else if (c.weight_format == MOE_WEIGHTS_BF16) {
    L.row_bytes.gu = H * 2;
    L.row_bytes.down = I * 2;
    GET(L.w_gu, (size_t)E * I * 2 * L.row_bytes.gu);
    GET(L.w_down, (size_t)E * H * L.row_bytes.down);
    const size_t row = (size_t)H * 2;
    MOE_CUDA(cudaMemcpy2D(L.w_gu, 2 * row, w->gate_dev, row, row, (size_t)E * I, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D(L.w_gu + row, 2 * row, w->up_dev, row, row, (size_t)E * I, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy(L.w_down, w->down_dev, (size_t)E * H * I * 2, cudaMemcpyDeviceToDevice));
  } else if (c.weight_format == MOE_WEIGHTS_INT4) {
    // One record per row: codes (K/2 bytes) then (scale, bias) bf16 pairs of the
    // K/64 groups (4 bytes each); rows padded to 32 bytes so that every row, and
    // every 32-byte code chunk the grouped GEMMs load, starts on a DRAM sector.
    L.row_bytes.gu = pad32(H / 2 + H / 16);
    L.row_bytes.down = pad32(I / 2 + I / 16);
    GET(L.w_gu, (size_t)E * I * 2 * L.row_bytes.gu);
    GET(L.w_down, (size_t)E * H * L.row_bytes.down);
    MOE_CUDA(cudaMemset(L.w_gu, 0, (size_t)E * I * 2 * L.row_bytes.gu));
    MOE_CUDA(cudaMemset(L.w_down, 0, (size_t)E * H * L.row_bytes.down));
    const size_t rg = (size_t)L.row_bytes.gu, rd = (size_t)L.row_bytes.down;
    const size_t rows_gu = (size_t)E * I, rows_d = (size_t)E * H;
    MOE_CUDA(cudaMemcpy2D(L.w_gu, 2 * rg, w->gate_dev, H / 2, H / 2, rows_gu, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D(L.w_gu + rg, 2 * rg, w->up_dev, H / 2, H / 2, rows_gu, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D(L.w_down, rd, w->down_dev, I / 2, I / 2, rows_d, cudaMemcpyDeviceToDevice));
    // gate rows are records 2i, up rows 2i + 1 (stride 2 * rg from the first of each)
    i4_group_params_kernel<<<1024, 256>>>((const uint16_t*)w->gate_scales_dev, (const uint16_t*)w->gate_biases_dev,
                                          L.w_gu, rows_gu, (int)(H / 64), (int64_t)(2 * rg), H / 2);
    MOE_CUDA(cudaGetLastError());
    i4_group_params_kernel<<<1024, 256>>>((const uint16_t*)w->up_scales_dev, (const uint16_t*)w->up_biases_dev,
                                          L.w_gu + rg, rows_gu, (int)(H / 64), (int64_t)(2 * rg), H / 2);
    MOE_CUDA(cudaGetLastError());
    i4_group_params_kernel<<<1024, 256>>>((const uint16_t*)w->down_scales_dev, (const uint16_t*)w->down_biases_dev,
                                          L.w_down, rows_d, (int)(I / 64), (int64_t)rd, I / 2);
    MOE_CUDA(cudaGetLastError());
  } else {
    // One record per row: codes (K/2 bytes) then scales (K/32 bytes); rows padded
    // to 32 bytes (sector-aligned code chunks, as for int4).
    L.row_bytes.gu = pad32(H / 2 + H / 32);
    L.row_bytes.down = pad32(I / 2 + I / 32);
    GET(L.w_gu, (size_t)E * I * 2 * L.row_bytes.gu);
    GET(L.w_down, (size_t)E * H * L.row_bytes.down);
    MOE_CUDA(cudaMemset(L.w_gu, 0, (size_t)E * I * 2 * L.row_bytes.gu));
    MOE_CUDA(cudaMemset(L.w_down, 0, (size_t)E * H * L.row_bytes.down));
    const size_t rg = (size_t)L.row_bytes.gu, rd = (size_t)L.row_bytes.down;
    const size_t rows_gu = (size_t)E * I, rows_d = (size_t)E * H;
    MOE_CUDA(cudaMemcpy2D(L.w_gu, 2 * rg, w->gate_dev, H / 2, H / 2, rows_gu, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D(L.w_gu + H / 2, 2 * rg, w->gate_scales_dev, H / 32, H / 32, rows_gu, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D(L.w_gu + rg, 2 * rg, w->up_dev, H / 2, H / 2, rows_gu, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D(L.w_gu + rg + H / 2, 2 * rg, w->up_scales_dev, H / 32, H / 32, rows_gu, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D(L.w_down, rd, w->down_dev, I / 2, I / 2, rows_d, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D(L.w_down + I / 2, rd, w->down_scales_dev, I / 32, I / 32, rows_d, cudaMemcpyDeviceToDevice));
  }

  // Shared expert (bf16): [Is][2][H] and [H][Is].
  if (!records_only) {
    GET(L.ws_gu, sizeof(uint16_t) * std::max<int64_t>(Is, 1) * 2 * H);
    GET(L.ws_down, sizeof(uint16_t) * std::max<int64_t>(Is, 1) * H);
  }
  if (Is > 0 && !records_only) {
    const size_t row = (size_t)H * 2;
    MOE_CUDA(cudaMemcpy2D(L.ws_gu, 2 * row, w->shared_gate_dev, row, row, (size_t)Is, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy2D((uint8_t*)L.ws_gu + row, 2 * row, w->shared_up_dev, row, row, (size_t)Is, cudaMemcpyDeviceToDevice));
    MOE_CUDA(cudaMemcpy(L.ws_down, w->shared_down_dev, (size_t)H * Is * 2, cudaMemcpyDeviceToDevice));
  }

  // Feature records for the record-streaming decode kernel: per (expert, i)
  // the gate row, the up row and the down column, contiguous (6H bytes).
  const bool bf16_stream = c.weight_format == MOE_WEIGHTS_BF16 && H <= moe::kStreamMaxHidden;
  const bool mx_stream = c.weight_format == MOE_WEIGHTS_MXFP4 && H <= moe::kStreamMxMaxHidden && H % 512 == 0;
  const bool i4_stream = c.weight_format == MOE_WEIGHTS_INT4 && H <= moe::kStreamMxMaxHidden && H % 512 == 0 &&
                         I % 64 == 0;
  if (bf16_stream || mx_stream || i4_stream) {
    const size_t row = (size_t)H * 2, rec = (size_t)moe::stream_record_stride((int)H);
    dim3 block(32, 8);
    if (bf16_stream) {
      GET(L.w_rec, (size_t)E * I * rec);
      MOE_CUDA(cudaMemset(L.w_rec, 0, (size_t)E * I * rec));
      MOE_CUDA(cudaMemcpy2D(L.w_rec, rec, w->gate_dev, row, row, (size_t)E * I, cudaMemcpyDeviceToDevice));
      MOE_CUDA(cudaMemcpy2D(L.w_rec + row, rec, w->up_dev, row, row, (size_t)E * I, cudaMemcpyDeviceToDevice));
      dim3 grid((unsigned)((I + 31) / 32), (unsigned)((H + 31) / 32), (unsigned)E);
      down_to_columns_kernel<<<grid, block>>>((const uint16_t*)w->down_dev, L.w_rec, (int)H, (int)I, (int)rec);
      MOE_CUDA(cudaGetLastError());
    } else if (i4_stream) {
      // int4 records: gate codes | up codes (block-shuffled as for MXFP4) | gate
      // (s, b) pairs | up (s, b) pairs (one 4-byte pair per 64 elements, padded
      // to 16) | down column codes; down pairs apart, one vector per (e, 64 features)
      const size_t i4s = (size_t)moe::stream_i4_record_stride((int)H);
      const size_t so = (size_t)((H / 16 + 15) / 16 * 16), nblk = (size_t)I / 64;
      const size_t rows = (size_t)E * I;
      GET(L.w_mx, rows * i4s);
      GET(L.mx_dsc, (size_t)E * nblk * H * 4);
      MOE_CUDA(cudaMemset(L.w_mx, 0, rows * i4s));
      mx_shuffle_codes_kernel<<<1024, 256>>>((const uint8_t*)w->gate_dev, L.w_mx, rows, (int)H, (int)i4s, 0);
      MOE_CUDA(cudaGetLastError());
      mx_shuffle_codes_kernel<<<1024, 256>>>((const uint8_t*)w->up_dev, L.w_mx, rows, (int)H, (int)i4s, (int)(H / 2));
      MOE_CUDA(cudaGetLastError());
      i4_group_params_kernel<<<1024, 256>>>((const uint16_t*)w->gate_scales_dev, (const uint16_t*)w->gate_biases_dev,
                                            L.w_mx, rows, (int)(H / 64), (int64_t)i4s, H);
      MOE_CUDA(cudaGetLastError());
      i4_group_params_kernel<<<1024, 256>>>((const uint16_t*)w->up_scales_dev, (const uint16_t*)w->up_biases_dev,
                                            L.w_mx, rows, (int)(H / 64), (int64_t)i4s, (int64_t)(H + so));
      MOE_CUDA(cudaGetLastError());
      dim3 g2((unsigned)(I / 64), (unsigned)(H / 64), (unsigned)E);
      mx_down_to_columns_kernel<<<g2, 256>>>((const uint8_t*)w->down_dev, L.w_mx, (int)H, (int)I, (int)i4s,
                                             (int)(H + 2 * so));
      MOE_CUDA(cudaGetLastError());
      i4_down_vectors_kernel<<<1024, 256>>>((const uint16_t*)w->down_scales_dev, (const uint16_t*)w->down_biases_dev,
                                            reinterpret_cast<uint32_t*>(L.mx_dsc), (int)E, (int)H, (int)nblk);
      MOE_CUDA(cudaGetLastError());
    } else {
      // MXFP4 records: gate codes | up codes | gate scales | up scales | down column codes
      const size_t mxs = (size_t)moe::stream_mx_record_stride((int)H);
      const size_t so = (size_t)((H / 32 + 15) / 16 * 16), nblk = (size_t)I / 32;
      GET(L.w_mx, (size_t)E * I * mxs);
      GET(L.mx_dsc, (size_t)E * nblk * H);
      MOE_CUDA(cudaMemset(L.w_mx, 0, (size_t)E * I * mxs));
      const size_t rows = (size_t)E * I;
      mx_shuffle_codes_kernel<<<1024, 256>>>((const uint8_t*)w->gate_dev, L.w_mx, rows, (int)H, (int)mxs, 0);
      MOE_CUDA(cudaGetLastError());
      mx_shuffle_codes_kernel<<<1024, 256>>>((const uint8_t*)w->up_dev, L.w_mx, rows, (int)H, (int)mxs, (int)(H / 2));
      MOE_CUDA(cudaGetLastError());
      MOE_CUDA(cudaMemcpy2D(L.w_mx + H, mxs, w->gate_scales_dev, H / 32, H / 32, rows, cudaMemcpyDeviceToDevice));
      MOE_CUDA(cudaMemcpy2D(L.w_mx + H + so, mxs, w->up_scales_dev, H / 32, H / 32, rows, cudaMemcpyDeviceToDevice));
      dim3 g2((unsigned)(I / 64), (unsigned)(H / 64), (unsigned)E);
      mx_down_to_columns_kernel<<<g2, 256>>>((const uint8_t*)w->down_dev, L.w_mx, (int)H, (int)I, (int)mxs,
                                             (int)(H + 2 * so));
      MOE_CUDA(cudaGetLastError());
      mx_down_scales_kernel<<<1024, 256>>>(w->down_scales_dev, L.mx_dsc, (int)E, (int)H, (int)nblk);
      MOE_CUDA(cudaGetLastError());
    }
    GET(L.ws_rec, std::max<int64_t>(Is, 1) * rec);
    MOE_CUDA(cudaMemset(L.ws_rec, 0, std::max<int64_t>(Is, 1) * rec));
    if (Is > 0) {
      MOE_CUDA(cudaMemcpy2D(L.ws_rec, rec, w->shared_gate_dev, row, row, (size_t)Is, cudaMemcpyDeviceToDevice));
      MOE_CUDA(cudaMemcpy2D(L.ws_rec + row, rec, w->shared_up_dev, row, row, (size_t)Is, cudaMemcpyDeviceToDevice));
      dim3 g1((unsigned)((Is + 31) / 32), (unsigned)((H + 31) / 32), 1u);
      down_to_columns_kernel<<<g1, block>>>((const uint16_t*)w->shared_down_dev, L.ws_rec, (int)H, (int)Is, (int)rec);
      MOE_CUDA(cudaGetLastError());
    }
  }
#undef GET
  L.mem_weight_bytes += o->allocs.bytes_total - mem0;
  return MOE_OK;
}

void destroy_owner(LayerOwner* o) {
  if (!o) return;
  cudaDeviceSynchronize();
  if (o->L.profile)
    for (int i = 0; i < 8; ++i) cudaEventDestroy(o->L.prof_ev[i]);
  moe::grouped_release(&o->L);
  o->allocs.free_all();
  delete o;
}

moe_status_t check_forward_args(moe_layer* L, const void* x, void* out, int32_t T) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)x & 15) || ((uintptr_t)out & 15)) return MOE_ERR_INVALID_ARG;
  const size_t bytes = (size_t)T * L->cfg.hidden * 2;
  const uintptr_t xa = (uintptr_t)x, oa = (uintptr_t)out;
  if (xa < oa + bytes && oa < xa + bytes) return MOE_ERR_INVALID_ARG;  // overlap
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_layer_create(const moe_layer_config_t* cfg, const moe_layer_weights_t* w, moe_layer_t** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status_t st = validate(cfg, w);
  if (st != MOE_OK) return st;

  LayerOwner* o = new (std::nothrow) LayerOwner();
  if (!o) return MOE_ERR_OOM;
  memset(&o->L, 0, sizeof(o->L));
  moe_layer& L = o->L;
  L.cfg = *cfg;
  cudaError_t e = cudaGetDevice(&L.device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L.num_sms, cudaDevAttrMultiProcessorCount, L.device);
  if (e != cudaSuccess) {
    delete o;
    return cuda_fail(e, "cudaGetDevice");
  }
  // Largest T whose SwiGLU outputs fit the down kernel's shared memory.
  L.decode_max_t = 0;
  for (int t = moe::kMaxDecodeT; t >= 1; --t) {
    if (moe::decode_smem_bytes_down(&L, t) <= 200 * 1024) { L.decode_max_t = t; break; }
  }

  if ((st = alloc_workspace(o)) != MOE_OK || (st = repack(o, w)) != MOE_OK) {
    destroy_owner(o);
    return st;
  }
  e = moe::decode_prepare(&L);
  if (e == cudaSuccess) e = moe::stream_prepare(&L);
  if (e == cudaSuccess) e = moe::stream_mx_prepare(&L);
  if (e == cudaSuccess) e = moe::grouped_prepare(&L);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    st = (e == cudaErrorMemoryAllocation) ? MOE_ERR_OOM : cuda_fail(e, "moe_layer_create");
    destroy_owner(o);
    return st;
  }
  snprintf(L.describe, sizeof(L.describe),
           "moe_layer H=%d E=%d k=%d I=%d Is=%d format=%s max_tokens=%d | "
           "T<=%d: decode GEMV path [%s] | "
           "T>%d: grouped path [grouped_router_tc, dispatch, grouped_gateup_tc (tcgen05%s), grouped_down_tc (tcgen05%s), "
           "combine]%s",
           cfg->hidden, cfg->num_experts, cfg->top_k, cfg->intermediate, cfg->shared_intermediate,
           cfg->weight_format == MOE_WEIGHTS_MXFP4 ? "mxfp4" : cfg->weight_format == MOE_WEIGHTS_INT4 ? "int4" : "bf16",
           cfg->max_tokens,
           (cfg->flags & MOE_FLAG_FORCE_GROUPED) ? 0 : L.decode_max_t,
           moe::stream_supported(&L, 1)
               ? "moe_decode_stream_kernel (cooperative: router with tagged logits, per-CTA top-k, bulk-copied "
                 "[gate|up|down column] records of the shared and routed experts with the down projection fused, "
                 "fp32 partial-output exchange)"
               : moe::stream_mx_supported(&L, 1)
               ? (cfg->weight_format == MOE_WEIGHTS_INT4
                      ? "moe_decode_stream_mx_kernel<int4> (cooperative: router with tagged logits, per-CTA top-k, "
                        "bulk-copied int4 [gate|up|down column] records as exact f16 integers on the tensor cores, "
                        "s * sum(q x) + b * sum(x) per group, bf16 shared-expert records, fp32 partial-output exchange)"
                      : "moe_decode_stream_mx_kernel (cooperative: router with tagged logits, per-CTA top-k, "
                        "bulk-copied MXFP4 [gate|up|down column] records decoded in registers, bf16 shared-expert "
                        "records, fp32 partial-output exchange)")
               : (cfg->weight_format == MOE_WEIGHTS_MXFP4
                      ? "moe_decode_fused_kernel<mxfp4> (cooperative: router+shared, routed gate/up, down+combine)"
                      : cfg->weight_format == MOE_WEIGHTS_INT4
                      ? "moe_decode_fused_kernel<int4> (cooperative: router+shared, routed gate/up, down+combine; "
                        "per group s * sum(q x) + b * sum(x))"
                      : "moe_decode_fused_kernel<bf16> (cooperative: router+shared, routed gate/up, down+combine)"),
           (cfg->flags & MOE_FLAG_FORCE_GROUPED) ? 0 : L.decode_max_t,
           cfg->weight_format == MOE_WEIGHTS_MXFP4 ? ", MXFP4 B rows decoded to f16 in the kernel"
           : cfg->weight_format == MOE_WEIGHTS_INT4 ? ", int4 B rows decoded to f16 in the kernel" : "",
           cfg->weight_format == MOE_WEIGHTS_MXFP4 ? ", MXFP4 B rows decoded to f16 in the kernel"
           : cfg->weight_format == MOE_WEIGHTS_INT4 ? ", int4 B rows decoded to f16 in the kernel" : "",
           (cfg->flags & MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT) ? " [test: forced wait timeout]" : "");
  if (!L.w_gu && L.w_rec) {   // one copy of the weights: say so
    const size_t n = strlen(L.describe);
    snprintf(L.describe + n, sizeof(L.describe) - n, " [one weight copy: grouped GEMMs read the feature records]");
  }
  *out = &o->L;
  return MOE_OK;
}

void moe_layer_destroy(moe_layer_t* layer) {
  if (!layer) return;
  destroy_owner(reinterpret_cast<LayerOwner*>(reinterpret_cast<char*>(layer) - offsetof(LayerOwner, L)));
}

moe_status_t moe_layer_forward_ex(moe_layer_t* L, const void* x, void* out, int32_t T,
                                  const float* logit_bias, void* stream) {
  moe_status_t st = check_forward_args(L, x, out, T);
  if (st != MOE_OK || T == 0) return st;
  if (logit_bias && ((uintptr_t)logit_bias & 3)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const bool grouped = (L->cfg.flags & MOE_FLAG_FORCE_GROUPED) || T > L->decode_max_t;
  // The grouped path's router takes E in multiples of 16.
  if (grouped && L->cfg.num_experts % 16 != 0) return MOE_ERR_UNSUPPORTED;
  L->prof_n = 0;
  cudaError_t e = grouped ? moe::launch_grouped(L, (const uint16_t*)x, (uint16_t*)out, T, logit_bias, s)
                          : moe::launch_decode(L, (const uint16_t*)x, (uint16_t*)out, T, logit_bias, s);
  if (e != cudaSuccess) return cuda_fail(e, grouped ? "launch_grouped" : "launch_decode");
  L->last_path = grouped ? MOE_PATH_GROUPED : MOE_PATH_DECODE_GEMV;
  L->last_T = T;
  L->last_logit_bias = logit_bias;
  return MOE_OK;
}

moe_status_t moe_layer_forward_chunked(moe_layer_t* L, const void* x, void* out, int32_t T, int32_t chunk,
                                       const float* logit_bias, void* stream) {
  if (!L || T < 0) return MOE_ERR_INVALID_ARG;
  if (chunk == 0) chunk = L->cfg.max_tokens;
  if (chunk < 1 || chunk > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || ((uintptr_t)x & 15) || ((uintptr_t)out & 15)) return MOE_ERR_INVALID_ARG;
  if (logit_bias && ((uintptr_t)logit_bias & 3)) return MOE_ERR_INVALID_ARG;
  const size_t H = (size_t)L->cfg.hidden, E = (size_t)L->cfg.num_experts;
  const size_t bytes = (size_t)T * H * 2;
  const uintptr_t xa = (uintptr_t)x, oa = (uintptr_t)out;
  if (xa < oa + bytes && oa < xa + bytes) return MOE_ERR_INVALID_ARG;  // overlap
  if (L->cfg.num_experts % 16 != 0) return MOE_ERR_UNSUPPORTED;        // grouped router tiles
  cudaStream_t s = (cudaStream_t)stream;
  L->prof_n = 0;
  for (int32_t t0 = 0; t0 < T; t0 += chunk) {
    const int32_t n = T - t0 < chunk ? T - t0 : chunk;
    const uint16_t* xc = (const uint16_t*)x + (size_t)t0 * H;   // H % 256 == 0: chunks stay 16-byte aligned
    uint16_t* oc = (uint16_t*)out + (size_t)t0 * H;
    const float* lb = logit_bias ? logit_bias + (size_t)t0 * E : nullptr;
    if (L->profile) L->prof_n = 0;  // stage timings describe the last chunk
    cudaError_t e = moe::launch_grouped(L, xc, oc, n, lb, s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_layer_forward_chunked");
    L->last_path = MOE_PATH_GROUPED;
    L->last_T = n;
    L->last_logit_bias = lb;
  }
  return MOE_OK;
}

moe_status_t moe_layer_forward(moe_layer_t* L, const void* x, void* out, int32_t T, void* stream) {
  return moe_layer_forward_ex(L, x, out, T, nullptr, stream);
}

moe_status_t moe_layer_forward_host(moe_layer_t* L, const void* x_host, void* out_host, int32_t T,
                                    const float* logit_bias_host, void* stream) {
  if (!L || T < 0 || T > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t bytes = (size_t)T * L->cfg.hidden * 2;
  MOE_CUDA(cudaMemcpyAsync(L->x_stage, x_host, bytes, cudaMemcpyHostToDevice, s));
  const float* lb = nullptr;
  if (logit_bias_host) {
    MOE_CUDA(cudaMemcpyAsync(L->bias_stage, logit_bias_host, sizeof(float) * (size_t)T * L->cfg.num_experts,
                             cudaMemcpyHostToDevice, s));
    lb = L->bias_stage;
  }
  moe_status_t st = moe_layer_forward_ex(L, L->x_stage, L->out_stage, T, lb, stream);
  if (st != MOE_OK) return st;
  MOE_CUDA(cudaMemcpyAsync(out_host, L->out_stage, bytes, cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  return MOE_OK;
}

moe_status_t moe_layer_get_routing(moe_layer_t* L, int32_t* idx, float* w, void* stream) {
  if (!L || L->last_path == MOE_PATH_NONE) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t n = (size_t)L->last_T * L->cfg.top_k;
  const int* src_idx = L->last_path == MOE_PATH_GROUPED ? L->grp.idx : L->dec.idx;
  const float* src_w = L->last_path == MOE_PATH_GROUPED ? L->grp.weights : L->dec.weights;
  if (idx) MOE_CUDA(cudaMemcpyAsync(idx, src_idx, n * sizeof(int), cudaMemcpyDeviceToDevice, s));
  if (w) MOE_CUDA(cudaMemcpyAsync(w, src_w, n * sizeof(float), cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

moe_status_t moe_layer_get_dispatch(moe_layer_t* L, int32_t* hist, int32_t* offsets, int32_t* perm,
                                    int32_t* pos, void* stream) {
  if (!L || L->last_path != MOE_PATH_GROUPED) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int E = L->cfg.num_experts;
  const size_t n = (size_t)L->last_T * L->cfg.top_k;
  if (hist) MOE_CUDA(cudaMemcpyAsync(hist, L->grp.hist, E * sizeof(int), cudaMemcpyDeviceToDevice, s));
  if (offsets) MOE_CUDA(cudaMemcpyAsync(offsets, L->grp.offsets, (E + 1) * sizeof(int), cudaMemcpyDeviceToDevice, s));
  if (perm) MOE_CUDA(cudaMemcpyAsync(perm, L->grp.perm, n * sizeof(int), cudaMemcpyDeviceToDevice, s));
  if (pos) MOE_CUDA(cudaMemcpyAsync(pos, L->grp.pos, n * sizeof(int), cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

moe_status_t moe_layer_get_block_map(moe_layer_t* L, int32_t* blocks, int32_t max_blocks, int32_t* num_blocks,
                                     void* stream) {
  if (!L || L->last_path != MOE_PATH_GROUPED || max_blocks < 0) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t n = (size_t)std::min(max_blocks, L->grp.max_tiles);
  if (blocks && n) MOE_CUDA(cudaMemcpyAsync(blocks, L->grp.tiles, n * 2 * sizeof(int), cudaMemcpyDeviceToDevice, s));
  if (num_blocks) MOE_CUDA(cudaMemcpyAsync(num_blocks, L->grp.num_tiles, sizeof(int), cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

moe_status_t moe_layer_get_memory(const moe_layer_t* L, int64_t* weight_bytes, int64_t* workspace_bytes) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (weight_bytes) *weight_bytes = L->mem_weight_bytes;
  if (workspace_bytes) *workspace_bytes = L->mem_workspace_bytes;
  return MOE_OK;
}

moe_status_t moe_layer_get_stats(moe_layer_t* L, void* stream, moe_stats_t* st) {
  if (!L || !st) return MOE_ERR_INVALID_ARG;
  memset(st, 0, sizeof(*st));
  st->path = L->last_path;
  st->tokens = L->last_T;
  if (L->last_path == MOE_PATH_NONE) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const auto& c = L->cfg;
  const int T = L->last_T, k = c.top_k, E = c.num_experts;
  std::vector<int> idx((size_t)T * k);
  const int* src = L->last_path == MOE_PATH_GROUPED ? L->grp.idx : L->dec.idx;
  MOE_CUDA(cudaMemcpyAsync(idx.data(), src, idx.size() * sizeof(int), cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  std::vector<int> rows(E, 0);
  for (int v : idx)
    if (v >= 0 && v < E) rows[v]++;
  int distinct = 0, maxrows = 0;
  for (int r : rows) {
    distinct += r > 0;
    maxrows = std::max(maxrows, r);
  }
  const int64_t H = c.hidden, I = c.intermediate, Is = c.shared_intermediate;
  const int64_t expert_bytes = E ? (2 * I * L->row_bytes.gu + H * L->row_bytes.down) : 0;
  const int64_t shared_bytes = 3 * Is * H * 2;
  const int64_t router_bytes = H * E * 4;
  st->distinct_experts = distinct;
  st->max_expert_rows = maxrows;
  st->weight_bytes = router_bytes + (int64_t)distinct * expert_bytes + shared_bytes;
  st->algorithmic_bytes = st->weight_bytes + 2 * (int64_t)T * H * 2 +
                          (L->last_logit_bias ? (int64_t)T * E * 4 : 0);
  st->flops = 2.0 * T * H * E + 2.0 * 3.0 * I * H * (double)T * k + 2.0 * 3.0 * Is * H * T;
  return MOE_OK;
}

moe_status_t moe_layer_sync_status(moe_layer_t* L, void* stream) {
  if (!L) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int code = 0;
  MOE_CUDA(cudaMemcpy(&code, L->err, sizeof(int), cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemset(L->err, 0, sizeof(int)));
  if (code != 0) {  // an aborted call can leave the grid-sync counters mid-generation
    MOE_CUDA(cudaMemset(L->dec.sync_ctr, 0, sizeof(unsigned long long) * 4));
    if (L->grp.dispatch_ctr) MOE_CUDA(cudaMemset(L->grp.dispatch_ctr, 0, sizeof(unsigned long long)));
    MOE_CUDA(cudaMemset(L->dec.logit_words, 0, sizeof(unsigned long long) * moe::kMaxDecodeT * L->cfg.num_experts));
    MOE_CUDA(cudaMemset(L->dec.partial, 0,
                        sizeof(unsigned long long) * (size_t)L->num_sms * moe::kMaxDecodeT * L->cfg.hidden));
  }
  if (code == moe::kDevTimeout) return MOE_ERR_TIMEOUT;
  if (code != 0) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

moe_status_t moe_layer_profile_enable(moe_layer_t* L, int32_t enable) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (enable && !L->profile) {
    for (int i = 0; i < 8; ++i) MOE_CUDA(cudaEventCreate(&L->prof_ev[i]));
    L->profile = 1;
  } else if (!enable && L->profile) {
    cudaDeviceSynchronize();
    for (int i = 0; i < 8; ++i) cudaEventDestroy(L->prof_ev[i]);
    L->profile = 0;
  }
  L->prof_n = 0;
  return MOE_OK;
}

moe_status_t moe_layer_profile_read(moe_layer_t* L, float* stage_ms, int32_t max_stages, int32_t* n_stages) {
  if (!L || !stage_ms || !n_stages || !L->profile || L->prof_n < 2) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(cudaEventSynchronize(L->prof_ev[L->prof_n - 1]));
  const int n = std::min<int>(L->prof_n - 1, max_stages);
  for (int i = 0; i < n; ++i) MOE_CUDA(cudaEventElapsedTime(&stage_ms[i], L->prof_ev[i], L->prof_ev[i + 1]));
  *n_stages = n;
  return MOE_OK;
}

const char* moe_layer_describe(const moe_layer_t* L) { return L ? L->describe : ""; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_OOM: return "MOE_ERR_OOM";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_cuda_error(void) { return g_cuda_error; }

}  // extern "C"
