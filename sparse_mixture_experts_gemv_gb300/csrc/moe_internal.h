// Host-side layer state shared by the API and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_layer.h"

namespace moe {

constexpr int kMaxDecodeT = MOE_DECODE_MAX_T;  // weight-streaming path limit
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 512;
constexpr int kMaxSlots = kMaxDecodeT * kMaxTopK;  // distinct experts in one window

// Routing metadata of one decode window, written by the router kernel.
struct DecodeMeta {
  int num_slots;                              // D: distinct routed experts in the window
  int slot_expert[kMaxSlots];                 // expert of slot d, first-appearance order
  signed char slot_j[kMaxSlots][kMaxDecodeT];  // j with idx[t][j] == slot_expert[d], or -1
};

// Byte sizes of one repacked row ("record") of each weight matrix.
struct RowBytes {
  int64_t gu;    // one gate or up row of a routed expert (codes + padded scales for MXFP4)
  int64_t down;  // one down row of a routed expert
};

struct DecodeWorkspace {
  float* logits;         // [kMaxDecodeT][E]
  int* idx;              // [kMaxDecodeT][k]
  float* weights;        // [kMaxDecodeT][k]
  DecodeMeta* meta;      // one
  float* h;              // [kMaxDecodeT * k][I]   SwiGLU outputs of routed assignments (t*k+j)
  float* h_shared;       // [kMaxDecodeT][Is]
  unsigned long long* sync_ctr;   // [4] monotonic counters: [0], [1] grid syncs of the
                                  // three-phase kernel; record-streaming kernels: [2] CTA exits
                                  // (the call tag), [3] partial-output arrivals (1 per CTA per call)
  unsigned long long* logit_words;  // [kMaxDecodeT][E] router logits tagged with the call
  unsigned long long* partial;  // [num_sms][H][kMaxDecodeT] 8-byte slots; the record-streaming
                                // kernels store fp32 partial outputs [num_sms][H][T] in it
};

struct GroupedWorkspace {
  int max_tokens;
  int max_tiles;
  float* logits;         // [T][E]
  int* idx;              // [T][k]
  float* weights;        // [T][k]
  int* hist;             // [E]
  int* offsets;          // [E + 1] grouped-row offsets (offsets[E] = T*k)
  int* chunk_counts;     // per 32-token chunk counts: uint8 [chunks][E] (fused dispatch) or
                         // int [E][chunks], then chunk bases (three-kernel dispatch)
  unsigned long long* dispatch_ctr;  // arrivals of the fused dispatch kernel (each CTA adds 1 per call)
  int dispatch_grid;     // CTAs of the fused dispatch kernel: min(SMs, chunks of max_tokens), fixed
  int* perm;             // [T*k]  assignment t*k+j at each grouped row
  int* pos;              // [T*k]  grouped row of each assignment
  int* tiles;            // int2 [max_tiles] (expert, first grouped row) of each 128-row block
  int* num_tiles;        // [1] number of routed 128-row blocks
  uint16_t* h;           // bf16 [T*k][I]  SwiGLU outputs in grouped order
  uint16_t* hs;          // bf16 [T][Is]   shared-expert SwiGLU outputs
  uint16_t* y;           // bf16 [T*k][H]  down outputs in grouped order
  uint16_t* ys;          // bf16 [T][H]    shared-expert down outputs
  // MXFP4 layers (routed B rows decoded inside the grouped GEMMs):
  uint16_t* x16;         // f16 [T][H]  x for the routed gate/up rows (h is f16 for routed rows)
  uint16_t* mx_gu_sc;    // gate/up scale pairs [E][H / 64][2I]: blocks 2kb (low byte), 2kb + 1
  uint16_t* mx_dn_sc;    // down scale pairs [E][I / 64][H]
  uint8_t* mx_gu_sref;   // largest scale byte of each gate/up row [E][2I]
  uint8_t* mx_dn_sref;   // largest scale byte of each down row [E][H]
  // int4 layers: (scale, bias) bf16 pairs per stage [E][K / 64][rows] (uint32 each)
  uint32_t* i4_gu_par;   // [E][H / 64][2I]
  uint32_t* i4_dn_par;   // [E][I / 64][H]
};

}  // namespace moe

struct moe_layer {
  moe_layer_config_t cfg;
  int device;
  int num_sms;
  int decode_max_t;      // largest T the weight-streaming path serves for this shape
  int64_t mem_weight_bytes;     // device bytes of the layer's resident weight copies and tables
  int64_t mem_workspace_bytes;  // device bytes of its workspaces

  // Repacked weights (owned).
  float* router_t;       // fp32 [E][H]   (W_r transposed: one row per expert)
  float* router_bias;    // fp32 [E]      (zeros when none was given)
  uint16_t* router_split;  // bf16 [3][E][H]  W_r^T = hi + mid + lo exactly (grouped path)
  uint8_t* w_gu;         // routed gate/up, [E][I][2][row_bytes.gu]  (gate row, up row per i)
  uint8_t* w_down;       // routed down,    [E][H][row_bytes.down]
  uint16_t* ws_gu;       // shared gate/up bf16 [Is][2][H]
  uint16_t* ws_down;     // shared down bf16 [H][Is]
  uint8_t* w_rec;        // routed records [E][I], each gate row | up row | down column (bf16,
                         // H each) + zero padding: stream_record_stride(H) bytes
                         // (bf16 layers with H <= kStreamMaxHidden; nullptr otherwise)
  uint8_t* ws_rec;       // shared-expert records [Is], same record format (also for MXFP4 layers)
  uint8_t* w_mx;         // 4-bit routed records [E][I] of the MXFP4 / int4 streaming kernel:
                         // gate codes | up codes | gate scales | up scales | down column codes
                         // (code orders for the tensor-core fragments, moe_stream_common.cuh);
                         // MXFP4 stream_mx_record_stride(H) bytes each, int4 stream_i4_record_stride(H)
  uint8_t* mx_dsc;       // down scales: MXFP4 [E][I / 32][H] bytes (one H-byte vector per 32 features),
                         // int4 [E][I / 64][H] (scale, bias) bf16 pairs
  moe::RowBytes row_bytes;

  moe::DecodeWorkspace dec;
  moe::GroupedWorkspace grp;
  int* err;              // device error word
  int* never_set;        // device flag nothing sets (timeout test)
  uint16_t* x_stage;     // bf16 [max_tokens][H]  forward_host staging
  uint16_t* out_stage;   // bf16 [max_tokens][H]
  float* bias_stage;     // fp32 [max_tokens][E]

  // Last forward.
  int last_path;
  int last_T;
  const float* last_logit_bias;
  void* tmaps;           // grouped-path tensor maps (host copy), see moe_grouped.cu
  // Per-stage profiling (moe_layer_profile_enable).
  int profile;
  cudaEvent_t prof_ev[8];
  int prof_n;            // events recorded by the last forward
  char describe[1024];
};

namespace moe {
// Keeps the text of a CUDA failure for moe_last_cuda_error; returns MOE_ERR_CUDA.
moe_status_t record_cuda_failure(cudaError_t e, const char* what);
// Records the next profiling event on s (no-op unless profiling is enabled).
inline void prof_mark(moe_layer* L, cudaStream_t s) {
  if (L->profile && L->prof_n < 8) cudaEventRecord(L->prof_ev[L->prof_n++], s);
}
// Launchers (moe_decode.cu / moe_grouped.cu). Return cudaSuccess or the launch error.
cudaError_t launch_decode(moe_layer* L, const uint16_t* x, uint16_t* out, int T,
                          const float* logit_bias, cudaStream_t s);
cudaError_t launch_grouped(moe_layer* L, const uint16_t* x, uint16_t* out, int T,
                           const float* logit_bias, cudaStream_t s);
cudaError_t grouped_prepare(moe_layer* L);   // tensor maps etc. at create
void grouped_release(moe_layer* L);
size_t decode_smem_bytes_down(const moe_layer* L, int T);
cudaError_t decode_prepare(moe_layer* L);
// Record-streaming decode kernel (moe_stream.cu).
bool stream_supported(const moe_layer* L, int T);
int stream_record_stride(int H);          // bytes per routed/shared record (6H + padding)
// Record-streaming decode kernel for MXFP4 routed experts (moe_stream_mx.cu).
bool stream_mx_supported(const moe_layer* L, int T);
int stream_mx_record_stride(int H);       // bytes per routed MXFP4 record
int stream_i4_record_stride(int H);       // bytes per routed groupwise affine int4 record (same kernel)
cudaError_t stream_mx_prepare(moe_layer* L);
cudaError_t launch_stream_mx(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* logit_bias,
                             cudaStream_t s);
constexpr int kStreamMxMaxHidden = 2560;  // largest H the MXFP4 streaming kernel serves
constexpr int kStreamMaxHidden = 2048;    // largest H the record-streaming kernel serves
cudaError_t stream_prepare(moe_layer* L);
cudaError_t launch_stream(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* logit_bias,
                          cudaStream_t s);
}  // namespace moe
