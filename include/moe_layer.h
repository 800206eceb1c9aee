/*
 * moe_layer.h -- C ABI of a single-GPU (GB300, sm_103a) sparse mixture-of-experts layer.
 *
 * The layer (forward pass only):
 *   logits[t,e] = sum_h x[t,h] * W_r[h,e] + router_bias[e] + logit_bias[t,e]     (fp32)
 *   idx[t,:]    = the k largest logits, descending; exact ties go to the lower index
 *   w[t,j]      = softmax(logits[t,:])[idx[t,j]] renormalised over the k selected
 *   y_e(x)      = W_down[e] * ( silu(W_gate[e] x) .* (W_up[e] x) ),  silu(z) = z/(1+e^-z)
 *   out[t,:]    = sum_j w[t,j] * y_{idx[t,j]}(x_t) + y_shared(x_t)                (bf16)
 *
 * Sources: "Optimizing on-device inference for Apple Silicon" -- section "Qwen
 * creates three different workload shapes" (a router scores 256 experts and
 * picks 8 per token), section "Keep expert routing on the GPU" (histogram,
 * prefix scan, scatter and block map stay on the GPU; the CPU never waits
 * inside the layer), section "Reduce intermediate and state traffic" (fused
 * gated gate/up projection; down projection fused with the routing score and
 * the shared-expert result). "Three ways to speed up MoE inference on DGX
 * Spark" -- section "Why decoding was slow in the first place" (512 routed
 * experts, 8 selected, one shared expert; MXFP4 expert weights) and its closing
 * advice to verify at startup which optimisation is actually active
 * (moe_layer_describe). The pages give no API; this interface is this
 * library's own.
 *
 * Conventions for every call:
 *  - Pointers named *_dev are device pointers (cudaMalloc'ed, or any memory the
 *    device can address); *_host are host pointers. Row-major, densest
 *    dimension last, no padding between rows.
 *  - bf16 is IEEE binary16 "brain float" (the top 16 bits of an fp32), passed
 *    as raw 16-bit words.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *  - Every function returns a moe_status_t; nothing throws or aborts. A
 *    failing CUDA runtime call returns MOE_ERR_CUDA and its text is kept for
 *    moe_last_cuda_error(). No function writes to stdout or stderr.
 *  - One moe_layer_t may be used by one host thread at a time.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, size out of range, bad enum       */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented shape (see moe_layer_create)     */
  MOE_ERR_OOM = 3,           /* device allocation failed; nothing is left allocated        */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed; see moe_last_cuda_error()      */
  MOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out; outputs are undefined  */
  MOE_ERR_DEVICE_CHECK = 6   /* a device-side check failed: an index out of range, or (MXFP4
                                and int4 layers) an activation beyond the f16 range of their
                                f16 operands; outputs are undefined                        */
} moe_status_t;

typedef enum {
  MOE_WEIGHTS_BF16 = 0,      /* routed experts in bf16                                     */
  MOE_WEIGHTS_MXFP4 = 1,     /* routed experts in MXFP4: e2m1 codes, two per byte with the
                                even element in the low nibble, plus one e8m0 scale byte per
                                32 consecutive elements along the contraction dimension;
                                value = e2m1(code) * 2^(scale-127). The shared expert stays
                                bf16 and the router fp32.                                  */
  MOE_WEIGHTS_INT4 = 2       /* routed experts in groupwise affine int4 ("Optimizing
                                on-device inference for Apple Silicon", section "Decode
                                weights during matrix multiplication"): unsigned 4-bit q, two
                                per byte with the even element in the low nibble, one bf16
                                scale s and one bf16 bias b per 64 consecutive elements along
                                the contraction dimension; value = q * s + b. The shared
                                expert stays bf16 and the router fp32. Served by the
                                three-phase decode kernel and the grouped path (decoded to f16
                                there: one rounding of q * s + b).                          */
} moe_weight_format_t;

/* Create-time flags (moe_layer_config_t.flags). */
#define MOE_FLAG_FORCE_GROUPED 0x1u        /* run every T through the grouped (prefill)
                                              path, also T <= MOE_DECODE_MAX_T; for tests */
#define MOE_FLAG_ONE_WEIGHT_COPY 0x2u      /* bf16 layers with hidden <= 2048: keep only the
                                              decode kernel's per-feature [gate | up | down
                                              column] records and have the grouped GEMMs read
                                              them too (resident weights ~1.0x instead of ~2x;
                                              the grouped down GEMM reads MN-major tiles and a
                                              T=4096 Qwen-shaped prefill call measured ~10%
                                              slower on GB300). Ignored for other layers.  */
#define MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT 0x100u  /* test only: the router kernel waits on a
                                              device flag that nothing sets; the bounded wait
                                              runs out (~2 ms) and the next status check
                                              reports MOE_ERR_TIMEOUT                       */

/* Largest T served by the weight-streaming (GEMV) path; larger T use the grouped
   tensor-core path. Verify windows of 2-5 rows and 2-token-per-draft batches fit.
   (The limit is lower when T*(k*I + Is)*4 bytes of SwiGLU outputs would exceed
   200 KB, see moe_layer_describe.) The grouped path needs E a multiple of 16;
   other layers return MOE_ERR_UNSUPPORTED for larger T. It serves both weight
   formats: MXFP4 routed rows are decoded inside the tensor-core GEMMs to f16 (e2m1
   times 2^(scale - the row's largest scale), exact for blocks within 2^23 of the
   row's largest), with x and the routed SwiGLU outputs in f16 there (exact for
   |x| in [2^-14, 65504]). A finite x or routed SwiGLU output above 65504 in
   magnitude would not fit those f16 operands: the call then reports
   MOE_ERR_DEVICE_CHECK (through moe_layer_sync_status) instead of returning
   infinities. The same holds for the f16 x of the MXFP4 and int4 decode kernels. */
#define MOE_DECODE_MAX_T 8

typedef struct {
  int32_t hidden;              /* H: multiple of 256, <= 8192                               */
  int32_t num_experts;         /* E: routed experts, k <= E <= 512                          */
  int32_t top_k;               /* k: 1..8                                                   */
  int32_t intermediate;        /* I: routed expert intermediate size, multiple of 128       */
  int32_t shared_intermediate; /* Is: shared expert intermediate size, multiple of 128      */
  int32_t max_tokens;          /* largest T a forward call may pass, >= 1                   */
  int32_t weight_format;       /* moe_weight_format_t                                       */
  uint32_t flags;              /* MOE_FLAG_*                                                */
} moe_layer_config_t;

/*
 * Weights, all device pointers, read only during moe_layer_create. The layer
 * copies and repacks them into memory it owns; the caller may free them as soon
 * as create returns.
 *   router_dev       fp32 [H, E]
 *   router_bias_dev  fp32 [E] per-expert logit bias, or NULL for none
 *   BF16 format:
 *     gate_dev, up_dev   bf16 [E, I, H]   (row = intermediate feature, H contiguous)
 *     down_dev           bf16 [E, H, I]   (row = output feature, I contiguous)
 *     *_scales_dev       unused (NULL)
 *   MXFP4 format:
 *     gate_dev, up_dev   uint8 codes [E, I, H/2];  gate_scales_dev, up_scales_dev uint8 [E, I, H/32]
 *     down_dev           uint8 codes [E, H, I/2];  down_scales_dev uint8 [E, H, I/32]
 *   INT4 format (H and I multiples of 64):
 *     gate_dev, up_dev   uint8 codes [E, I, H/2];  gate/up scales and biases bf16 [E, I, H/64]
 *                        (gate_scales_dev, gate_biases_dev, ...: byte pointers to bf16 data)
 *     down_dev           uint8 codes [E, H, I/2];  down scales and biases bf16 [E, H, I/64]
 *   *_biases_dev are used by the INT4 format only (NULL otherwise).
 *   shared_gate_dev, shared_up_dev  bf16 [Is, H];  shared_down_dev bf16 [H, Is]
 */
typedef struct {
  const float* router_dev;
  const float* router_bias_dev;
  const void* gate_dev;
  const void* up_dev;
  const void* down_dev;
  const uint8_t* gate_scales_dev;
  const uint8_t* up_scales_dev;
  const uint8_t* down_scales_dev;
  const void* shared_gate_dev;
  const void* shared_up_dev;
  const void* shared_down_dev;
  const void* gate_biases_dev;
  const void* up_biases_dev;
  const void* down_biases_dev;
} moe_layer_weights_t;

typedef struct moe_layer moe_layer_t;

/* Path ids reported by moe_layer_get_stats. */
#define MOE_PATH_NONE 0
#define MOE_PATH_DECODE_GEMV 1     /* T <= MOE_DECODE_MAX_T: router -> gate/up GEMV -> down+combine */
#define MOE_PATH_GROUPED 2         /* router -> dispatch -> grouped tcgen05 GEMMs -> combine       */

typedef struct {
  int32_t path;                /* MOE_PATH_* of the last forward                           */
  int32_t tokens;              /* T of the last forward                                     */
  int32_t distinct_experts;    /* routed experts touched by the last forward                */
  int32_t max_expert_rows;     /* largest number of tokens routed to one expert             */
  int64_t weight_bytes;        /* bytes of weights the path must read once (router, touched
                                  routed experts, shared expert)                            */
  int64_t algorithmic_bytes;   /* weight_bytes + activations in/out                         */
  double flops;                /* 2*(router) + 2*3*I*H per (token, expert) + shared, useful  */
} moe_stats_t;

/*
 * Create a layer: validates the config (MOE_ERR_INVALID_ARG for out-of-range
 * values, MOE_ERR_UNSUPPORTED for shapes outside the limits above), allocates
 * device memory for the repacked weights and a workspace sized for max_tokens,
 * and repacks on the current device. Synchronous: returns after the repack has
 * finished. On failure *out is NULL and nothing stays allocated.
 */
moe_status_t moe_layer_create(const moe_layer_config_t* cfg, const moe_layer_weights_t* w,
                              moe_layer_t** out);

/* Free everything the layer owns (synchronises the device first). NULL is accepted. */
void moe_layer_destroy(moe_layer_t* layer);

/*
 * out = layer(x) for T tokens. x_dev: bf16 [T, H]; out_dev: bf16 [T, H]; both
 * 16-byte aligned and not overlapping. 0 <= T <= max_tokens (T == 0 is a no-op).
 * Enqueued on `stream`; no allocation, no host synchronisation, no host readback
 * of routing decisions. The workspace is owned by the layer, so calls on one layer
 * must be ordered (same stream, or ordered by events). A device-side error from
 * an earlier call (MOE_ERR_TIMEOUT / MOE_ERR_DEVICE_CHECK) is returned by
 * moe_layer_sync_status. After such an error the outputs of every later call are
 * undefined until moe_layer_sync_status has been called: the weight-streaming
 * kernels then return at once instead of computing (and instead of waiting out
 * their time limits on counters the failed call left mid-generation).
 */
moe_status_t moe_layer_forward(moe_layer_t* layer, const void* x_dev, void* out_dev, int32_t T,
                               void* stream);

/*
 * As moe_layer_forward, plus an optional per-(token, expert) fp32 logit bias
 * logit_bias_dev [T, E] added to the router logits before top-k (NULL = none).
 */
moe_status_t moe_layer_forward_ex(moe_layer_t* layer, const void* x_dev, void* out_dev, int32_t T,
                                  const float* logit_bias_dev, void* stream);

/*
 * Long-prompt forward in chunks ("Optimizing on-device inference for Apple
 * Silicon", section on prompt chunking: a long prompt is pushed through the layer
 * a chunk of rows at a time, so the workspace stays sized for one chunk).
 * x_dev, out_dev: bf16 [T, H] device, 16-byte aligned, not overlapping; T >= 0
 * may exceed max_tokens. chunk: rows per chunk, 1 <= chunk <= max_tokens, or 0
 * for max_tokens. logit_bias_dev: optional fp32 [T, E] (NULL = none). Every chunk,
 * including a short last one, runs the grouped tensor-core path, whose result for
 * a token does not depend on the other tokens of its chunk: the output is
 * bit-identical for every chunk size (and equal to one moe_layer_forward call with
 * MOE_FLAG_FORCE_GROUPED when T fits max_tokens). Chunks are enqueued back to back
 * on `stream` and reuse the layer's workspace in stream order; no allocation, no
 * host synchronisation. Diagnostics (get_stats, get_routing, get_dispatch) then
 * describe the last chunk. Errors: MOE_ERR_INVALID_ARG (layer NULL, T < 0, chunk
 * out of range, bad pointers), MOE_ERR_UNSUPPORTED (E not a multiple of 16),
 * MOE_ERR_CUDA (launch failure; earlier chunks may have been enqueued).
 */
moe_status_t moe_layer_forward_chunked(moe_layer_t* layer, const void* x_dev, void* out_dev, int32_t T,
                                       int32_t chunk, const float* logit_bias_dev, void* stream);

/*
 * Host-buffer forward: copies x_host (bf16 [T, H]) to the device, runs the layer
 * on `stream`, copies the result to out_host (bf16 [T, H]) and synchronises the
 * stream before returning. Pinned (page-locked) host buffers give asynchronous
 * copies; pageable buffers work but are slower. logit_bias_host may be NULL.
 */
moe_status_t moe_layer_forward_host(moe_layer_t* layer, const void* x_host, void* out_host,
                                    int32_t T, const float* logit_bias_host, void* stream);

/*
 * Statistics of the last forward. Synchronises `stream` and reads the routing
 * back (diagnostic call, not for the hot loop).
 */
moe_status_t moe_layer_get_stats(moe_layer_t* layer, void* stream, moe_stats_t* stats);

/*
 * Copy the routing of the last forward: idx_dev int32 [T, k], weights_dev fp32
 * [T, k] (device pointers; either may be NULL). Enqueued on `stream`.
 */
moe_status_t moe_layer_get_routing(moe_layer_t* layer, int32_t* idx_dev, float* weights_dev,
                                   void* stream);

/*
 * Copy the dispatch of the last grouped-path forward (MOE_ERR_INVALID_ARG after a
 * decode-path forward). All int32 device pointers, any may be NULL:
 *   hist_dev [E]        assignments per routed expert
 *   offsets_dev [E+1]   exclusive prefix sum of hist
 *   perm_dev [T*k]      assignment t*k+j at each grouped row, token order within an expert
 *   pos_dev [T*k]       grouped row of assignment t*k+j
 * Enqueued on `stream`.
 */
moe_status_t moe_layer_get_dispatch(moe_layer_t* layer, int32_t* hist_dev, int32_t* offsets_dev,
                                    int32_t* perm_dev, int32_t* pos_dev, void* stream);

/*
 * Copy the block map of the last grouped-path forward (MOE_ERR_INVALID_ARG after a
 * decode-path forward): the list of MOE_GROUPED_BLOCK_ROWS-row blocks of grouped
 * routed rows that the grouped GEMMs take as their M tiles ("Optimizing on-device
 * inference for Apple Silicon", section "Keep expert routing on the GPU": the dispatch
 * writes the block list on the GPU). Block b covers grouped rows
 * [row0, min(row0 + MOE_GROUPED_BLOCK_ROWS, offsets[e+1])) of expert e; blocks are in
 * increasing expert order, then increasing row0.
 *   blocks_dev      int32 [max_blocks][2] device: (e, row0) of each block; the first
 *                   min(max_blocks, capacity) entries are copied, where capacity is
 *                   ceil(max_tokens * k / MOE_GROUPED_BLOCK_ROWS) + E + 1; entries at or
 *                   after the block count are unspecified
 *   num_blocks_dev  int32 [1] device: the block count written by the dispatch
 * Either pointer may be NULL. max_blocks < 0 is MOE_ERR_INVALID_ARG. Enqueued on
 * `stream`.
 */
#define MOE_GROUPED_BLOCK_ROWS 128
moe_status_t moe_layer_get_block_map(moe_layer_t* layer, int32_t* blocks_dev, int32_t max_blocks,
                                     int32_t* num_blocks_dev, void* stream);

/*
 * Device memory the layer holds (host outputs; either pointer may be NULL):
 *   weight_bytes     its copies of the weights and the tables derived from them
 *                    (router, routed experts, shared expert, scale tables). By
 *                    default a layer keeps the decode kernels' feature records and
 *                    the grouped GEMMs' row layouts (~2x the expert bytes); with
 *                    MOE_FLAG_ONE_WEIGHT_COPY a bf16 layer with hidden <= 2048 keeps
 *                    the records alone (~1.0x).
 *   workspace_bytes  staging buffers and per-call scratch sized by max_tokens.
 * The caller's weight buffers passed to moe_layer_create are not counted (the layer
 * copies them and does not keep the pointers). NULL layer is MOE_ERR_INVALID_ARG.
 */
moe_status_t moe_layer_get_memory(const moe_layer_t* layer, int64_t* weight_bytes, int64_t* workspace_bytes);

/*
 * Synchronise `stream`, then read and clear the device error word: MOE_OK,
 * MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK (or MOE_ERR_CUDA if the stream itself
 * failed).
 */
moe_status_t moe_layer_sync_status(moe_layer_t* layer, void* stream);

/*
 * A static string naming the kernels instantiated for this layer and the path
 * each T range takes, e.g. to verify at startup which path is active.
 */
const char* moe_layer_describe(const moe_layer_t* layer);

/*
 * Per-stage timing (diagnostic). With profiling enabled, moe_layer_forward
 * records a CUDA event before the first kernel and after each stage's kernel
 * on the call's stream; the stages run without programmatic overlap while
 * enabled. moe_layer_profile_read synchronises on the last event and writes the
 * elapsed milliseconds of each stage of the last forward into stage_ms
 * (up to max_stages values) and their number into *n_stages. Stage names, in
 * order: decode path "router_shared", "routed_gateup", "down_combine"; grouped
 * path "router", "dispatch", "grouped_gateup", "grouped_down", "combine".
 */
moe_status_t moe_layer_profile_enable(moe_layer_t* layer, int32_t enable);
moe_status_t moe_layer_profile_read(moe_layer_t* layer, float* stage_ms, int32_t max_stages,
                                    int32_t* n_stages);

/*
 * Routing without any device allocation (no counterpart on the pages; this is
 * an entry point of this library for callers that cannot call cudaMalloc, for
 * example a host framework that owns all device memory through its own pool and
 * forbids raw allocations, or a real-time caller that must not allocate once it
 * is running).
 *
 * Computes, for T tokens, the fp32 router logits x . W_r (+ router_bias[e])
 * (+ logit_bias[t][e]), the top-k experts (descending, exact ties to the lower
 * index) and their renormalised softmax weights -- the same routing
 * moe_layer_forward does -- from buffers the caller passes:
 *   x_dev            bf16 [T, H], 8-byte aligned
 *   router_t_dev     fp32 [E, H] (W_r transposed: one row of H per expert), 16-byte aligned
 *   router_bias_dev  fp32 [E] or NULL;  logit_bias_dev fp32 [T, E] or NULL
 *   idx_dev          int32 [T, k] out;  weights_dev fp32 [T, k] out
 * Scratch: the T*E router logits live in one fixed device array inside this
 * library (MOE_NOALLOC_MAX_TOKENS * MOE_NOALLOC_MAX_EXPERTS floats = 16 KB),
 * held by every GPU that loads the library until the process exits. T above
 * MOE_NOALLOC_MAX_TOKENS, E above MOE_NOALLOC_MAX_EXPERTS or k above 8 return
 * MOE_ERR_UNSUPPORTED. Every call overwrites the whole logits region it uses
 * before reading it, so nothing needs clearing, but all calls share the array:
 * calls that overlap on the GPU (unordered streams, or several host threads)
 * race. The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture. The
 * address is kept per device and per CUDA context: after a device reset the next
 * call looks it up again. Enqueued on `stream`; no host synchronisation.
 */
#define MOE_NOALLOC_MAX_TOKENS 8
#define MOE_NOALLOC_MAX_EXPERTS 512
moe_status_t moe_route_topk_noalloc(const void* x_dev, const float* router_t_dev, const float* router_bias_dev,
                                    const float* logit_bias_dev, int32_t T, int32_t H, int32_t E, int32_t k,
                                    int32_t* idx_dev, float* weights_dev, void* stream);

/* ------------------------------------------------------------------------
 * Online-FP8 output projection (LM head), a second GEMV on the same engine
 * ("Three ways to speed up MoE inference on DGX Spark", section "Optimization
 * 2": the bf16 head, hidden 2,560 -> 157,184 vocabulary entries, is read in full
 * for every decoded token; quantizing it to FP8 when it is built halves those
 * bytes). Codes are FP8 E4M3 (OCP: bias 7, largest finite 448, no infinities),
 * one fp32 scale per output row s_v = amax_h |W[v, h]| / 448 (1 for an all-zero
 * row), q = E4M3(W / s_v) rounded to nearest even with saturation to +-448.
 * logits[t, v] = s_v * sum_h E4M3(q[v, h]) * x[t, h], accumulated in fp32;
 * activations stay bf16.
 * ------------------------------------------------------------------------ */
typedef struct moe_lmhead moe_lmhead_t;
#define MOE_LMHEAD_MAX_T 4          /* tokens per forward (decode, verify windows) */
#define MOE_LMHEAD_MAX_HIDDEN 8192

/*
 * Quantize W (w_dev: bf16 [vocab, hidden] device, row-major, 16-byte aligned) into
 * codes and scales the head owns; the caller may free w_dev afterwards.
 * Synchronous. hidden must be a multiple of 256 and <= MOE_LMHEAD_MAX_HIDDEN
 * (else MOE_ERR_UNSUPPORTED); vocab >= 1. Errors: MOE_ERR_INVALID_ARG,
 * MOE_ERR_OOM, MOE_ERR_CUDA. On failure *out is NULL and nothing stays allocated.
 */
moe_status_t moe_lmhead_create(int32_t hidden, int32_t vocab, const void* w_dev, moe_lmhead_t** out);

/*
 * logits_dev fp32 [T, vocab] = head(x_dev bf16 [T, hidden]); 0 <= T <=
 * MOE_LMHEAD_MAX_T (T == 0 is a no-op). x_dev 16-byte aligned, logits_dev 4-byte
 * aligned, not overlapping. One kernel enqueued on `stream`; no allocation, no
 * host synchronisation. Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA.
 */
moe_status_t moe_lmhead_forward(moe_lmhead_t* head, const void* x_dev, float* logits_dev, int32_t T,
                                void* stream);

/*
 * Copy the quantized weights out (diagnostic): codes_dev uint8 [vocab, hidden],
 * scales_dev fp32 [vocab] (device pointers; either may be NULL). Enqueued on
 * `stream`.
 */
moe_status_t moe_lmhead_get_weights(moe_lmhead_t* head, void* codes_dev, float* scales_dev, void* stream);

/* Free the head (synchronises the device first). NULL is accepted. */
void moe_lmhead_destroy(moe_lmhead_t* head);

/* Name of a status code (static string). */
const char* moe_status_string(moe_status_t status);

/* Text of the last failing CUDA runtime call in this thread ("" if none). */
const char* moe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
