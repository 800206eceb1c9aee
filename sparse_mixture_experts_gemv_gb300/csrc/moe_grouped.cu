// Grouped (prefill) path of the MoE layer: many tokens per call.
//
// "Optimizing on-device inference for Apple Silicon", sections "Prefill: reuse
// weights, keep routing on the GPU" and "Keep expert routing on the GPU": the
// grouped GEMM needs each expert's activation rows together, so after top-k a
// histogram counts the assignments per expert, a prefix scan turns the counts
// into offsets, a scatter writes the token rows into per-expert groups and a
// block map lists the fixed-size row blocks the grouped GEMM processes -- all
// on the GPU, with no host round trip inside the layer. Section "Match tile
// size to expert load": expert loads are uneven, so tiles follow the actual
// per-expert row counts (128-row blocks here, any count per expert).
//
// Kernels, chained with programmatic dependent launch:
//   grouped_gemm<ROUTER>  fp32-exact router logits on the tensor cores: W_r is
//                         split exactly into three bf16 terms (hi + mid + lo), x is
//                         bf16, so every product is exact and the accumulation is
//                         fp32 (each staged x tile meets all three terms, all
//                         MMAs into one TMEM accumulator).
//   topk_hist             per-token top-k + renormalised softmax weights; per
//                         32-token chunk expert histogram.
//   dispatch_scan         per-expert totals, chunk bases, offsets, block map.
//   dispatch_scatter      grouped row of every (token, slot), token order kept.
//   grouped_gemm<SWIGLU>  gate/up for every expert group (+ the shared expert
//                         over all tokens), A rows gathered from x by cp.async,
//                         SwiGLU in the epilogue, bf16 h in grouped order.
//   grouped_gemm<STORE>   down projection of every group (TMA A = h), bf16 y.
//   combine               out[t] = sum_j w[t,j] y[pos[t,j]] + y_shared[t].
// A chunked forward (moe_layer_forward_chunked) repeats this chain per chunk.
//
// The grouped GEMM is a persistent, warp-specialised tcgen05 kernel: warp 0
// issues TMA loads, warp 1 owns tensor memory and issues the MMAs, warps 2-5
// drain the double-buffered TMEM accumulators; for gathered A, warps 6-9 copy
// the token rows with cp.async into the 128-byte-swizzled layout.
//
// 4-bit routed experts ("Optimizing on-device inference for Apple Silicon",
// section "Decode weights during matrix multiplication"; "Three ways to speed up
// MoE inference on DGX Spark", section "Optimization 1"): for MXFP4 and
// groupwise affine int4 layers, eight more converter warps turn each stage's
// 4-bit rows (copied into a raw ring) into the f16 B tile in shared memory, and
// the routed MMAs are f16 x f16 (x and the SwiGLU outputs in f16); x is
// converted once per call by bf16_to_f16 before the router.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_sm100.cuh"

namespace moe {
namespace {

using namespace sm100;

constexpr int BM = 128;                  // rows (tokens) per tile = TMEM lanes
static_assert(BM == MOE_GROUPED_BLOCK_ROWS, "block map rows of the C ABI");
constexpr int BK = 64;                   // bf16 per 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kStageA = BM * BK * 2;     // 16 KB
constexpr int kStageB = 256 * BK * 2;    // 32 KB (N up to 256)
constexpr int kTmemCols = 512;           // two 256-column fp32 accumulators
constexpr int kGatherAhead = 2;          // stages between an A row's L2 prefetch and its copy
constexpr int kChunk = 32;               // tokens per dispatch chunk (one per warp of the top-k CTA)
constexpr size_t kDispatchMaskSmem = 128 * 1024;  // largest dynamic shared memory of the fused dispatch
constexpr size_t kDispatchRedSmem = 2 * 4096 * sizeof(int);   // its per-part count table
constexpr size_t kGemmSmem = (size_t)kStages * (kStageA + kStageB) + 1024 /*align*/ + 256 /*barriers*/;
// MXFP4 B operands: a separate ring of raw stages (e2m1 codes of 256 B rows x 64
// K, 32 bytes a row, then the rows' scale pairs) that converter warps decode into
// the f16 B stage of the main ring.
constexpr int kRaw = 3;
constexpr int kRawCodes = 256 * (BK / 2);  // 8 KB
constexpr int kRawParMax = 256 * 4;        // per-row stage parameters: MXFP4 2 scale bytes, int4 (s, b) bf16
constexpr int kRawStage = kRawCodes + kRawParMax;
// B operand kinds of the grouped GEMM: bf16 rows by TMA, or 4-bit rows decoded in the kernel.
enum BKind { B_BF16 = 0, B_MXFP4 = 1, B_INT4 = 2 };
constexpr size_t kGemmSmemMx = kGemmSmem + (size_t)kRaw * kRawStage;
constexpr int kConvThreads = 256;          // one B row per converter thread

enum Epi { EPI_ROUTER = 0, EPI_SWIGLU = 1, EPI_STORE = 2 };

struct GemmParams {
  // Tiles: routed M-blocks come from the block map (count in device memory),
  // shared-expert M-blocks cover the tokens directly.
  const int2* mtiles;       // [R] (expert, first grouped row); nullptr for the router
  const int* num_routed;    // device count R (nullptr: R = n_routed_static)
  int n_routed_static;
  int n_shared_mtiles;      // S
  int nt_routed, nt_shared; // N tiles per M-block
  int ks_routed, ks_shared; // 64-wide K steps per tile
  int ks_part;              // router: K steps per bf16 term
  int BN;
  int max_mtiles;           // capacity of the block map
  int E;
  int T;
  int k;
  const int* offsets;       // [E + 1] grouped-row offsets
  // gathered A (gate/up)
  const uint16_t* x;        // bf16 [T][H]
  int H;
  const int* perm;          // [T*k] assignment t*k+j at each grouped row
  // B rows of expert e start at e * b_rows_per_expert (routed map)
  int b_rows_per_expert;
  // bf16 B from the decode kernels' feature records (0: row layouts): the number
  // of features per routed expert. Gate/up tiles then come from a 3-D map
  // {H, gate/up, feature} (K-major, as the row layout), down tiles from the
  // records' down columns as four 64 x 64 MN-major boxes per stage.
  int b_rec;
  // epilogue outputs
  uint16_t* out_routed; int ld_routed;
  uint16_t* out_shared; int ld_shared;
  float* logits; const float* router_bias; const float* logit_bias;
  int* err;
  // 4-bit routed experts (B rows decoded in the kernel): routed A operands are f16
  // (x16 for the gathered gate/up rows, f16 h for the down rows).
  const uint16_t* x16;      // f16 [T][H]
  const void* q_par;        // per-stage row parameters [E][K / 64][b_rows_per_expert]:
                            // MXFP4 uint16 scale pairs, int4 uint32 (scale, bias) bf16 pairs
  const uint8_t* mx_sref;   // MXFP4: reference exponent of each B row [E][b_rows_per_expert]
};

struct TileInfo {
  bool shared;
  int e, row0, row_end, nt, ks;
};

__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int R, int tile) {
  TileInfo ti;
  const int routed_tiles = R * p.nt_routed;
  if (tile < routed_tiles) {
    const int m = tile / p.nt_routed;
    ti.shared = false;
    ti.nt = tile % p.nt_routed;
    ti.ks = p.ks_routed;
    if (p.mtiles) {
      const int2 mt = p.mtiles[m];
      const int TK = p.T * p.k;
      if (mt.x < 0 || mt.x >= p.E || mt.y < 0 || mt.y >= TK) {  // inconsistent block map
        set_error(p.err, kDevCheck);
        ti.e = 0; ti.row0 = 0; ti.row_end = 0;
      } else {
        ti.e = mt.x;
        ti.row0 = mt.y;
        ti.row_end = min(p.offsets[mt.x + 1], TK);
      }
    } else {  // router: plain token blocks
      ti.e = 0;
      ti.row0 = m * BM;
      ti.row_end = p.T;
    }
  } else {
    const int t2 = tile - routed_tiles;
    ti.shared = true;
    ti.e = p.E;
    ti.nt = t2 % p.nt_shared;
    ti.row0 = (t2 / p.nt_shared) * BM;
    ti.row_end = p.T;
    ti.ks = p.ks_shared;
  }
  return ti;
}

// Instruction descriptor of kind::f16 with f16 A and B (format 0), fp32
// accumulation, both operands K-major, shape M x N.
constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 2^d as a pair of f16 (d <= 15): normal down to 2^-14, subnormal down to 2^-24,
// zero below.
__device__ __forceinline__ uint32_t pow2_f16x2(int d) {
  d = min(d, 15);
  const uint32_t h = d >= -14 ? (uint32_t)(d + 15) << 10 : (d >= -24 ? 1u << (d + 24) : 0u);
  return h | (h << 16);
}
__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Two fp32 -> f16 pair, lo in the low half (round to nearest even).
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Eight e2m1 codes (one 32-bit word, element 2i in the low nibble of byte i)
// times the f16 pair f -> eight f16 in element order.
__device__ __forceinline__ uint4 e2m1x8_to_f16(uint32_t w, uint32_t f) {
  return make_uint4(hmul2_f16(e2m1x2_to_f16x2(w), f), hmul2_f16(e2m1x2_to_f16x2(w >> 8), f),
                    hmul2_f16(e2m1x2_to_f16x2(w >> 16), f), hmul2_f16(e2m1x2_to_f16x2(w >> 24), f));
}

// Eight unsigned 4-bit codes (one word, element 2i in the low nibble of byte i)
// -> f16(q * s + b) for the f16 pairs s2 = {s, s}, b2 = {b, b}: q is made exact in
// f16 as (0x6400 | q) - 1024, then one fused multiply-add rounds once.
__device__ __forceinline__ uint32_t u4x2_affine_f16x2(uint32_t byte, uint32_t s2, uint32_t b2) {
  const uint32_t w = 0x64006400u | (byte & 0x0Fu) | ((byte & 0xF0u) << 12);
  uint32_t q, r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(q) : "r"(w), "r"(0x64006400u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(s2), "r"(b2));
  return r;
}
__device__ __forceinline__ uint4 u4x8_affine_f16(uint32_t w, uint32_t s2, uint32_t b2) {
  return make_uint4(u4x2_affine_f16x2(w, s2, b2), u4x2_affine_f16x2(w >> 8, s2, b2),
                    u4x2_affine_f16x2(w >> 16, s2, b2), u4x2_affine_f16x2(w >> 24, s2, b2));
}

// BQ = B_MXFP4: routed B rows are MXFP4 (e2m1 codes + one e8m0 scale per 32 K). The
// producer copies each stage's codes (TMA, 32 bytes x 256 rows) and the rows'
// scale pairs (one bulk copy) into a raw ring; converter warps decode them into
// the f16 B stage: e2m1 -> f16 (exact) times 2^(s - sref), sref being the row's
// largest scale, so the stage is exact f16 for blocks within 2^23 of the row's
// largest; the epilogue multiplies column n by 2^(sref[n] - 127). Routed A rows
// are f16 then (x16 for gate/up, f16 h for down) and the MMA kind is f16 x f16;
// shared-expert tiles stay bf16 x bf16 through TMA. BQ = B_INT4: the same
// pipeline with groupwise affine int4 rows; one stage of K = 64 is one group,
// and the converter writes f16(q * s + b) with one fused multiply-add (one
// rounding); no column factor.
template <int EPI, bool GATHER, int BQ>
__global__ void __launch_bounds__((GATHER ? 320 : 192) + (BQ != B_BF16 ? kConvThreads : 0), 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA_r, const __grid_constant__ CUtensorMap mapA_s,
                    const __grid_constant__ CUtensorMap mapB_r, const __grid_constant__ CUtensorMap mapB_s,
                    const GemmParams p) {
  constexpr bool MXB = BQ != B_BF16;           // B rows decoded by converter warps
  constexpr int kParBytes = BQ == B_INT4 ? 4 : 2;   // stage parameters per B row
  constexpr int kConvWarp0 = GATHER ? 10 : 6;  // first converter warp (MXB)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageA;
  uint8_t* sRaw = sB + kStages * kStageB;  // MXB: raw ring
  uint64_t* full = (uint64_t*)(sRaw + (MXB ? kRaw * kRawStage : 0));
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* raw_full = acc_empty + 2;
  uint64_t* raw_empty = raw_full + kRaw;
  uint64_t* drain = raw_empty + kRaw;
  uint32_t* tmem_slot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1 + (GATHER ? 128 : 0) + (MXB ? kConvThreads : 0));
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
    }
    for (int q = 0; q < kRaw; ++q) {
      mbar_init(&raw_full[q], 1);
      mbar_init(&raw_empty[q], kConvThreads);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mapB_r);
    prefetch_tmap(&mapB_s);
    if (!GATHER) { prefetch_tmap(&mapA_r); prefetch_tmap(&mapA_s); }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();  // routing / dispatch / SwiGLU outputs of this call are complete
  pdl_launch_dependents();

  int R = p.num_routed ? ldg_cg_s32(p.num_routed) : p.n_routed_static;
  if (R < 0 || R > p.max_mtiles) {
    if (threadIdx.x == 0) set_error(p.err, kDevCheck);
    R = 0;
  }
  const int total = R * p.nt_routed + p.n_shared_mtiles * p.nt_shared;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, rit = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < total && !stop && !*abort_flag; tile += gridDim.x) {
        const TileInfo ti = decode_tile(p, R, tile);
        const bool mxt = MXB && !ti.shared;
        for (int kb = 0; kb < ti.ks; ++kb, ++it) {
          const int kcol = kb * BK;
          if (mxt) {  // raw codes and scale pairs of this stage's 256 B rows
            const int q = rit % kRaw;
            if (!mbar_wait(&raw_empty[q], ((rit / kRaw) & 1) ^ 1, p.err, abort_flag)) { stop = true; break; }
            mbar_arrive_expect_tx(&raw_full[q], (uint32_t)(kRawCodes + 256 * kParBytes));
            const int brow = ti.e * p.b_rows_per_expert + ti.nt * 256;
            tma_load_2d(sRaw + q * kRawStage, &mapB_r, kb * (BK / 2), brow, &raw_full[q]);
            bulk_copy_g2s(sRaw + q * kRawStage + kRawCodes,
                          reinterpret_cast<const uint8_t*>(p.q_par) +
                              (((size_t)ti.e * ti.ks + kb) * p.b_rows_per_expert + ti.nt * 256) * kParBytes,
                          (uint32_t)(256 * kParBytes), &raw_full[q]);
            ++rit;
          }
          const int s = it % kStages;
          if (!mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, p.err, abort_flag)) { stop = true; break; }
          const uint32_t bbytes = mxt ? 0u : (uint32_t)p.BN * BK * 2 * (EPI == EPI_ROUTER ? 3 : 1);
          mbar_arrive_expect_tx(&full[s], bbytes + (GATHER ? 0u : (uint32_t)kStageA));
          if (EPI == EPI_ROUTER) {  // the three bf16 terms of W_r share this A tile
#pragma unroll
            for (int part = 0; part < 3; ++part)
              tma_load_2d(sB + s * kStageB + part * p.BN * BK * 2, &mapB_r, kcol, part * p.E + ti.nt * p.BN, &full[s]);
          } else if (!mxt) {
            const CUtensorMap* mb = ti.shared ? &mapB_s : &mapB_r;
            if (BQ == B_BF16 && p.b_rec && EPI == EPI_SWIGLU) {   // features nt*128 .. +127, {gate, up} rows
              tma_load_3d(sB + s * kStageB, mb, kcol, 0, (ti.shared ? 0 : ti.e * p.b_rec) + ti.nt * (p.BN / 2),
                          &full[s]);
            } else if (BQ == B_BF16 && p.b_rec) {   // down columns: K rows = features, 64 n a box
              const int krow = (ti.shared ? 0 : ti.e * p.b_rec) + kcol;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tma_load_2d(sB + s * kStageB + j * (64 * BK * 2), mb, ti.nt * p.BN + 64 * j, krow, &full[s]);
            } else {
              const int brow = (ti.shared ? 0 : ti.e * p.b_rows_per_expert) + ti.nt * p.BN;
              tma_load_2d(sB + s * kStageB, mb, kcol, brow, &full[s]);
            }
          }
          if (!GATHER) tma_load_2d(sA + s * kStageA, ti.shared ? &mapA_s : &mapA_r, kcol, ti.row0, &full[s]);
        }
      }
      if (*abort_flag) {  // let copies already issued land before the CTA exits
        for (uint32_t q = (it > (uint32_t)kStages ? it - kStages : 0); q < it; ++q)
          mbar_wait(&full[q % kStages], (q / kStages) & 1, p.err, abort_flag, 20000000LL, false);
        if (MXB)
          for (uint32_t q = (rit > (uint32_t)kRaw ? rit - kRaw : 0); q < rit; ++q)
            mbar_wait(&raw_full[q % kRaw], (q / kRaw) & 1, p.err, abort_flag, 20000000LL, false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_bf = idesc_bf16_f32(BM, p.BN), idesc_h = idesc_f16_f32(BM, p.BN);
      // down tiles from records: B is MN-major (transpose-B bit of the instruction descriptor)
      const bool b_mn = BQ == B_BF16 && EPI == EPI_STORE && p.b_rec != 0;
      const uint32_t idesc_bmn = idesc_bf | kIdescTransposeB;
      uint32_t it = 0, tc = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++tc) {
        const TileInfo ti = decode_tile(p, R, tile);
        const uint32_t idesc = (MXB && !ti.shared) ? idesc_h : b_mn ? idesc_bmn : idesc_bf;
        const int ab = tc & 1;
        if (!mbar_wait(&acc_empty[ab], ((tc >> 1) & 1) ^ 1, p.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + ab * 256;
        bool ok = true;
        for (int kb = 0; kb < ti.ks; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&full[s], (it / kStages) & 1, p.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kStageA), b0 = smem_u32(sB + s * kStageB);
          constexpr int kTerms = (EPI == EPI_ROUTER) ? 3 : 1;
#pragma unroll
          for (int part = 0; part < kTerms; ++part) {
            const uint32_t bp = b0 + part * p.BN * BK * 2;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // K-major B: the next 16 K columns are 32 bytes on; MN-major B: 16 K rows
              // of 128 bytes on (two 8-row groups), the 64-column boxes 8 KB apart
              const uint64_t bdesc = b_mn ? smem_desc_sw128_mn(bp + kk * 2048, 64 * BK * 2)
                                          : smem_desc_sw128(bp + kk * 32);
              mma_bf16(d, smem_desc_sw128(a0 + kk * 32), bdesc, idesc, (kb | kk | part) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&acc_full[ab]);
      }
      // all issued MMAs complete before tensor memory is released
      mma_commit(drain);
      mbar_wait(drain, 0, p.err, abort_flag, 2000000000LL, false);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;      // tile row = TMEM lane
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++tc) {
      const TileInfo ti = decode_tile(p, R, tile);
      const bool mxt = MXB && !ti.shared;
      const int ab = tc & 1;
      if (!mbar_wait(&acc_full[ab], (tc >> 1) & 1, p.err, abort_flag)) break;
      tc_fence_after();
      const int gr = ti.row0 + r;
      const bool valid = gr < ti.row_end;
      const uint32_t taddr = tmem + ab * 256 + ((uint32_t)(q * 32) << 16);
      for (int c0 = 0; c0 < p.BN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(taddr + c0, v);
        if (!valid) continue;
        if (BQ == B_MXFP4 && mxt) {  // column n of a decoded MXFP4 tile carries 2^(127 - sref[n])
          const uint4* sr = reinterpret_cast<const uint4*>(p.mx_sref + (size_t)ti.e * p.b_rows_per_expert +
                                                           ti.nt * p.BN + c0);
          const uint4 s0 = __ldg(sr), s1 = __ldg(sr + 1);
          const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = __float_as_uint(__uint_as_float(v[i]) * e8m0_to_f32((sw[i >> 2] >> (8 * (i & 3))) & 0xFFu));
        }
        if (EPI == EPI_SWIGLU) {
          // columns alternate gate / up of intermediate features i0 + c0/2 + (0..15)
          uint32_t packed[8];
          bool h_range = false;   // a routed f16 h above the f16 range: reported, never silently infinite
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float h0 = swiglu(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]));
            const float h1 = swiglu(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            if (mxt) h_range |= f16_overflows(h0) || f16_overflows(h1);
            packed[i] = mxt ? f32x2_to_f16x2(h0, h1)   // f16 A of the MXFP4 down GEMM
                            : (uint32_t)f32_to_bf16_rne(h0) | ((uint32_t)f32_to_bf16_rne(h1) << 16);
          }
          if (h_range) set_error(p.err, kDevCheck);
          uint16_t* dst = ti.shared ? p.out_shared + (size_t)gr * p.ld_shared
                                    : p.out_routed + (size_t)gr * p.ld_routed;
          dst += ti.nt * (p.BN / 2) + c0 / 2;
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        } else if (EPI == EPI_STORE) {
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = (uint32_t)f32_to_bf16_rne(__uint_as_float(v[2 * i])) |
                        ((uint32_t)f32_to_bf16_rne(__uint_as_float(v[2 * i + 1])) << 16);
          uint16_t* dst = ti.shared ? p.out_shared + (size_t)gr * p.ld_shared
                                    : p.out_routed + (size_t)gr * p.ld_routed;
          dst += ti.nt * p.BN + c0;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            reinterpret_cast<uint4*>(dst)[i] =
                make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        } else {  // EPI_ROUTER: fp32 logits + biases
          const int e0 = ti.nt * p.BN + c0;
          const int ncol = min(32, p.BN - c0);
          float* dst = p.logits + (size_t)gr * p.E + e0;
          const float* lb = p.logit_bias ? p.logit_bias + (size_t)gr * p.E + e0 : nullptr;
          for (int i = 0; i < ncol; i += 4) {
            float4 o;
            o.x = __uint_as_float(v[i + 0]) + p.router_bias[e0 + i + 0];
            o.y = __uint_as_float(v[i + 1]) + p.router_bias[e0 + i + 1];
            o.z = __uint_as_float(v[i + 2]) + p.router_bias[e0 + i + 2];
            o.w = __uint_as_float(v[i + 3]) + p.router_bias[e0 + i + 3];
            if (lb) { o.x += lb[i]; o.y += lb[i + 1]; o.z += lb[i + 2]; o.w += lb[i + 3]; }
            *reinterpret_cast<float4*>(dst + i) = o;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[ab]);
    }
  } else if (GATHER && warp < 10) {
    // ------------------------------------------------------------ A gather (gate/up)
    // Eight threads copy one 128-byte row of a stage (thread j of the eight takes
    // 16-byte chunk j), so one cp.async instruction of a warp covers four whole
    // rows (four cache lines) instead of one chunk of 32 different rows: the
    // gather is bound by L1TEX requests. Thread t copies chunk t % 8 of rows
    // t / 8 + 16 i, i = 0..7. For bf16 layers the first thread of each row also
    // requests the row's line kGatherAhead stages on into L2, so a copy usually
    // waits for L2, not DRAM (gate/up at T = 4096 on GB300: 203 -> 182 us; the
    // 4-bit kernels, whose converters share the issue slots, were 6-10 us slower
    // with it, and prefetching 4-12 stages on gained less).
    const int tid = threadIdx.x - 192;
    const int jc = tid & 7, rb = tid >> 3;
    uint32_t it = 0;
    int pending = -1;
    for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
      const TileInfo ti = decode_tile(p, R, tile);
      const uint16_t* xa = (MXB && !ti.shared) ? p.x16 : p.x;  // routed 4-bit tiles take f16 rows
      const uint16_t* src[8];
      uint32_t nbytes[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int gr = ti.row0 + rb + 16 * i;
        int token = -1;
        if (gr < ti.row_end) {
          if (ti.shared) {
            token = gr;
          } else {
            const int a = p.perm[gr];
            if (a >= 0 && a < p.T * p.k) token = a / p.k;
            else set_error(p.err, kDevCheck);
          }
        }
        src[i] = xa + (size_t)(token < 0 ? 0 : token) * p.H + 8 * jc;
        nbytes[i] = token < 0 ? 0u : 16u;   // rows past the group's end are written as zeros
      }
      bool ok = true;
      for (int kb = 0; kb < ti.ks; ++kb, ++it) {
        const int s = it % kStages;
        if (!mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
        uint8_t* dst = sA + s * kStageA + ((jc ^ (rb & 7)) << 4);   // (rb + 16 i) % 8 == rb % 8
#pragma unroll
        for (int i = 0; i < 8; ++i) cp_async_16(dst + (rb + 16 * i) * 128, src[i] + kb * BK, nbytes[i]);
        cp_async_commit();
        if (!MXB && jc == 0 && kb + kGatherAhead < ti.ks) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (nbytes[i]) prefetch_l2(src[i] + (kb + kGatherAhead) * BK);
        }
        if (pending >= 0) {
          cp_async_wait<1>();
          fence_proxy_async_smem();
          mbar_arrive(&full[pending]);
        }
        pending = s;
      }
      if (!ok) break;
    }
    cp_async_wait<0>();
    if (pending >= 0) {
      fence_proxy_async_smem();
      mbar_arrive(&full[pending]);
    }
  } else if (MXB) {
    // ------------------------------------------------------------ MXFP4 B converter
    const int r = threadIdx.x - kConvWarp0 * 32;   // B row of the tile this thread decodes
    uint32_t it = 0, rit = 0;
    for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
      const TileInfo ti = decode_tile(p, R, tile);
      const bool mxt = !ti.shared;
      const int sref = (BQ == B_MXFP4 && mxt)
                           ? (int)__ldg(p.mx_sref + (size_t)ti.e * p.b_rows_per_expert + ti.nt * 256 + r) : 0;
      bool ok = true;
      for (int kb = 0; kb < ti.ks; ++kb, ++it) {
        const int s = it % kStages;
        if (!mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, p.err, abort_flag)) { ok = false; break; }
        if (mxt) {
          const int q = rit % kRaw;
          if (!mbar_wait(&raw_full[q], (rit / kRaw) & 1, p.err, abort_flag)) { ok = false; break; }
          const uint8_t* rb = sRaw + q * kRawStage;
          const uint4 c0 = *reinterpret_cast<const uint4*>(rb + r * 32);
          const uint4 c1 = *reinterpret_cast<const uint4*>(rb + r * 32 + 16);
          ++rit;
          const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint8_t* dst = sB + s * kStageB + r * 128;
          if (BQ == B_MXFP4) {
            const uint32_t sc = *reinterpret_cast<const uint16_t*>(rb + kRawCodes + 2 * r);
            const uint32_t f0 = pow2_f16x2((int)(sc & 0xFFu) - sref), f1 = pow2_f16x2((int)(sc >> 8) - sref);
#pragma unroll
            for (int j = 0; j < 8; ++j)   // 16-byte chunk j = K elements 8j..8j+7 (block 2kb for j < 4)
              *reinterpret_cast<uint4*>(dst + ((j ^ (r & 7)) << 4)) = e2m1x8_to_f16(w[j], j < 4 ? f0 : f1);
          } else {   // int4: this stage is group kb of the row
            const uint32_t sb = *reinterpret_cast<const uint32_t*>(rb + kRawCodes + 4 * r);
            const uint32_t s2 = f32x2_to_f16x2(bf16_lo(sb), bf16_lo(sb)), b2 = f32x2_to_f16x2(bf16_hi(sb), bf16_hi(sb));
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(dst + ((j ^ (r & 7)) << 4)) = u4x8_affine_f16(w[j], s2, b2);
          }
          fence_proxy_async_smem();
          // The raw slot is released only once its values have been used: an
          // arrival issued right after the loads can be observed (and the slot
          // refilled by the next bulk copy) before those loads have read shared
          // memory, which showed as stale rows of whole converter warps.
          mbar_arrive(&raw_empty[q]);
        }
        mbar_arrive(&full[s]);
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ===========================================================================
// Routing: top-k per token, per-chunk histogram
// ===========================================================================
__global__ void __launch_bounds__(1024)
topk_hist_kernel(const float* __restrict__ logits, int T, int E, int k, int* __restrict__ idx,
                 float* __restrict__ weights, int* __restrict__ chunk_counts) {
  __shared__ int s_count[kMaxExperts];
  pdl_wait();
  pdl_launch_dependents();
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_count[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int tl = warp; tl < kChunk; tl += 32) {
    const int t = blockIdx.x * kChunk + tl;
    if (t >= T) break;
    if (E <= 256) warp_topk<1>(logits + (size_t)t * E, E, k, lane, idx + (size_t)t * k, weights + (size_t)t * k);
    else warp_topk<2>(logits + (size_t)t * E, E, k, lane, idx + (size_t)t * k, weights + (size_t)t * k);
    __syncwarp();
    if (lane < k) atomicAdd(&s_count[idx[(size_t)t * k + lane]], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(size_t)e * gridDim.x + blockIdx.x] = s_count[e];
}

// One CTA. Counts are [E][chunks]: warp w scans the chunk counts of experts
// w, w + 32, ... (exclusive, 32 chunks per pass with warp shuffles) into chunk
// bases and expert totals; then exclusive scans over the experts give the
// grouped-row offsets and the 128-row block map.
__global__ void __launch_bounds__(1024)
dispatch_scan_kernel(int* __restrict__ chunk_counts /* in: counts, out: bases */, int num_chunks, int E, int T,
                     int k, int* __restrict__ hist, int* __restrict__ offsets, int2* __restrict__ mtiles,
                     int* __restrict__ num_routed, int max_mtiles, int* __restrict__ err) {
  __shared__ int s_tot[1024];
  __shared__ int s_tiles[1024];
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Scan of one expert's chunk counts; v holds chunks c0 + lane, c0 + 32 + lane, ...
  auto scan_row = [&](int e, int* row, int c0, int nq, const int (&v)[4], int& run) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < nq) {
        const int c = c0 + 32 * q + lane;
        int incl = v[q];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += n;
        }
        if (c < num_chunks) row[c] = run + incl - v[q];   // exclusive base of chunk c for expert e
        run += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
  };
  if (num_chunks <= 128) {
    // up to 128 chunks: the four rows a warp scans at a time are loaded at once
    // (one round trip for 16 loads a lane instead of one per 32 chunks)
    for (int e0 = warp; e0 < E; e0 += 32 * 4) {
      int v[4][4];
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = e0 + 32 * x, c = 32 * q + lane;
          v[x][q] = (e < E && c < num_chunks) ? chunk_counts[(size_t)e * num_chunks + c] : 0;
        }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int e = e0 + 32 * x;
        if (e < E) {
          int run = 0;
          scan_row(e, chunk_counts + (size_t)e * num_chunks, 0, 4, v[x], run);
          if (lane == 0) {
            hist[e] = run;
            s_tot[e] = run;
            s_tiles[e] = (run + BM - 1) / BM;
          }
        }
      }
    }
  } else {
    for (int e = warp; e < E; e += 32) {
      int* row = chunk_counts + (size_t)e * num_chunks;
      int run = 0;
      for (int c0 = 0; c0 < num_chunks; c0 += 128) {
        int v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = c0 + 32 * q + lane;
          v[q] = c < num_chunks ? row[c] : 0;
        }
        scan_row(e, row, c0, 4, v, run);
      }
      if (lane == 0) {
        hist[e] = run;
        s_tot[e] = run;
        s_tiles[e] = (run + BM - 1) / BM;
      }
    }
  }
  for (int e = E + threadIdx.x; e < (int)blockDim.x; e += blockDim.x) { s_tot[e] = 0; s_tiles[e] = 0; }
  __syncthreads();
  const int e = threadIdx.x;
  const int run = (e < E) ? s_tot[e] : 0;
  // exclusive scans over experts (E <= 512, simple two-array Hillis-Steele)
  for (int d = 1; d < blockDim.x; d <<= 1) {
    int a = 0, b = 0;
    if (e >= d) { a = s_tot[e - d]; b = s_tiles[e - d]; }
    __syncthreads();
    s_tot[e] += a;
    s_tiles[e] += b;
    __syncthreads();
  }
  if (e < E) {
    const int off = s_tot[e] - run;  // exclusive
    const int ntile = (run + BM - 1) / BM;
    const int tile0 = s_tiles[e] - ntile;
    offsets[e] = off;
    for (int m = 0; m < ntile; ++m) {
      if (tile0 + m < max_mtiles) mtiles[tile0 + m] = make_int2(e, off + m * BM);
      else set_error(err, kDevCheck);
    }
    if (e == E - 1) {
      offsets[E] = off + run;  // == T * k
      *num_routed = tile0 + ntile;
    }
  }
}

// Grouped row of every assignment: offsets[e] + chunk base + rank within the
// chunk, the rank counting the chunk's earlier tokens that chose e (one warp
// walks the chunk's tokens in order; a token's k experts are distinct).
__global__ void __launch_bounds__(256)
dispatch_scatter_kernel(const int* __restrict__ idx, const int* __restrict__ chunk_bases,
                        const int* __restrict__ offsets, int T, int E, int k, int* __restrict__ perm,
                        int* __restrict__ pos, int* __restrict__ err) {
  __shared__ int s_next[kMaxExperts];
  __shared__ int s_e[kChunk * kMaxTopK];
  pdl_wait();
  pdl_launch_dependents();
  const int t0 = blockIdx.x * kChunk;
  const int ntok = min(kChunk, T - t0);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    s_next[e] = offsets[e] + chunk_bases[(size_t)e * gridDim.x + blockIdx.x];
  for (int q = threadIdx.x; q < ntok * k; q += blockDim.x) s_e[q] = idx[(size_t)t0 * k + q];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    for (int tl = 0; tl < ntok; ++tl) {
      if (lane < k) {
        const size_t aidx = (size_t)(t0 + tl) * k + lane;
        const int e = s_e[tl * k + lane];
        if (e < 0 || e >= E) {
          set_error(err, kDevCheck);
        } else {
          const int g = s_next[e]++;  // distinct experts within a token: no two lanes share e
          if (g < 0 || g >= T * k) {
            set_error(err, kDevCheck);
          } else {
            perm[g] = (int)aidx;
            pos[aidx] = g;
          }
        }
      }
      __syncwarp();
    }
  }
}

// Routing and dispatch in one cooperative launch of G CTAs (all co-resident; G
// is fixed per layer, so that the arrival counter grows by G every call and a
// call's generation is the counter / G), CTA b owning the S consecutive 32-token
// chunks [b*S, (b+1)*S) (none for the last CTAs when T is small):
//   1. top-k of each owned token (one warp per token), and per owned chunk a
//      32-bit token mask per expert in shared memory (bit t: the chunk's token t
//      chose e); the chunk's per-expert counts go to counts[c][e] as bytes.
//   2. one bounded grid barrier (arrival counter, every CTA adds 1 per call).
//   3. every CTA reads all counts and forms, per expert, the total and the rows
//      of the chunks before its own; an exclusive scan over experts gives the
//      grouped-row offsets. CTA 0 writes hist, offsets and the 128-row block map.
//   4. the grouped row of assignment (t, j) with expert e is offsets[e] + the
//      rows of e in earlier chunks + the tokens of its own chunk before t that
//      chose e (a population count of the mask): all assignments at once.
// The result is the same as that of the three kernels above (grouped rows in
// increasing token order within each expert); only the launch count differs.
__global__ void __launch_bounds__(1024, 1)
route_dispatch_kernel(const float* __restrict__ logits, int T, int E, int k, int S, int* __restrict__ idx,
                      float* __restrict__ weights, uint8_t* __restrict__ counts /* [chunks][E] */,
                      unsigned long long* __restrict__ ctr, int* __restrict__ hist, int* __restrict__ offsets,
                      int2* __restrict__ mtiles, int* __restrict__ num_routed, int max_mtiles,
                      int* __restrict__ perm, int* __restrict__ pos, int* __restrict__ err) {
  extern __shared__ uint32_t s_dyn[];
  uint32_t* s_mask = s_dyn;                        // [S][E]
  int* s_red = reinterpret_cast<int*>(s_dyn + S * E);   // [2][4096]: per-part totals, rows before
  __shared__ int s_pre[kMaxExperts];               // rows of e before the current chunk
  __shared__ int s_tot[kMaxExperts];               // rows of e in all chunks, then exclusive offsets
  __shared__ int s_wsum[2][32];
  __shared__ int s_ok;
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunks = (T + kChunk - 1) / kChunk;
  const int c0 = blockIdx.x * S, c1 = min(chunks, c0 + S);
  for (int q = tid; q < S * E; q += blockDim.x) s_mask[q] = 0u;
  for (int e = tid; e < E; e += blockDim.x) { s_pre[e] = 0; s_tot[e] = 0; }
  // after an earlier error (outputs undefined until the status is read) a CTA
  // only takes part in the barrier, so that the arrival counter stays whole
  if (tid == 0) s_ok = *reinterpret_cast<volatile int*>(err) == 0;
  __syncthreads();
  const bool live = s_ok != 0;
  // 1. top-k and the owned chunks' masks
  for (int c = live ? c0 : c1; c < c1; ++c) {
    const int t = c * kChunk + warp;
    if (t < T) {
      if (E <= 256) warp_topk<1>(logits + (size_t)t * E, E, k, lane, idx + (size_t)t * k, weights + (size_t)t * k);
      else warp_topk<2>(logits + (size_t)t * E, E, k, lane, idx + (size_t)t * k, weights + (size_t)t * k);
      __syncwarp();
      if (lane < k) {
        const int e = idx[(size_t)t * k + lane];
        if (e >= 0 && e < E) atomicOr(&s_mask[(c - c0) * E + e], 1u << warp);
        else set_error(err, kDevCheck);
      }
    }
  }
  __syncthreads();
  if (live)
    for (int q = tid; q < (c1 - c0) * E; q += blockDim.x) counts[(size_t)c0 * E + q] = (uint8_t)__popc(s_mask[q]);
  // 2. grid barrier
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned long long gen = atomicAdd(ctr, 1ull) / gridDim.x;
    const unsigned long long target = (gen + 1) * gridDim.x;
    const long long t0 = clock64();
    int ok = 1;
    unsigned long long v;
    do {
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if (clock64() - t0 > 4000000000LL) {  // ~2 s: something is wrong, do not hang the GPU
        set_error(err, kDevTimeout);
        ok = 0;
        break;
      }
    } while (true);
    __threadfence();
    s_ok = ok && live && *reinterpret_cast<volatile int*>(err) == 0;
  }
  __syncthreads();
  pdl_launch_dependents();
  if (!s_ok || (c0 >= c1 && blockIdx.x != 0)) return;
  // 3. per-expert totals and rows before this CTA's chunks; counts are read as
  //    4-expert words, P parts of the chunk range per word column, and the parts
  //    are added in part order (plain stores, no contended atomics)
  const int W = E / 4;                   // words per chunk row (E % 16 == 0)
  const int P = (int)blockDim.x / W;     // >= 2 for E <= 512; P * E <= 4096
  {
    const int part = tid / W, wcol = tid - part * W;
    if (part < P) {
      int pre[4] = {0, 0, 0, 0}, tot[4] = {0, 0, 0, 0};
      const uint32_t* cw = reinterpret_cast<const uint32_t*>(counts);
#pragma unroll 8
      for (int c = part; c < chunks; c += P) {
        const uint32_t v = __ldcg(cw + (size_t)c * W + wcol);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int n = (int)((v >> (8 * b)) & 0xFFu);
          tot[b] += n;
          if (c < c0) pre[b] += n;
        }
      }
      *reinterpret_cast<int4*>(s_red + part * E + 4 * wcol) = make_int4(tot[0], tot[1], tot[2], tot[3]);
      *reinterpret_cast<int4*>(s_red + 4096 + part * E + 4 * wcol) = make_int4(pre[0], pre[1], pre[2], pre[3]);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int tot = 0, pre = 0;
    for (int q = 0; q < P; ++q) {
      tot += s_red[q * E + e];
      pre += s_red[4096 + q * E + e];
    }
    s_tot[e] = tot;
    s_pre[e] = pre;
  }
  __syncthreads();
  // exclusive scans over experts of the rows and of the 128-row blocks
  {
    const int e = tid;
    const int n = e < E ? s_tot[e] : 0;
    const int nb = (n + BM - 1) / BM;
    int a = n, b = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xFFFFFFFFu, a, o), y = __shfl_up_sync(0xFFFFFFFFu, b, o);
      if (lane >= o) { a += x; b += y; }
    }
    if (lane == 31) { s_wsum[0][warp] = a; s_wsum[1][warp] = b; }
    __syncthreads();
    if (warp == 0) {
      int x = s_wsum[0][lane], y = s_wsum[1][lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int xs = __shfl_up_sync(0xFFFFFFFFu, x, o), ys = __shfl_up_sync(0xFFFFFFFFu, y, o);
        if (lane >= o) { x += xs; y += ys; }
      }
      s_wsum[0][lane] = x - s_wsum[0][lane];   // exclusive over warps
      s_wsum[1][lane] = y - s_wsum[1][lane];
    }
    __syncthreads();
    const int off = s_wsum[0][warp] + a - n, tile0 = s_wsum[1][warp] + b - nb;
    if (e < E) {
      s_tot[e] = off;
      if (blockIdx.x == 0) {
        hist[e] = n;
        offsets[e] = off;
        for (int m = 0; m < nb; ++m) {
          if (tile0 + m < max_mtiles) mtiles[tile0 + m] = make_int2(e, off + m * BM);
          else set_error(err, kDevCheck);
        }
        if (e == E - 1) {
          offsets[E] = off + n;   // == T * k
          *num_routed = tile0 + nb;
        }
      }
    }
  }
  __syncthreads();
  // 4. grouped rows of the owned chunks' assignments
  for (int c = c0; c < c1; ++c) {
    const uint32_t* mask = s_mask + (c - c0) * E;
    const int t = c * kChunk + (tid >> 5), j = lane;   // warp = token of the chunk, lane = slot
    if (t < T && j < k) {
      const size_t a = (size_t)t * k + j;
      const int e = idx[a];
      if (e >= 0 && e < E) {
        const int g = s_tot[e] + s_pre[e] + __popc(mask[e] & ((1u << (tid >> 5)) - 1u));
        if (g >= 0 && g < T * k) {
          perm[g] = (int)a;
          pos[a] = g;
        } else {
          set_error(err, kDevCheck);
        }
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) s_pre[e] += __popc(mask[e]);
    __syncthreads();
  }
}

// out[t, :] = sum_j w[t, j] * y[pos[t, j], :] + y_shared[t, :], fp32 sum, bf16 out.
__global__ void __launch_bounds__(256)
combine_kernel(const uint16_t* __restrict__ y, const uint16_t* __restrict__ ys, const int* __restrict__ pos,
               const float* __restrict__ w, int T, int H, int k, int has_shared, uint16_t* __restrict__ out,
               int* __restrict__ err) {
  pdl_wait();
  pdl_launch_dependents();
  const int chunks = H / 8;
  const size_t n = (size_t)T * chunks;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n; q += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(q / chunks), c = (int)(q % chunks);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    uint4 yv[kMaxTopK];
    float wt[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {  // issue all row loads first
      wt[j] = 0.f;
      if (j < k) {
        const int r = pos[(size_t)t * k + j];
        if (r < 0 || r >= T * k) {
          set_error(err, kDevCheck);
        } else {
          wt[j] = w[(size_t)t * k + j];
          yv[j] = *reinterpret_cast<const uint4*>(y + (size_t)r * H + 8 * c);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {  // then add them in j order
      if (j < k && wt[j] != 0.f) {
        const uint4 v = yv[j];
        const float wtj = wt[j];
        acc[0] = fmaf(wtj, bf16_lo(v.x), acc[0]); acc[1] = fmaf(wtj, bf16_hi(v.x), acc[1]);
        acc[2] = fmaf(wtj, bf16_lo(v.y), acc[2]); acc[3] = fmaf(wtj, bf16_hi(v.y), acc[3]);
        acc[4] = fmaf(wtj, bf16_lo(v.z), acc[4]); acc[5] = fmaf(wtj, bf16_hi(v.z), acc[5]);
        acc[6] = fmaf(wtj, bf16_lo(v.w), acc[6]); acc[7] = fmaf(wtj, bf16_hi(v.w), acc[7]);
      }
    }
    if (has_shared) {
      const uint4 v = *reinterpret_cast<const uint4*>(ys + (size_t)t * H + 8 * c);
      acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x); acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
      acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z); acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
    }
    uint4 o;
    o.x = (uint32_t)f32_to_bf16_rne(acc[0]) | ((uint32_t)f32_to_bf16_rne(acc[1]) << 16);
    o.y = (uint32_t)f32_to_bf16_rne(acc[2]) | ((uint32_t)f32_to_bf16_rne(acc[3]) << 16);
    o.z = (uint32_t)f32_to_bf16_rne(acc[4]) | ((uint32_t)f32_to_bf16_rne(acc[5]) << 16);
    o.w = (uint32_t)f32_to_bf16_rne(acc[6]) | ((uint32_t)f32_to_bf16_rne(acc[7]) << 16);
    *reinterpret_cast<uint4*>(out + (size_t)t * H + 8 * c) = o;
  }
}

// x (bf16) -> f16 for the routed rows of MXFP4 layers (8 values a thread-step;
// exact for |x| in [2^-14, 65504], rounded to nearest even below).
__global__ void __launch_bounds__(256)
bf16_to_f16_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ y, size_t n8, int* __restrict__ err) {
  pdl_wait();
  pdl_launch_dependents();
  bool x_range = false;   // |x| above the f16 range: reported, never rounded to infinity silently
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n8; q += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[q];
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) x_range |= f16_overflows(bf16_lo(w4[i])) || f16_overflows(bf16_hi(w4[i]));
    reinterpret_cast<uint4*>(y)[q] =
        make_uint4(f32x2_to_f16x2(bf16_lo(v.x), bf16_hi(v.x)), f32x2_to_f16x2(bf16_lo(v.y), bf16_hi(v.y)),
                   f32x2_to_f16x2(bf16_lo(v.z), bf16_hi(v.z)), f32x2_to_f16x2(bf16_lo(v.w), bf16_hi(v.w)));
  }
  if (x_range) set_error(err, kDevCheck);
}

// Scale tables of an MXFP4 matrix for the grouped GEMMs. Rows are `row_bytes`
// apart, each K / 2 code bytes then K / 32 e8m0 scale bytes; `rpe` rows per
// expert. sref[row] = the row's largest scale byte; sc[e][kb][row in expert] =
// the scales of blocks 2kb (low byte) and 2kb + 1, so one stage's 256 rows are
// 512 contiguous bytes.
__global__ void mx_grouped_scales_kernel(const uint8_t* __restrict__ w, int64_t row_bytes, int K, int rpe,
                                         size_t rows, uint16_t* __restrict__ sc, uint8_t* __restrict__ sref) {
  const int nkb = K / 64;
  for (size_t row = blockIdx.x * (size_t)blockDim.x + threadIdx.x; row < rows; row += (size_t)gridDim.x * blockDim.x) {
    const uint8_t* s = w + row * row_bytes + K / 2;
    const size_t e = row / rpe, rr = row % rpe;
    uint32_t mx = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      const uint32_t a = s[2 * kb], b = s[2 * kb + 1];
      mx = max(mx, max(a, b));
      sc[(e * nkb + kb) * rpe + rr] = (uint16_t)(a | (b << 8));
    }
    sref[row] = (uint8_t)mx;
  }
}

// Per-stage (scale, bias) pairs of an int4 matrix for the grouped GEMMs: rows are
// `row_bytes` apart, each K / 2 code bytes then K / 64 (scale, bias) bf16 pairs;
// par[e][kb][row in expert] = the pair of group kb, so one stage's 256 rows are
// 1 KB contiguous.
__global__ void i4_grouped_params_kernel(const uint8_t* __restrict__ w, int64_t row_bytes, int K, int rpe,
                                         size_t rows, uint32_t* __restrict__ par) {
  const int nkb = K / 64;
  for (size_t row = blockIdx.x * (size_t)blockDim.x + threadIdx.x; row < rows; row += (size_t)gridDim.x * blockDim.x) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(w + row * row_bytes + K / 2);
    const size_t e = row / rpe, rr = row % rpe;
    for (int kb = 0; kb < nkb; ++kb) par[(e * nkb + kb) * rpe + rr] = src[kb];
  }
}

// ===========================================================================
// Host side
// ===========================================================================
struct GroupedMaps {
  CUtensorMap router_split;  // B router: [3E][H] bf16, box {64, BNr}
  CUtensorMap w_gu;          // B gate/up routed: [E*2I][H], box {64, 256}
                             // (MXFP4: code bytes [E*2I][row], box {32, 256})
  CUtensorMap ws_gu;         // B gate/up shared: [2Is][H], box {64, 256}
  CUtensorMap h;             // A down routed: [Tmax*k][I], box {64, 128}
  CUtensorMap hs;            // A down shared: [Tmax][Is], box {64, 128}
  CUtensorMap w_down;        // B down routed: [E*H][I], box {64, 256}
                             // (MXFP4: code bytes [E*H][row], box {32, 256})
  CUtensorMap ws_down;       // B down shared: [H][Is], box {64, 256}
                             // (record layout: see encode_rec_gu / encode_rec_down)
  int router_bn;
  bool b_rec;                // B of the bf16 GEMMs from the feature records
};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
  if (g_encode) return cudaSuccess;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
  g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  return cudaSuccess;
}

// 2-D bf16 map over a row-major [rows][cols] matrix, box {64 cols, box_rows rows},
// 128-byte swizzle, zero fill outside the matrix.
cudaError_t encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D map over bf16 feature records ([rows][rec_bytes], gate row then up row of H
// elements at the start of each): dims {H, 2, rows}, box {64, 2, 128}, so one
// stage lands as 256 rows of 128 bytes -- feature f's gate row, then its up row --
// with the 128-byte swizzle, exactly as the row layout's box {64, 256}.
cudaError_t encode_rec_gu(CUtensorMap* m, const void* base, uint64_t rows, uint64_t H, uint64_t rec_bytes) {
  cuuint64_t dims[3] = {H, 2, rows};
  cuuint64_t strides[2] = {H * 2, rec_bytes};
  cuuint32_t box[3] = {(cuuint32_t)BK, 2, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
// 2-D map over the records' down columns (H bf16 at byte 4H of each record):
// dims {H, rows}, box {64 outputs, 64 features}: a 64 x 64 MN-major block of B
// (64 K rows of 128 bytes, 128-byte swizzle).
cudaError_t encode_rec_down(CUtensorMap* m, const uint8_t* rec, uint64_t rows, uint64_t H, uint64_t rec_bytes) {
  cuuint64_t dims[2] = {H, rows};
  cuuint64_t strides[1] = {rec_bytes};
  cuuint32_t box[2] = {64, (cuuint32_t)BK};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t*>(rec + 4 * H), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D byte map over [rows][row_bytes] (MXFP4 code rows), box {32 bytes, 256 rows},
// no swizzle: one stage's codes land as 256 dense 32-byte rows.
cudaError_t encode_codes(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes) {
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(BK / 2), 256};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <class K, class... A>
cudaError_t launch_pdl(K kernel, int grid, int block, size_t smem, cudaStream_t s, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The same with all CTAs co-resident (they wait on one another).
template <class K, class... A>
cudaError_t launch_coop_pdl(K kernel, int grid, int block, size_t smem, cudaStream_t s, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

cudaError_t grouped_prepare(moe_layer* L) {
  const auto& c = L->cfg;
  auto& g = L->grp;
  const int Tm = c.max_tokens, k = c.top_k, E = c.num_experts, H = c.hidden, I = c.intermediate,
            Is = c.shared_intermediate;
  memset(&g, 0, sizeof(g));
  g.max_tokens = Tm;
  const int chunks = (Tm + kChunk - 1) / kChunk;
  g.max_tiles = (Tm * k + BM - 1) / BM + E + 1;
  const size_t TK = (size_t)Tm * k;
  cudaError_t e;
#define GALLOC(ptr, bytes)                                                    \
  do {                                                                        \
    e = cudaMalloc((void**)&(ptr), (bytes) ? (bytes) : 16);                   \
    if (e != cudaSuccess) return e;                                           \
    L->mem_workspace_bytes += (int64_t)((bytes) ? (bytes) : 16);              \
  } while (0)
  GALLOC(g.logits, sizeof(float) * (size_t)Tm * E);
  GALLOC(g.idx, sizeof(int) * TK);
  GALLOC(g.weights, sizeof(float) * TK);
  GALLOC(g.hist, sizeof(int) * (E + 1));
  GALLOC(g.offsets, sizeof(int) * (E + 2));
  GALLOC(g.chunk_counts, sizeof(int) * (size_t)chunks * E);
  GALLOC(g.dispatch_ctr, sizeof(unsigned long long));
  g.dispatch_grid = chunks < L->num_sms ? chunks : L->num_sms;
  if ((e = cudaMemset(g.dispatch_ctr, 0, sizeof(unsigned long long))) != cudaSuccess) return e;
  GALLOC(g.perm, sizeof(int) * TK);
  GALLOC(g.pos, sizeof(int) * TK);
  GALLOC(g.tiles, sizeof(int2) * g.max_tiles);
  GALLOC(g.num_tiles, sizeof(int) * 4);
  GALLOC(g.h, sizeof(uint16_t) * TK * I);
  GALLOC(g.hs, sizeof(uint16_t) * (size_t)Tm * (Is > 0 ? Is : 1));
  GALLOC(g.y, sizeof(uint16_t) * TK * H);
  GALLOC(g.ys, sizeof(uint16_t) * (size_t)Tm * H);
  const bool mx = c.weight_format == MOE_WEIGHTS_MXFP4;
  const bool i4 = c.weight_format == MOE_WEIGHTS_INT4;
  if (i4) {
    GALLOC(g.x16, sizeof(uint16_t) * (size_t)Tm * H);
    GALLOC(g.i4_gu_par, sizeof(uint32_t) * (size_t)E * (H / 64) * 2 * I);
    GALLOC(g.i4_dn_par, sizeof(uint32_t) * (size_t)E * (I / 64) * H);
    i4_grouped_params_kernel<<<1024, 256>>>(L->w_gu, L->row_bytes.gu, H, 2 * I, (size_t)E * 2 * I, g.i4_gu_par);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    i4_grouped_params_kernel<<<1024, 256>>>(L->w_down, L->row_bytes.down, I, H, (size_t)E * H, g.i4_dn_par);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (mx) {
    GALLOC(g.x16, sizeof(uint16_t) * (size_t)Tm * H);
    GALLOC(g.mx_gu_sc, sizeof(uint16_t) * (size_t)E * (H / 64) * 2 * I);
    GALLOC(g.mx_dn_sc, sizeof(uint16_t) * (size_t)E * (I / 64) * H);
    GALLOC(g.mx_gu_sref, (size_t)E * 2 * I);
    GALLOC(g.mx_dn_sref, (size_t)E * H);
    mx_grouped_scales_kernel<<<1024, 256>>>(L->w_gu, L->row_bytes.gu, H, 2 * I, (size_t)E * 2 * I, g.mx_gu_sc,
                                            g.mx_gu_sref);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mx_grouped_scales_kernel<<<1024, 256>>>(L->w_down, L->row_bytes.down, I, H, (size_t)E * H, g.mx_dn_sc,
                                            g.mx_dn_sref);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
#undef GALLOC
  {  // the per-stage scale / (s, b) tables are weights, not workspace
    const int64_t blocks = (int64_t)E * (H / 64) * 2 * I + (int64_t)E * (I / 64) * H;
    const int64_t tables = i4 ? 4 * blocks : mx ? 2 * blocks + (int64_t)E * 2 * I + (int64_t)E * H : 0;
    L->mem_workspace_bytes -= tables;
    L->mem_weight_bytes += tables;
  }

  if ((e = get_encoder()) != cudaSuccess) return e;
  GroupedMaps* m = new GroupedMaps();
  L->tmaps = m;
  m->router_bn = (E % 64 == 0) ? 64 : (E % 32 == 0 ? 32 : 16);  // N tile dividing E (E % 16 == 0)
  if ((e = encode_2d(&m->router_split, L->router_split, 3ull * E, H, m->router_bn)) != cudaSuccess) return e;
  if ((e = encode_2d(&m->h, g.h, TK, I, BM)) != cudaSuccess) return e;
  m->b_rec = !mx && !i4 && L->w_gu == nullptr;   // bf16 layers that keep only the feature records
  const uint64_t rec_bytes = (uint64_t)stream_record_stride(H);
  if (m->b_rec) {
    if (!L->w_rec || (Is > 0 && !L->ws_rec)) return cudaErrorInvalidValue;
    if ((e = encode_rec_gu(&m->w_gu, L->w_rec, (uint64_t)E * I, H, rec_bytes)) != cudaSuccess) return e;
    if ((e = encode_rec_down(&m->w_down, L->w_rec, (uint64_t)E * I, H, rec_bytes)) != cudaSuccess) return e;
  } else if (!mx && !i4) {
    if ((e = encode_2d(&m->w_gu, L->w_gu, (uint64_t)E * 2 * I, H, 256)) != cudaSuccess) return e;
    if ((e = encode_2d(&m->w_down, L->w_down, (uint64_t)E * H, I, 256)) != cudaSuccess) return e;
  } else {
    if ((e = encode_codes(&m->w_gu, L->w_gu, (uint64_t)E * 2 * I, (uint64_t)L->row_bytes.gu)) != cudaSuccess) return e;
    if ((e = encode_codes(&m->w_down, L->w_down, (uint64_t)E * H, (uint64_t)L->row_bytes.down)) != cudaSuccess)
      return e;
  }
  if (Is > 0 && m->b_rec) {
    if ((e = encode_rec_gu(&m->ws_gu, L->ws_rec, (uint64_t)Is, H, rec_bytes)) != cudaSuccess) return e;
    if ((e = encode_2d(&m->hs, g.hs, (uint64_t)Tm, Is, BM)) != cudaSuccess) return e;
    if ((e = encode_rec_down(&m->ws_down, L->ws_rec, (uint64_t)Is, H, rec_bytes)) != cudaSuccess) return e;
  } else if (Is > 0) {
    if ((e = encode_2d(&m->ws_gu, L->ws_gu, 2ull * Is, H, 256)) != cudaSuccess) return e;
    if ((e = encode_2d(&m->hs, g.hs, (uint64_t)Tm, Is, BM)) != cudaSuccess) return e;
    if ((e = encode_2d(&m->ws_down, L->ws_down, (uint64_t)H, Is, 256)) != cudaSuccess) return e;
  } else {
    m->ws_gu = m->w_gu;
    m->hs = m->h;
    m->ws_down = m->w_down;
  }
  constexpr auto kSmemAttr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  e = cudaFuncSetAttribute(route_dispatch_kernel, kSmemAttr, (int)kDispatchMaskSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI_ROUTER, false, B_BF16>, kSmemAttr, (int)kGemmSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI_SWIGLU, true, B_BF16>, kSmemAttr, (int)kGemmSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI_STORE, false, B_BF16>, kSmemAttr, (int)kGemmSmem);
  if (e == cudaSuccess && mx)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI_SWIGLU, true, B_MXFP4>, kSmemAttr, (int)kGemmSmemMx);
  if (e == cudaSuccess && mx)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI_STORE, false, B_MXFP4>, kSmemAttr, (int)kGemmSmemMx);
  if (e == cudaSuccess && i4)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI_SWIGLU, true, B_INT4>, kSmemAttr, (int)kGemmSmemMx);
  if (e == cudaSuccess && i4)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI_STORE, false, B_INT4>, kSmemAttr, (int)kGemmSmemMx);
  return e;
}

void grouped_release(moe_layer* L) {
  auto& g = L->grp;
  void* ptrs[] = {g.logits, g.idx, g.weights, g.hist, g.offsets, g.chunk_counts, g.dispatch_ctr, g.perm, g.pos,
                  g.tiles, g.num_tiles, g.h, g.hs, g.y, g.ys, g.x16, g.mx_gu_sc, g.mx_dn_sc, g.i4_gu_par, g.i4_dn_par,
                  g.mx_gu_sref, g.mx_dn_sref};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  memset(&g, 0, sizeof(g));
  delete reinterpret_cast<GroupedMaps*>(L->tmaps);
  L->tmaps = nullptr;
}

cudaError_t launch_grouped(moe_layer* L, const uint16_t* x, uint16_t* out, int T, const float* logit_bias,
                           cudaStream_t s) {
  const auto& c = L->cfg;
  auto& g = L->grp;
  GroupedMaps* m = reinterpret_cast<GroupedMaps*>(L->tmaps);
  const int E = c.num_experts, k = c.top_k, H = c.hidden, I = c.intermediate, Is = c.shared_intermediate;
  const int mt_tokens = (T + BM - 1) / BM;
  const int chunks = (T + kChunk - 1) / kChunk;
  cudaError_t e;

  CUtensorMap map_x;
  if ((e = encode_2d(&map_x, x, (uint64_t)T, H, BM)) != cudaSuccess) return e;

  GemmParams base;
  memset(&base, 0, sizeof(base));
  base.E = E; base.T = T; base.k = k; base.H = H; base.err = L->err; base.max_mtiles = g.max_tiles;
  const bool mx = c.weight_format == MOE_WEIGHTS_MXFP4;
  const bool i4 = c.weight_format == MOE_WEIGHTS_INT4;

  // 1. router logits (tensor cores, exact 3-term split of W_r); MXFP4 layers
  //    first convert x to f16 for the routed gate/up rows.
  prof_mark(L, s);
  if (mx || i4) {
    const size_t n8 = (size_t)T * H / 8;
    int grid = (int)((n8 + 255) / 256);
    if (grid > 4 * L->num_sms) grid = 4 * L->num_sms;
    e = launch_pdl(bf16_to_f16_kernel, grid, 256, 0, s, x, g.x16, n8, L->err);
    if (e != cudaSuccess) return e;
  }
  {
    GemmParams p = base;
    p.mtiles = nullptr; p.num_routed = nullptr;
    p.BN = m->router_bn;
    p.n_routed_static = mt_tokens; p.nt_routed = E / p.BN; p.ks_part = H / BK; p.ks_routed = H / BK;
    p.n_shared_mtiles = 0; p.nt_shared = 1; p.ks_shared = 0;
    p.logits = g.logits; p.router_bias = L->router_bias; p.logit_bias = logit_bias;
    const int tiles = mt_tokens * p.nt_routed;
    e = launch_pdl(grouped_gemm_kernel<EPI_ROUTER, false, B_BF16>, tiles < L->num_sms ? tiles : L->num_sms, 192,
                   kGemmSmem, s, map_x, map_x, m->router_split, m->router_split, p);
    if (e != cudaSuccess) return e;
  }
  prof_mark(L, s);
  // 2-4. top-k, histogram, scan, block map, scatter: one cooperative launch
  //      while the owned chunks' masks fit in shared memory, else three kernels
  const int G = g.dispatch_grid, S = (chunks + G - 1) / G;
  const size_t mask_smem = sizeof(uint32_t) * (size_t)S * E + kDispatchRedSmem;
  if (T > 0 && mask_smem <= kDispatchMaskSmem) {
    e = launch_coop_pdl(route_dispatch_kernel, G, 1024, mask_smem, s, (const float*)g.logits, T, E, k, S, g.idx,
                        g.weights, reinterpret_cast<uint8_t*>(g.chunk_counts), g.dispatch_ctr, g.hist, g.offsets,
                        (int2*)g.tiles, g.num_tiles, g.max_tiles, g.perm, g.pos, L->err);
    if (e != cudaSuccess) return e;
  } else {
    e = launch_pdl(topk_hist_kernel, chunks, 1024, 0, s, (const float*)g.logits, T, E, k, g.idx, g.weights,
                   g.chunk_counts);
    if (e != cudaSuccess) return e;
    e = launch_pdl(dispatch_scan_kernel, 1, 1024, 0, s, g.chunk_counts, chunks, E, T, k, g.hist, g.offsets,
                   (int2*)g.tiles, g.num_tiles, g.max_tiles, L->err);
    if (e != cudaSuccess) return e;
    e = launch_pdl(dispatch_scatter_kernel, chunks, 256, 0, s, (const int*)g.idx, (const int*)g.chunk_counts,
                   (const int*)g.offsets, T, E, k, g.perm, g.pos, L->err);
    if (e != cudaSuccess) return e;
  }
  prof_mark(L, s);
  // 5. gate/up + SwiGLU (routed groups, then the shared expert over all tokens)
  {
    GemmParams p = base;
    p.mtiles = (const int2*)g.tiles; p.num_routed = g.num_tiles; p.offsets = g.offsets;
    p.BN = 256;
    p.nt_routed = 2 * I / 256; p.ks_routed = H / BK;
    p.n_shared_mtiles = Is > 0 ? mt_tokens : 0; p.nt_shared = Is > 0 ? 2 * Is / 256 : 1; p.ks_shared = H / BK;
    p.x = x; p.perm = g.perm; p.b_rows_per_expert = 2 * I; p.b_rec = m->b_rec ? I : 0;
    p.out_routed = g.h; p.ld_routed = I; p.out_shared = g.hs; p.ld_shared = Is;
    if (mx) {
      p.x16 = g.x16; p.q_par = g.mx_gu_sc; p.mx_sref = g.mx_gu_sref;
      e = launch_pdl(grouped_gemm_kernel<EPI_SWIGLU, true, B_MXFP4>, L->num_sms, 320 + kConvThreads, kGemmSmemMx, s,
                     map_x, map_x, m->w_gu, m->ws_gu, p);
    } else if (i4) {
      p.x16 = g.x16; p.q_par = g.i4_gu_par;
      e = launch_pdl(grouped_gemm_kernel<EPI_SWIGLU, true, B_INT4>, L->num_sms, 320 + kConvThreads, kGemmSmemMx, s,
                     map_x, map_x, m->w_gu, m->ws_gu, p);
    } else {
      e = launch_pdl(grouped_gemm_kernel<EPI_SWIGLU, true, B_BF16>, L->num_sms, 320, kGemmSmem, s, map_x, map_x,
                     m->w_gu, m->ws_gu, p);
    }
    if (e != cudaSuccess) return e;
  }
  prof_mark(L, s);
  // 6. down projection (routed groups + shared)
  {
    GemmParams p = base;
    p.mtiles = (const int2*)g.tiles; p.num_routed = g.num_tiles; p.offsets = g.offsets;
    p.BN = 256;
    p.nt_routed = H / 256; p.ks_routed = I / BK;
    p.n_shared_mtiles = Is > 0 ? mt_tokens : 0; p.nt_shared = H / 256; p.ks_shared = Is > 0 ? Is / BK : 1;
    p.b_rows_per_expert = H; p.b_rec = m->b_rec ? I : 0;
    p.out_routed = g.y; p.ld_routed = H; p.out_shared = g.ys; p.ld_shared = H;
    if (mx) {
      p.q_par = g.mx_dn_sc; p.mx_sref = g.mx_dn_sref;
      e = launch_pdl(grouped_gemm_kernel<EPI_STORE, false, B_MXFP4>, L->num_sms, 192 + kConvThreads, kGemmSmemMx, s,
                     m->h, m->hs, m->w_down, m->ws_down, p);
    } else if (i4) {
      p.q_par = g.i4_dn_par;
      e = launch_pdl(grouped_gemm_kernel<EPI_STORE, false, B_INT4>, L->num_sms, 192 + kConvThreads, kGemmSmemMx, s,
                     m->h, m->hs, m->w_down, m->ws_down, p);
    } else {
      e = launch_pdl(grouped_gemm_kernel<EPI_STORE, false, B_BF16>, L->num_sms, 192, kGemmSmem, s, m->h, m->hs,
                     m->w_down, m->ws_down, p);
    }
    if (e != cudaSuccess) return e;
  }
  prof_mark(L, s);
  // 7. weighted combine
  {
    const size_t n = (size_t)T * (H / 8);
    int grid = (int)((n + 255) / 256);
    if (grid > 8 * L->num_sms) grid = 8 * L->num_sms;
    e = launch_pdl(combine_kernel, grid, 256, 0, s, (const uint16_t*)g.y, (const uint16_t*)g.ys,
                   (const int*)g.pos, (const float*)g.weights, T, H, k, Is > 0 ? 1 : 0, out, L->err);
    if (e != cudaSuccess) return e;
  }
  prof_mark(L, s);
  return cudaSuccess;
}

}  // namespace moe
