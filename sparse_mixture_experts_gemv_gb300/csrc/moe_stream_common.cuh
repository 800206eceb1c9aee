// Pieces shared by the record-streaming decode kernels (bf16 experts in
// moe_stream.cu, MXFP4 experts in moe_stream_mx.cu): the CTA layout (16
// consumer warps + 1 producer warp), the router with tagged logits, the
// per-CTA top-k and slot list of a token window, the record ranges of a CTA,
// and the exchange that adds the CTAs' partial outputs.
//
// Tagged words: a 64-bit global word {call tag (high 32 bits), fp32 value}
// written with one single-copy-atomic store. A reader that sees the current
// call's tag also sees the value written with it, so publishing data needs no
// fence and reading it needs no separate barrier. The tag of a call is
// (calls completed) + 1, where calls completed = ctr / G and every CTA adds 1
// to ctr when it leaves: no CTA leaves a call before it has read everything
// the other CTAs of that call publish, and every CTA reads ctr before it
// publishes anything.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_sm100.cuh"

namespace moe {
namespace stream {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;            // + one producer warp
constexpr int kMaxRingGroups = 16;
constexpr int kMaxRouterRows = 16;                   // router rows per CTA
constexpr long long kSpinBudget = 4000000000LL;      // ~2 s of SM cycles: then give up

MOE_DEV unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Same load without a compiler memory barrier, so that a batch of them can be
// issued back to back (each is still a single-copy-atomic relaxed load).
MOE_DEV unsigned long long ld_relaxed_u64_nc(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
MOE_DEV void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
MOE_DEV unsigned long long tagged(unsigned long long tag, float v) {
  return (tag << 32) | (unsigned long long)__float_as_uint(v);
}
// Barrier among the 16 consumer warps only (the producer warp never joins it).
MOE_DEV void consumers_sync() { asm volatile("bar.sync 1, %0;" :: "n"(kConsumers) : "memory"); }
// Consumer barrier that also returns whether any consumer thread passed a true v.
MOE_DEV bool consumers_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r) : "r"((uint32_t)v), "n"(kConsumers) : "memory");
  return r != 0;
}

// Routing of the window, in shared memory.
struct RouteSmem {
  int idx[kMaxDecodeT * kMaxTopK];        // [t][j] selected experts, descending logits
  float w[kMaxDecodeT * kMaxTopK];        // [t][j] renormalised softmax weights
  int slot_of[kMaxDecodeT * kMaxTopK];    // scratch of the slot build
  unsigned tmask[kMaxSlots];              // tokens using each slot
  DecodeMeta meta;                        // slots: distinct experts, first-appearance order
};

// ---------------------------------------------------------------------------
// Warp-level tensor-core fragments (PTX ldmatrix / mma.sync).
// ---------------------------------------------------------------------------
MOE_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
MOE_DEV void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// D = A(16x16, row) * B(16x8, col) + D; bf16 inputs, fp32 accumulators.
MOE_DEV void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Same with f16 inputs.
MOE_DEV void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                           uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Fragment coordinates of a lane in an m16n8k16 tile: row group g = lane / 4,
// column pair c = lane % 4. C/D: rows g and g + 8, columns (tokens) 2c, 2c + 1.

// One warp's part of the gate/up tile of up to 8 bf16 records (rows 0-7 = gate
// rows of records 0-7, rows 8-15 = their up rows) at `gbase` (records `stride`
// bytes apart; records >= nvalid read the zero row): K = [k0, k0 + 16 * nsteps)
// of H against x (bf16, rows XP elements apart, tokens >= T read as zero).
// Returns the partial tile (fragment layout).
template <int MAXSTEPS>
MOE_DEV void bf16_gu_tile(uint32_t gbase, int stride, int nvalid, int H, int T, int XP, uint32_t xs_u32,
                          uint32_t zero_u32, int k0, int nsteps, float (&out)[4]) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
  const int q = lane >> 3, r = lane & 7;     // ldmatrix: lane supplies row r of matrix q
  const bool real = r < nvalid;
  const uint32_t rowaddr = real ? gbase + (uint32_t)(r * stride + ((q & 1) ? 2 * H : 0) + (q >> 1) * 16) : zero_u32;
  float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // even / odd k-steps
#pragma unroll
  for (int st = 0; st < MAXSTEPS; ++st) {
    if (st < nsteps) {
      const int kabs = k0 + 16 * st;
      uint32_t a0, a1, a2, a3;
      ldsm_x4(real ? rowaddr + 2 * kabs : zero_u32, a0, a1, a2, a3);
      uint32_t b0 = 0u, b1 = 0u;
      if (gq < T) {
        const uint32_t xa = xs_u32 + (uint32_t)(2 * (gq * XP + kabs + 2 * cq));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b0) : "r"(xa));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b1) : "r"(xa + 16));
      }
      mma_16816(d[st & 1], a0, a1, a2, a3, b0, b1);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) out[e] = d[0][e] + d[1][e];
}

// One warp's output tiles of the down projection of up to 8 bf16 records:
// acc[j] += sum_r down_r[n] * c[r][t] for tiles n0 = 16 * (warp + 16 j), with
// c given as bf16 hi + lo fragments (bhi, blo: c[2cq..2cq+1][token gq]). The
// down columns start 4H bytes into each record.
template <int MAXTILES>
MOE_DEV void bf16_down_tiles(uint32_t gbase, int stride, int nvalid, int H, int ntile, uint32_t zero_u32, uint32_t bhi,
                             uint32_t blo, float (&acc)[MAXTILES][4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane & 7, half = (lane >> 3) & 1;   // ldmatrix.x2: lanes 0-15 supply rows
  const bool real = r < nvalid;
  const uint32_t dbase = gbase + (uint32_t)(r * stride + 4 * H + half * 16);
#pragma unroll
  for (int j = 0; j < MAXTILES; ++j) {
    if (j < ntile) {
      const int n0 = 16 * (warp + kConsumerWarps * j);
      uint32_t a0, a1;
      ldsm_x2_trans(real ? dbase + 2 * n0 : zero_u32, a0, a1);
      // K = 16: records 0-7 against c_hi, the same records again against c_lo
      mma_16816(acc[j], a0, a1, a0, a1, bhi, blo);
    }
  }
}

// ---------------------------------------------------------------------------
// MXFP4 records on the tensor cores.
// ---------------------------------------------------------------------------
// Record layout (bytes; so = scale segment, pad16(H / 32)):
//   [0, H/2)        gate codes, shuffled per 32-element block (below)
//   [H/2, H)        up codes, shuffled the same way
//   [H, H+so)       gate scales, one e8m0 byte per 32-element block
//   [H+so, H+2so)   up scales
//   [H+2so, ...)    down column codes in 16-row tiles (below)
// Block shuffle: a 32-element block is 16 code bytes, byte j = elements 2j
// (low nibble), 2j+1. Stored word c (bytes 4c .. 4c+3) = original bytes c, c+4,
// c+8, c+12: exactly the four code pairs lane (g, c) of an m16n8k16 A fragment
// needs for one row over the block's two 16-wide k-steps (k = 2c, 2c+8 of the
// first step, then of the second).
// Down tiles, per pair of records (features 2p, 2p + 1; groups and CTA ranges
// start at even features): for 16-row tile t and g < 8, bytes 16t' + 2g and
// 16t' + 2g + 1 hold rows 16t + g and 16t + g + 8, each byte both features'
// codes of that row (feature 2p in the low nibble) -- the code pair lane (g, c)
// of an A fragment needs for K columns 2c, 2c + 1. Tiles t < H / 32 are in
// record 2p's column (t' = t), the rest in record 2p + 1's (t' = t - H / 32).
// The four code bytes of w (byte i = elements 2i, 2i+1) -> four f16x2, byte i
// in o[i]: one move splits the word into bytes, then one conversion each.
MOE_DEV void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}
// The two code bytes of the low half of w -> two f16x2.
MOE_DEV void e2m1x4_to_f16x2x2(uint32_t w, uint32_t& o0, uint32_t& o1) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %2;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n}"
      : "=r"(o0), "=r"(o1) : "r"(w));
}

struct MxLayout {
  int up_codes, gate_scales, up_scales, down_tiles;
};
MOE_DEV MxLayout mx_layout(int H, int so) { return MxLayout{H / 2, H, H + so, H + 2 * so}; }

// One warp's part of the gate/up tiles of up to 16 MXFP4 records (tile m:
// rows 0-7 = gate rows of records 8m .. 8m+7, rows 8-15 = their up rows), over
// 32-element blocks [blk0, blk0 + NBLK) of H. Each block's two k-steps go to a
// fresh accumulator that is then scaled by the row's block scale and added.
// x16: f16 x, rows XP halves apart. Records >= nvalid count as zero. UNROLL:
// how far the block loop is unrolled (one-token kernels roll it: their group
// code is fetched cold once per call and a short body wins there).
template <int MAXMT, int NBLK, int UNROLL = NBLK>
MOE_DEV void mx_gu_tiles(const uint8_t* gbase, int stride, int nvalid, int nmt, const MxLayout& ly, int T, int XP,
                         const uint16_t* x16, int blk0, float (&out)[MAXMT][4]) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
#pragma unroll
  for (int m = 0; m < MAXMT; ++m) out[m][0] = out[m][1] = out[m][2] = out[m][3] = 0.f;
#pragma unroll UNROLL
  for (int bi = 0; bi < NBLK; ++bi) {
    const int blk = blk0 + bi;
    uint32_t b[2][2] = {{0u, 0u}, {0u, 0u}};   // x fragments of the block's two k-steps
    if (gq < T) {
      const uint16_t* xr = x16 + gq * XP + 32 * blk + 2 * cq;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        b[ks][0] = *reinterpret_cast<const uint32_t*>(xr + 16 * ks);
        b[ks][1] = *reinterpret_cast<const uint32_t*>(xr + 16 * ks + 8);
      }
    }
#pragma unroll
    for (int m = 0; m < MAXMT; ++m) {
      if (m < nmt) {
        const int r = 8 * m + gq;
        uint32_t gw = 0u, uw = 0u;
        float gs = 0.f, us = 0.f;
        if (r < nvalid) {
          const uint8_t* rec = gbase + (size_t)r * stride;
          gw = *reinterpret_cast<const uint32_t*>(rec + 16 * blk + 4 * cq);
          uw = *reinterpret_cast<const uint32_t*>(rec + ly.up_codes + 16 * blk + 4 * cq);
          gs = e8m0_to_f32(rec[ly.gate_scales + blk]);
          us = e8m0_to_f32(rec[ly.up_scales + blk]);
        }
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t ga[4], ua[4];   // byte i of the words: k-step i / 2, k columns 2cq (i even) / 2cq + 8 (i odd)
        e2m1x8_to_f16x2x4(gw, ga);
        e2m1x8_to_f16x2x4(uw, ua);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          mma_16816_f16(d, ga[2 * ks], ua[2 * ks], ga[2 * ks + 1], ua[2 * ks + 1], b[ks][0], b[ks][1]);
        out[m][0] = fmaf(gs, d[0], out[m][0]);
        out[m][1] = fmaf(gs, d[1], out[m][1]);
        out[m][2] = fmaf(us, d[2], out[m][2]);
        out[m][3] = fmaf(us, d[3], out[m][3]);
      }
    }
  }
}

// One warp's output tiles of the down projection of up to 16 MXFP4 records
// (K = the records): acc[j] += sum_r code_r[n] * scale_v(r)[n] * c[r][t] for
// tiles n0 = 16 * (warp + 16 j), j < NTILE = H / 256. The records use one or two down-scale
// vectors (nv; sv0, sv1: H bytes, one per output row). For vector v, c comes
// as f16 fragments scaled by 2^-cexp, with c = 0 for the records of the other
// vector (bh[v][0..1]: c'[2cq..2cq+1][token gq], c'[2cq+8..2cq+9][gq]). The
// shift puts the group's largest |c'| in [2^14, 2^15), so every c keeps the
// f16 significand (relative error 2^-12, far inside the MXFP4 bound); A
// fragments are built once per tile for both vectors.
template <int NTILE>
MOE_DEV void mx_down_tiles(const uint8_t* gbase, int stride, int nvalid, const MxLayout& ly, int nv,
                           const uint8_t* sv0, const uint8_t* sv1, float cexp2, const uint32_t (&bh)[2][2],
                           float (&acc)[NTILE][4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, cq = lane & 3;
  // pairs cq (records 2cq, 2cq + 1: K columns 2cq, 2cq + 1) and cq + 4 (K columns 2cq + 8, 2cq + 9);
  // nvalid is even, so a pair is present or absent as a whole
  const uint8_t* pa = gbase + (size_t)(2 * cq) * stride + ly.down_tiles + 2 * gq;
  const uint8_t* pb = pa + (size_t)8 * stride;
  const bool va = 2 * cq < nvalid, vb = 2 * cq + 8 < nvalid;
#pragma unroll
  for (int j = 0; j < NTILE; ++j) {
    {
      const int tt = warp + kConsumerWarps * j, n0 = 16 * tt;
      // tiles tt < H / 32 = 8 NTILE (j < NTILE / 2) in the pair's first record, the rest in its second
      constexpr int kHalf = NTILE / 2;
      const int sel = j >= kHalf ? 1 : 0;
      const int off = sel * stride + 16 * (warp + kConsumerWarps * (j - sel * kHalf));
      const uint32_t ua = va ? *reinterpret_cast<const uint16_t*>(pa + off) : 0u;
      const uint32_t ub = vb ? *reinterpret_cast<const uint16_t*>(pb + off) : 0u;
      uint32_t a0, a1, a2, a3;
      e2m1x4_to_f16x2x2(ua, a0, a1);   // rows n0+g, n0+g+8
      e2m1x4_to_f16x2x2(ub, a2, a3);
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        if (v < nv) {
          const uint8_t* sv = v ? sv1 : sv0;
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_16816_f16(d, a0, a1, a2, a3, bh[v][0], bh[v][1]);
          const float f0 = e8m0_to_f32(sv[n0 + gq]) * cexp2, f1 = e8m0_to_f32(sv[n0 + gq + 8]) * cexp2;
          acc[j][0] = fmaf(f0, d[0], acc[j][0]);
          acc[j][1] = fmaf(f0, d[1], acc[j][1]);
          acc[j][2] = fmaf(f1, d[2], acc[j][2]);
          acc[j][3] = fmaf(f1, d[3], acc[j][3]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Groupwise affine int4 records on the tensor cores ("Optimizing on-device
// inference for Apple Silicon", section "Decode weights during matrix
// multiplication": 4-bit weights with a bf16 scale and bias per group of 64,
// value q * s + b, q unsigned). The record layout is the MXFP4 one (codes
// block-shuffled the same way, down columns in the same paired 16-row tiles);
// the scale segments hold one 4-byte (s, b) pair (s in the low half) per 64
// elements, and the down columns' pairs live in vectors of H pairs per
// (expert, 64 features). A dot product over a 32-element block is
// s * sum(q x) + b * sum(x): the tensor cores take q exactly as f16 integers,
// and sum(x) of every block and token is staged once per call.
// ---------------------------------------------------------------------------
// Two unsigned 4-bit codes of one byte (element 2i in the low nibble) -> f16x2,
// exact: 0x6400 | q is the f16 1024 + q, and 1024 is subtracted in f16.
MOE_DEV uint32_t u4x2_to_f16x2(uint32_t byte) {
  const uint32_t w = 0x64006400u | (byte & 0x0Fu) | ((byte & 0xF0u) << 12);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0x64006400u));
  return r;
}

// One warp's part of the gate/up tiles of up to 16 int4 records, as
// mx_gu_tiles: each block's two k-steps go to a fresh accumulator d, then
// out += s * d + b * sum(x of the block) per (row, token). xsum: fp32
// [token][block], tokens XSP floats apart.
template <int MAXMT, int NBLK>
MOE_DEV void i4_gu_tiles(const uint8_t* gbase, int stride, int nvalid, int nmt, const MxLayout& ly, int T, int XP,
                         const uint16_t* x16, const float* xsum, int XSP, int blk0, float (&out)[MAXMT][4]) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
#pragma unroll
  for (int m = 0; m < MAXMT; ++m) out[m][0] = out[m][1] = out[m][2] = out[m][3] = 0.f;
#pragma unroll 1   // rolled: keeps the int4 loop body in the instruction cache (measured faster)
  for (int bi = 0; bi < NBLK; ++bi) {
    const int blk = blk0 + bi;
    uint32_t b[2][2] = {{0u, 0u}, {0u, 0u}};
    if (gq < T) {
      const uint16_t* xr = x16 + gq * XP + 32 * blk + 2 * cq;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        b[ks][0] = *reinterpret_cast<const uint32_t*>(xr + 16 * ks);
        b[ks][1] = *reinterpret_cast<const uint32_t*>(xr + 16 * ks + 8);
      }
    }
    const float xs0 = 2 * cq < T ? xsum[(2 * cq) * XSP + blk] : 0.f;
    const float xs1 = 2 * cq + 1 < T ? xsum[(2 * cq + 1) * XSP + blk] : 0.f;
#pragma unroll
    for (int m = 0; m < MAXMT; ++m) {
      if (m < nmt) {
        const int r = 8 * m + gq;
        uint32_t gw = 0u, uw = 0u, gp = 0u, up = 0u;
        if (r < nvalid) {
          const uint8_t* rec = gbase + (size_t)r * stride;
          gw = *reinterpret_cast<const uint32_t*>(rec + 16 * blk + 4 * cq);
          uw = *reinterpret_cast<const uint32_t*>(rec + ly.up_codes + 16 * blk + 4 * cq);
          gp = *reinterpret_cast<const uint32_t*>(rec + ly.gate_scales + 4 * (blk >> 1));
          up = *reinterpret_cast<const uint32_t*>(rec + ly.up_scales + 4 * (blk >> 1));
        }
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          mma_16816_f16(d, u4x2_to_f16x2(gw >> (16 * ks)), u4x2_to_f16x2(uw >> (16 * ks)),
                        u4x2_to_f16x2(gw >> (16 * ks + 8)), u4x2_to_f16x2(uw >> (16 * ks + 8)), b[ks][0], b[ks][1]);
        const float gs = bf16_lo(gp), gb = bf16_hi(gp), us = bf16_lo(up), ub = bf16_hi(up);
        out[m][0] = fmaf(gs, d[0], fmaf(gb, xs0, out[m][0]));
        out[m][1] = fmaf(gs, d[1], fmaf(gb, xs1, out[m][1]));
        out[m][2] = fmaf(us, d[2], fmaf(ub, xs0, out[m][2]));
        out[m][3] = fmaf(us, d[3], fmaf(ub, xs1, out[m][3]));
      }
    }
  }
}

// Sums over the records of c' (the same B fragments as the down tiles): an mma
// against an all-ones A fragment, so each lane gets sum_r c'[r][2cq] and
// sum_r c'[r][2cq + 1].
MOE_DEV void colsum_f16(const uint32_t (&bh)[2], const uint32_t (&bl)[2], float& s0, float& s1) {
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  constexpr uint32_t one2 = 0x3C003C00u;   // f16 pair (1, 1)
  mma_16816_f16(d, one2, one2, one2, one2, bh[0], bh[1]);
  mma_16816_f16(d, one2, one2, one2, one2, bl[0], bl[1]);
  s0 = d[0];
  s1 = d[1];
}

// One warp's output tiles of the down projection of up to 16 int4 records, as
// mx_down_tiles: d = sum_r q[n][r] c'[r][t], then per row n of vector v,
// acc += s_n * 2^cexp * d + b_n * csum[v][t] (csum: the unscaled sums of c
// over the vector's records for tokens 2cq, 2cq + 1).
template <int NTILE>
MOE_DEV void i4_down_tiles(const uint8_t* gbase, int stride, int nvalid, const MxLayout& ly, int nv,
                           const uint32_t* pv0, const uint32_t* pv1, float cexp2, const uint32_t (&bh)[2][2],
                           const uint32_t (&bl)[2][2], const float (&csum)[2][2], float (&acc)[NTILE][4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, cq = lane & 3;
  const uint8_t* pa = gbase + (size_t)(2 * cq) * stride + ly.down_tiles + 2 * gq;
  const uint8_t* pb = pa + (size_t)8 * stride;
  const bool va = 2 * cq < nvalid, vb = 2 * cq + 8 < nvalid;
#pragma unroll
  for (int j = 0; j < NTILE; ++j) {
    const int tt = warp + kConsumerWarps * j, n0 = 16 * tt;
    constexpr int kHalf = NTILE / 2;
    const int sel = j >= kHalf ? 1 : 0;
    const int off = sel * stride + 16 * (warp + kConsumerWarps * (j - sel * kHalf));
    const uint32_t ua = va ? *reinterpret_cast<const uint16_t*>(pa + off) : 0u;
    const uint32_t ub = vb ? *reinterpret_cast<const uint16_t*>(pb + off) : 0u;
    const uint32_t a0 = u4x2_to_f16x2(ua);        // row n0+g
    const uint32_t a1 = u4x2_to_f16x2(ua >> 8);   // row n0+g+8
    const uint32_t a2 = u4x2_to_f16x2(ub);
    const uint32_t a3 = u4x2_to_f16x2(ub >> 8);
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      if (v < nv) {
        const uint32_t* pv = v ? pv1 : pv0;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816_f16(d, a0, a1, a2, a3, bh[v][0], bh[v][1]);
        mma_16816_f16(d, a0, a1, a2, a3, bl[v][0], bl[v][1]);
        const uint32_t p0 = pv[n0 + gq], p1 = pv[n0 + gq + 8];
        const float s0 = bf16_lo(p0) * cexp2, b0 = bf16_hi(p0), s1 = bf16_lo(p1) * cexp2, b1 = bf16_hi(p1);
        acc[j][0] = fmaf(s0, d[0], fmaf(b0, csum[v][0], acc[j][0]));
        acc[j][1] = fmaf(s0, d[1], fmaf(b0, csum[v][1], acc[j][1]));
        acc[j][2] = fmaf(s1, d[2], fmaf(b1, csum[v][0], acc[j][2]));
        acc[j][3] = fmaf(s1, d[3], fmaf(b1, csum[v][1], acc[j][3]));
      }
    }
  }
}

// c as an f16 hi + lo pair (packed with its neighbour) after scaling by s.
MOE_DEV void f16_hilo2(float c0, float c1, float s, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(c0 * s, c1 * s);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(c0 * s - hf.x, c1 * s - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
// c as a bf16 hi + lo pair (packed with its neighbour).
MOE_DEV void bf16_hilo2(float c0, float c1, uint32_t& hi, uint32_t& lo) {
  const uint16_t h0 = f32_to_bf16_rne(c0), h1 = f32_to_bf16_rne(c1);
  const uint16_t l0 = f32_to_bf16_rne(c0 - __uint_as_float((uint32_t)h0 << 16));
  const uint16_t l1 = f32_to_bf16_rne(c1 - __uint_as_float((uint32_t)h1 << 16));
  hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
  lo = (uint32_t)l0 | ((uint32_t)l1 << 16);
}

// Record range of this CTA. Shared-expert records [sh0, sh1) are known before
// routing; routed records [u0, u1) index the window's D x I (slot, feature)
// pairs. When there are at least G routed pairs the two ranges are balanced
// jointly (a CTA with one more shared record gets one fewer routed record).
// All counts fit 32 bits (U <= 64 slots x 4096 features, G < 1024), and only
// unsigned 32-bit division is used: 64-bit division is a long software
// sequence that would sit on the producer's critical path.
struct Ranges {
  int sh0, sh1;
  int u0, u1;
};
MOE_DEV Ranges cta_ranges(unsigned b, unsigned G, unsigned Is, unsigned U) {
  Ranges r;
  r.sh0 = (int)(b * Is / G);
  r.sh1 = (int)((b + 1) * Is / G);
  if (U >= G) {
    const unsigned N = U + Is;
    r.u0 = (int)(b * N / G) - r.sh0;
    r.u1 = (int)((b + 1) * N / G) - r.sh1;
  } else {
    r.u0 = (int)(b * U / G);
    r.u1 = (int)((b + 1) * U / G);
  }
  return r;
}

// Poll one token's E tagged logit words until all carry `tag`, then select its
// top-k (bounded: false after ~2 s without every word arriving).
template <int GK>
MOE_DEV bool poll_topk(const unsigned long long* words, int E, int k, unsigned long long tag, int lane, int* out_e,
                       float* out_w) {
  uint32_t key[GK][8];
  int jj[GK][8];
  const unsigned long long want = tag & 0xFFFFFFFFull;
  const long long t0 = clock64();
  bool ok = false;
  while (true) {
    unsigned long long w[GK][8];
#pragma unroll
    for (int g = 0; g < GK; ++g)   // every load in flight before any is used
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = lane + 32 * (8 * g + q);
        w[g][q] = (e < E) ? ld_relaxed_u64_nc(words + e) : (want << 32);
      }
    bool mine = true;
#pragma unroll
    for (int g = 0; g < GK; ++g)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = lane + 32 * (8 * g + q);
        mine &= (w[g][q] >> 32) == want;
        key[g][q] = (e < E) ? f32_order_key(__uint_as_float((uint32_t)w[g][q])) : 0u;
      }
    ok = __all_sync(0xFFFFFFFFu, mine);
    if (ok || clock64() - t0 > kSpinBudget) break;
  }
  warp_topk_keys<GK>(key, jj, k, lane, out_e, out_w);
  return ok;
}

// Consumer warps: this CTA's router logits (rows b, b + G, ... of the fp32
// router, at most kMaxRouterRows), split into parts over the 16 warps, summed
// in warp order, plus the router bias and the optional per-token logit bias,
// published as tagged words [t][E]. The number of parts P follows from the
// largest row count of any CTA, not from this CTA's own, so that every logit
// of the layer is the same sequence of fp32 operations: two experts with equal
// router columns get bitwise equal logits, and the exact-tie rule (lower index
// first) then decides between them. The row loads are issued before waiting
// for x (x_bar). Every consumer thread has waited on x_bar when this returns.
// When `rows_smem` is not null, the producer has bulk-copied this CTA's router
// rows there (row m at rows_smem + m * H, completing on x_bar with x): a bulk
// copy lands as soon as x does, while per-thread global loads of the rows
// arrived about a microsecond later on GB300.
template <int TMAX>
MOE_DEV void router_publish(const uint16_t* xs, int XP, int T, int H, int E, const float* router_t,
                            const float* router_bias, const float* logit_bias, unsigned long long* words,
                            unsigned long long tag, uint64_t* x_bar, int* err, int* s_abort,
                            float (*s_rpart)[TMAX], const float* rows_smem = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int nr_rows = (E - b + G - 1) / G;
  const int P = max(1, kConsumerWarps / ((E + G - 1) / G));   // warps per row, the same in every CTA
  const int items = nr_rows * P;
  const int H4 = H / 4;
  // the bias terms are loaded now, so that they do not add a memory round trip
  // after the dot products
  // The logits are stored by the last four consumer warps, never by the warps
  // that poll them in route_window (warps 0 .. T-1): a warp's first poll right
  // after its own store took 1.2-1.7 us on GB300, against ~0.2 us otherwise.
  const int pt = (int)threadIdx.x - (kConsumers - 128);   // nr_rows * T <= 128
  float rbias = 0.f, lbias = 0.f;
  if (pt >= 0 && pt < nr_rows * T) {
    const int m = pt / T, t = pt - m * T;
    const int e = b + m * G;
    rbias = router_bias[e];
    if (logit_bias) lbias = logit_bias[(size_t)t * E + e];
  }
  bool x_ready = false;
  if (warp < items) {
    const int m = warp / P, p = warp - m * P;
    const float* row = rows_smem ? rows_smem + (size_t)m * H : router_t + (size_t)(b + m * G) * H;
    const int c0 = p * H4 / P, c1 = (p + 1) * H4 / P;
    float acc[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
    // Column blocks of 32 lanes x QV 16-byte loads. One-token kernels take
    // QV = 2: this code runs once per call and is mostly fetched cold, so a short
    // body wins (GB300: Qwen-shaped T=1 -0.5 us, Ling-shaped -1.3 us); windows of
    // several tokens keep QV = 8, whose larger body holds more row loads in
    // flight when the rows come from global memory (QV = 2 cost Ling T=4 1.1 us).
    constexpr int QV = TMAX == 1 ? 2 : 8;
    for (int cb = c0; cb < c1; cb += 32 * QV) {
      uint4 v[QV];
      if (rows_smem && !x_ready) {   // the rows arrive with x
        volatile int never = 0;
        if (!sm100::mbar_wait(x_bar, 0, err, &never, kSpinBudget, false)) *s_abort = 1;
        x_ready = true;
      }
#pragma unroll
      for (int q = 0; q < QV; ++q) {
        const int c = cb + lane + 32 * q;
        if (c < c1) v[q] = rows_smem ? *reinterpret_cast<const uint4*>(row + 4 * c) : ldg_stream(row + 4 * c);
      }
      if (!x_ready) {
        volatile int never = 0;
        if (!sm100::mbar_wait(x_bar, 0, err, &never, kSpinBudget, false)) *s_abort = 1;
        x_ready = true;
      }
#pragma unroll
      for (int q = 0; q < QV; ++q) {
        const int c = cb + lane + 32 * q;
        if (c < c1) {
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (t < T) {
              const uint2 xx = *reinterpret_cast<const uint2*>(xs + t * XP + 4 * c);
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
        const float sum = warp_sum(acc[t]);
        if (lane == 0) s_rpart[warp][t] = sum;
      }
    }
  }
  if (!x_ready) {   // x is needed later by every warp
    volatile int never = 0;
    if (!sm100::mbar_wait(x_bar, 0, err, &never, kSpinBudget, false)) *s_abort = 1;
  }
  consumers_sync();
  if (pt >= 0 && pt < nr_rows * T) {   // logit = partial sums in warp order + biases
    const int m = pt / T, t = pt - m * T;
    const int e = b + m * G;
    float sl = 0.f;
    for (int p = 0; p < P; ++p) sl += s_rpart[m * P + p][t];
    sl += rbias;
    if (logit_bias) sl += lbias;
    st_relaxed_u64(words + (size_t)t * E + e, tagged(tag, sl));
  }
}

// Consumer warps: top-k of every token (warp t polls token t's logits), then
// warp 0 lists the distinct experts of the window in first-appearance order
// (slots) with, per slot, the position j of its expert in each token's top-k
// (-1 if the token did not choose it) and the mask of tokens using it.
// The caller synchronises the CTA before the slots are read.
MOE_DEV void route_window(const unsigned long long* words, int T, int E, int k, unsigned long long tag, RouteSmem& rs,
                          int* err, int* s_abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < T) {
    const int t = warp;
    bool ok;
    if (E <= 256) ok = poll_topk<1>(words + (size_t)t * E, E, k, tag, lane, rs.idx + t * k, rs.w + t * k);
    else ok = poll_topk<2>(words + (size_t)t * E, E, k, tag, lane, rs.idx + t * k, rs.w + t * k);
    if (!ok) {
      if (lane == 0) set_error(err, kDevTimeout);
      *s_abort = 1;
    }
  }
  if (T > 1) consumers_sync();
  if (warp != 0) return;
  if (T == 1) {   // one token: its k experts are the slots, in order
    if (lane < k) {
      const int e = rs.idx[lane];
      if (e < 0 || e >= E) {   // only NaN logits can get here
        set_error(err, kDevCheck);
        *s_abort = 1;
      }
      rs.meta.slot_expert[lane] = e;
      rs.tmask[lane] = 1u;
#pragma unroll
      for (int t = 0; t < kMaxDecodeT; ++t) rs.meta.slot_j[lane][t] = (signed char)(t == 0 ? lane : -1);
    }
    if (lane == 0) rs.meta.num_slots = k;
    return;
  }
  const int n = T * k;
  // assignment ai = lane + 32 h2; its expert's first position in the window:
  // __match_any_sync finds it among positions 0-31 (and, for h2 = 1, among
  // 32-63), a shuffle scan checks positions 0-31 for h2 = 1 (T * k > 32 only)
  int e2[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int ai = lane + 32 * h2;
    e2[h2] = ai < n ? rs.idx[ai] : -1 - ai;   // a value no other lane holds
    if (ai < n && (e2[h2] < 0 || e2[h2] >= E)) {
      set_error(err, kDevCheck);
      *s_abort = 1;
    }
  }
  bool first[2] = {false, false};
  int firstpos[2] = {0, 0};
  firstpos[0] = __ffs(__match_any_sync(0xFFFFFFFFu, e2[0])) - 1;
  first[0] = lane < n && firstpos[0] == lane;
  if (n > 32) {
    int pos = 32 + __ffs(__match_any_sync(0xFFFFFFFFu, e2[1])) - 1;
    for (int j = 31; j >= 0; --j)
      if (__shfl_sync(0xFFFFFFFFu, e2[0], j) == e2[1]) pos = j;
    firstpos[1] = pos;
    first[1] = lane + 32 < n && pos == lane + 32;
  }
  const unsigned m0 = __ballot_sync(0xFFFFFFFFu, first[0]);
  const unsigned m1 = __ballot_sync(0xFFFFFFFFu, first[1]);
  const unsigned lt = (1u << lane) - 1u;
  if (first[0]) rs.slot_of[lane] = __popc(m0 & lt);
  if (first[1]) rs.slot_of[lane + 32] = __popc(m0) + __popc(m1 & lt);
  __syncwarp();
  const int D = __popc(m0) + __popc(m1);
  for (int q = lane; q < D * kMaxDecodeT; q += 32) rs.meta.slot_j[q / kMaxDecodeT][q % kMaxDecodeT] = -1;
  for (int q = lane; q < D; q += 32) rs.tmask[q] = 0u;
  __syncwarp();
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int ai = lane + 32 * h2;
    if (ai < n) {
      const int slot = rs.slot_of[firstpos[h2]];
      if (first[h2]) rs.meta.slot_expert[slot] = rs.idx[ai];
      rs.meta.slot_j[slot][ai / k] = (signed char)(ai % k);
      atomicOr(&rs.tmask[slot], 1u << (ai / k));
    }
  }
  if (lane == 0) rs.meta.num_slots = D;
}

// ---------------------------------------------------------------------------
// Exchange of partial outputs. Every CTA holds fp32 partial sums of all H
// output rows over the records it streamed; the output is their sum over the
// G CTAs. CTA b reduces the rows [8 u0, 8 u1) of the 8-row units split evenly
// over the grid, for every token.
// ---------------------------------------------------------------------------
// Floats per output row in the partial buffer: T itself for one token, else T
// rounded up to even so that a token pair is one 8-byte store.
MOE_DEV int exchange_pitch(int T) { return T == 1 ? 1 : T + (T & 1); }

struct RowSlice {
  int n0, nrow;
};
MOE_DEV RowSlice exchange_rows(int b, int G, int H) {
  const unsigned U = (unsigned)H / 8u;
  const int u0 = (int)((unsigned)b * U / (unsigned)G), u1 = (int)((unsigned)(b + 1) * U / (unsigned)G);
  return {8 * u0, 8 * (u1 - u0)};
}

// ---------------------------------------------------------------------------
// Exchange with plain fp32 partials and one arrival counter. Each CTA stores
// its partial outputs as fp32, float (b, n, t) at (b * H + n) * TP + t, then
// makes them visible GPU-wide (fence) before it adds 1 to the arrival counter;
// one thread per CTA waits (acquire) until the counter shows every CTA of this
// call, and the CTA then pulls the rows [8 u0, 8 u1) of all G sources into
// shared memory in one pass of 16-byte L2 copies. (Publishing tagged 8-byte
// words and re-copying stale blocks until every tag was current moved twice
// the bytes and was ~1 us slower on GB300.) The counter only grows: this
// call's CTAs wait for `target` arrivals (calls before it included), and every
// CTA adds exactly 1 per call on every exit path.
//
// ONE_TOKEN = 1 compiles the one-token store alone. The 4-bit kernels use it
// for their one-token instances (0.4-0.5 us less per cold call, same-box A/B
// on GB300); the bf16 kernel keeps the run-time branch, which measured 0.3 us
// faster there.
// ---------------------------------------------------------------------------
template <int ONE_TOKEN = 0>
MOE_DEV void publish_tile_f32(float* partial, int b, int H, int T, int n0, const float (&acc)[4]) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
  const int TP = exchange_pitch(T);
  if (ONE_TOKEN || T == 1) {
    if (cq == 0) {
      partial[(size_t)b * H + n0 + gq] = acc[0];
      partial[(size_t)b * H + n0 + gq + 8] = acc[2];
    }
  } else if (!ONE_TOKEN && 2 * cq < T) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      *reinterpret_cast<float2*>(partial + ((size_t)b * H + n0 + gq + 8 * h) * TP + 2 * cq) =
          make_float2(acc[2 * h], acc[2 * h + 1]);
  }
}

MOE_DEV unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// This CTA's arrival after its partials are stored (consumer threads, after a
// consumer barrier; thread 0 only). Also used on the exit paths of a CTA that
// aborts, so that the others do not wait for it.
MOE_DEV void exchange_arrive(unsigned long long* arrivals) {
  __threadfence();
  atomicAdd(arrivals, 1ull);
}

// Consumer warps, after every warp of this CTA has stored its tiles with
// publish_tile_f32: arrive, wait for all G CTAs of this call, pull this CTA's
// rows of all G partials into `stage` (one pass; collect_f32_fits checks that
// it holds them), add the G values of each output in a fixed order (four
// threads per output, thread i over the sources [iG/4, (i+1)G/4), combined as
// (s0 + s1) + (s2 + s3)) and write bf16. Ends with a consumer barrier.
MOE_DEV void collect_outputs_f32(const float* partial, float* stage, unsigned long long* arrivals,
                                 unsigned long long target, int T, int H, uint16_t* out, int* err, int* s_abort) {
  const int G = gridDim.x, b = blockIdx.x;
  const int TP = exchange_pitch(T);
  const RowSlice rs = exchange_rows(b, G, H);
  const int blk = rs.nrow * TP;                       // floats of one source's block
  const unsigned bu = (unsigned)blk / 4u;             // 16-byte units of one block
  const int nout = rs.nrow * T;
  __threadfence();                                    // this thread's partials are visible GPU-wide
  consumers_sync();                                   // every warp's partials are stored
  if (threadIdx.x == 0) exchange_arrive(arrivals);
  // the arrivals are polled from another warp than the one that just added to
  // the counter (see router_publish: a warp's first poll after its own store is slow)
  if (threadIdx.x == 32) {
    const long long t0 = clock64();
    while (ld_acquire_u64(arrivals) < target) {
      if (clock64() - t0 > kSpinBudget) {
        set_error(err, kDevTimeout);
        *s_abort = 1;
        break;
      }
    }
    __threadfence();
  }
  consumers_sync();
  const bool aborted = *s_abort != 0;
  if (!aborted && nout > 0) {
    for (unsigned u = threadIdx.x; u < (unsigned)G * bu; u += kConsumers) {
      const unsigned q = u / bu, w = u - q * bu;
      sm100::cp_async_16(stage + (size_t)q * blk + 4 * w, partial + ((size_t)q * H + rs.n0) * TP + 4 * w, 16u);
    }
    sm100::cp_async_commit();
    sm100::cp_async_wait<0>();
    consumers_sync();
    // Four threads per output: thread i adds the sources [iG/4, (i+1)G/4) in
    // order (the loop is unrolled so that the loads overlap; consecutive
    // threads read neighbouring words of a source block, without bank
    // conflicts), then the four sums are combined as (s0 + s1) + (s2 + s3): the
    // same association on every call, so the result does not depend on timing.
    // (32 threads per output with a butterfly was slower: 16-way bank
    // conflicts on the staged blocks.)
    constexpr int kOut = 2;   // outputs per thread: 4 * nout <= kOut * kConsumers
    float sum[kOut] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < kOut; ++r) {
      const int o4 = (int)threadIdx.x + r * kConsumers;
      if (o4 < 4 * nout) {
        const int o = o4 >> 2, i = o4 & 3;
        const int nl = o / T, t = o - nl * T;
        const int p0 = (int)((unsigned)i * (unsigned)G / 4u), p1 = (int)((unsigned)(i + 1) * (unsigned)G / 4u);
        const float* src = stage + nl * TP + t;
        float acc = 0.f;
#pragma unroll 8
        for (int p = p0; p < p1; ++p) acc += src[(size_t)p * blk];
        sum[r] = acc;
      }
    }
#pragma unroll
    for (int r = 0; r < kOut; ++r) {
      const int o4 = (int)threadIdx.x + r * kConsumers;   // lanes 4o .. 4o + 3 share one output
      const float s0 = sum[r], s1 = __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
      const float lo = s0 + s1;                           // (s0 + s1) on lanes 4o, 4o + 1; (s2 + s3) on the others
      const float hi = __shfl_xor_sync(0xFFFFFFFFu, lo, 2);
      if (o4 < 4 * nout && (o4 & 3) == 0) {
        const int o = o4 >> 2, nl = o / T, t = o - nl * T;
        out[(size_t)t * H + rs.n0 + nl] = f32_to_bf16_rne(lo + hi);
      }
    }
  }
  consumers_sync();
}

// Whether the fp32 exchange can run: all G sources' blocks of this CTA's rows
// fit in one pass of `stage_bytes`, and four threads per output need at most
// two outputs per consumer thread.
inline bool collect_f32_fits(int G, int H, int T, size_t stage_bytes) {
  const int U = H / 8;
  const int nrow = 8 * ((U + G - 1) / G);
  const int TP = T == 1 ? 1 : T + (T & 1);
  return (size_t)G * nrow * TP * 4 <= stage_bytes && 4 * nrow * T <= 2 * kConsumers;
}

}  // namespace stream
}  // namespace moe
