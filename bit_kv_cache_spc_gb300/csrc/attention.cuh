// Attn([T_t, T'_{t+1}], C' U C_kappa): the two-query decode attention of the
// SpeCache page (section 3 "Decoding", Algorithm 3) over the packed low-bit
// copy C', with the fetched 16-bit rows C_kappa used in place of their
// low-bit copies, plus the bf16 residual window.
//
// This header holds the device code and the per-variant host helpers; each
// (bit width, group size) is instantiated in a translation unit of its own
// (attn_b1g32.cu, attn_b1g64.cu, attn_b2g32.cu, attn_b2g64.cu) and reached by
// the host code of attention.cu through an AttnVariant table.
//
// One launch per call, split-K over tokens (flash-decoding style):
//   * grid (chunks, B*Hkv).  The 16-bit rows of a (b, hkv) (residual window
//     first, then the fetched rows) are split into contiguous ranges over all
//     warps of its CTAs; every warp first reduces its range on CUDA cores,
//     while its first low-bit stages are already in flight, and the resulting
//     softmax state seeds its low-bit accumulators.  Then each warp scans its
//     share of the CTA's range of records of C' (a record holds one 32- or
//     64-token group; a 64-token record is processed as two 32-token halves
//     that share its key (min, max) table).
//   * every CTA merges its warps' states into one partial (running max, sum,
//     unnormalised output) per query row.  The partials are merged into the
//     bf16 output and the log-sum-exp by combine_kernel, launched right after
//     the grid; when all CTAs of a (b, hkv) form one resident thread-block
//     cluster they stay in shared memory and are merged through distributed
//     shared memory instead (cluster_combine); inside spc_decode_step the last
//     CTA of a (b, hkv) to finish (an atomic ticket) merges them.
//
// Low-bit tile arithmetic.  With k^ = z + s*b (b the code, z and s per key
// group), the logit of query row q is  sum_c q_c s_c b_c + sum_c q_c z_c.  The
// first term is a 16x8x16 tensor-core product per 8 tokens and 16 channels:
//   A = (q o s) for the 8 query rows (2 tokens x G <= 4 heads), split into an
//       fp16 high part (rows 0..7) and the fp16 residual (rows 8..15), so the
//       speculative logits keep ~22 significant bits;
//   B = the key bits, exact: each an fp16 power of two that depends only on
//       the token column (one AND of a rotated record word, see key_frag),
//       divided out of the logit per column; the high plane at 2 bits
//       multiplies a doubled A.
// The value side o = sum_n p_n (z_n + s_n b_n) is the same product with
// A = value bits (channels x tokens) and B = p o s (tokens x query rows); the
// p*z term is accumulated on CUDA cores.  Softmax runs in base 2 with the
// scale folded into q.  z and s of a group are computed once per warp into
// shared memory and read back by the lanes that need them.
#pragma once

#include <cooperative_groups.h>
#include <math_constants.h>

#include "common.cuh"
#include "select.cuh"

namespace spc {

// ---- tensor memory (TMEM) as on-chip storage of the speculative logits ----
// (spc_decode_step without a global spec_logits buffer).  A CTA allocates
// kTmemCols columns of its SM's tensor memory (128 lanes x 512 columns of 32
// bits); warp w may touch lanes 32 (w % 4) .. 32 (w % 4) + 31 only.
constexpr uint32_t kTmemCols = 128;
// One whole warp: allocate, write the base address to *smem_dst, and give up
// the right to allocate more (so that other CTAs on the SM can allocate).
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(smem_dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
// One whole warp (the allocating one), after every access has completed.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
// Lane l of the warp writes 4 consecutive columns of TMEM lane (taddr lane + l),
// waited for in the same statement (the source registers are then free).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, float4 v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)), "r"(__float_as_uint(v.w))
      : "memory");
}
// The matching read, waited for in the same statement (its registers are
// undefined until the wait).
__device__ __forceinline__ float4 tmem_ld4(uint32_t taddr) {
  uint32_t x, y, z, w;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(x), "=r"(y), "=r"(z), "=r"(w)
      : "r"(taddr)
      : "memory");
  return make_float4(__uint_as_float(x), __uint_as_float(y), __uint_as_float(z), __uint_as_float(w));
}
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
// At 1 bit the scaled query lives in registers across the low-bit loop; at 2
// bits (twice the code words per group) it is read from shared memory to
// keep the loop within the register budget of 4 CTAs per SM.
template <int BITS>
struct QueryInRegisters {
  static constexpr bool value = BITS == 1;
};
constexpr int kSlots = kWarps;  // CTA merge slots: one per warp
constexpr int kMaxCluster = 16;  // CTAs of one (b, hkv) that the clustered combine accepts
constexpr float kNeg = -1e30f;  // finite "minus infinity": keeps max/rescale arithmetic NaN-free
constexpr int kPartStride = 132; // floats per (cta, row) partial: m, l, pad, pad, o[128]
constexpr int kZsPitch = 17;     // float4s per t block of a z/s table (16 + 1 pad)
constexpr int kZsBytes = 2 * 4 * kZsPitch * 16;  // key and value tables of one warp
constexpr int kMergePitch = kD + 4;              // padded row of the CTA merge buffer
constexpr int kTilePitch = kD + 4;               // padded row of a warp's query / output transfer tile

// Record layout and pipeline of one (bit width, group size).  A record holds
// one group: 32 tokens at g = 32, 64 at g = 64 (two 32-token halves whose code
// planes follow one another, the group's key and value (min, max) once).
template <int BITS, int GROUP>
struct Layout {
  static constexpr int H = GROUP / 32;                                      // 32-token halves per record
  static constexpr int RB = GROUP == 32 ? 1024 * (BITS + 1) : 2048 * BITS + 1024;  // record bytes
  static constexpr int KMETA = 512 * BITS * H;                              // key (min, max) words
  static constexpr int VCODES = KMETA + 512;                                // value code planes
  static constexpr int VMETA = VCODES + 512 * BITS * H;                     // value (min, max) words
  static constexpr int STAGES = GROUP == 32 ? (BITS == 1 ? 4 : 3) : (BITS == 1 ? 3 : 2);  // per warp
  // a stage: the record, a 16-byte slot (bitmap words), 512 spare bytes (they keep the stages and the
  // z/s table large enough for the 16-bit-row prologue's batches of 16 rows)
  static constexpr int PFROW = RB + 16;
  static constexpr int STAGE = PFROW + 512;
  static constexpr int WARP_BYTES = STAGES * STAGE + kZsBytes;
  static constexpr int DYN = kWarps * WARP_BYTES;  // dynamic shared memory of one CTA
  // 16-bit rows staged per batch in a warp's stages after the first and its
  // z/s table: 16, or 8 when 16 padded rows do not fit
  static constexpr int TAIL = (STAGES - 1) * STAGE + kZsBytes;
  static constexpr int ROWB = TAIL >= 16 * (512 + 16) ? 16 : 8;
  static_assert(ROWB * (512 + 16) <= TAIL, "a row batch fits a warp's free stages");
  static_assert(RB % 512 == 0, "a record is streamed as whole 512-byte warp copies");
};

struct AttnArgs {
  const uint8_t* records;
  const uint16_t* resid;
  const uint16_t* q;
  const uint16_t* kv_self;  // [B][Hkv][2][D] bf16 or null: the speculative token's own key and value
  const int32_t* idx;
  const uint32_t* bitmap;
  const uint16_t* staging;
  float* spec_logits;
  float* part;          // [BH][chunks][kMaxRows][kPartStride]
  uint32_t* tickets;    // [BH], zero between calls
  uint16_t* out;        // [B][2][Hq][D]
  float* lse;           // [B][2][Hq] or null
  int32_t k;
  int32_t Hq, Hkv, G, nq, r, q_groups_cap, resid_cap;
  int32_t units_cap;  // records per (b, hkv): q_groups_cap at g = 32, (q_groups_cap + 1) / 2 at g = 64
  int32_t chunks, groups_per_chunk;
  int32_t Lcap;
  int32_t ext_combine;  // 1: the CTAs only store their partials; combine_kernel, launched next, merges them
  float qscale;  // softmax scale * log2(e)
  // Pre-fetch riding on this launch (spc_merged_attn_fetch): rows pf_idx of
  // the mapped host cache pf_host go to pf_staging; pf_rows = B*Hkv*pf_k.
  const uint16_t* pf_host;  // device address of [B][Hkv][pf_ncap][2][D] bf16, or null
  const int32_t* pf_idx;    // [B][Hkv][pf_k]
  uint16_t* pf_staging;     // [B][Hkv][pf_k][2][D]
  int64_t pf_ncap;
  int32_t pf_k, pf_rows;
  // Rows still staged from the previous selection: pf_src[rr] >= 0 is the
  // row's slot in pf_prev ([B][Hkv][pf_prev_k][2][D], device), whose copy
  // replaces the host read; null when every row comes from the host.
  const int32_t* pf_src;
  const uint16_t* pf_prev;
  int32_t pf_prev_k;
  // Fused ArgTopK (spc_decode_step): per (b, hkv) the sel_k positions with the
  // largest speculative probability go to sel_idx / sel_bitmap.  ready and
  // tickets2 are per-(b, hkv) words (zero between calls); cand holds each
  // chunk's candidates (key, position), cand_cap per chunk; fault is set when
  // a wait ran out.
  int32_t* sel_idx;       // [BH][sel_k]
  int32_t* sel_src;       // [BH][sel_k] or null: each selected position's index in idx (the previous selection)
  uint32_t* sel_bitmap;   // [BH][q_groups_cap]
  uint32_t* ready;
  uint32_t* tickets2;
  uint32_t* fault;
  uint32_t* cand;         // [BH][chunks][cand_cap][2]
  int32_t sel_k, sel_keff, cand_cap;
  // On-chip selection (spec_logits == nullptr): the speculative logits stay in
  // TMEM; the fetched rows' logits go to sel_rowlog [BH][k][4] instead.
  int32_t sel_onchip;
  float* sel_rowlog;
};

// A lone set bit at position p of an fp16 half (p = 10..14, the exponent
// field) is the power of two 2^(2^(p-10) - 15); pos_comp(p) is its inverse.
__host__ __device__ constexpr float pos_comp(int p) {
  return p == 10 ? 16384.f : p == 11 ? 8192.f : p == 12 ? 2048.f : p == 13 ? 128.f : 0.5f;
}

// Key bits.  Record word j of lane (gid, t) holds, for token 8 nt + gid and
// channel pair e = 4j + i (channels 16 (e >> 1) + 8 (e & 1) + 2t + {0, 1}),
// the two bits that a left rotation by 4i brings to bits 11 + nt and 27 + nt:
// so one AND of the rotated word is the B fragment {0, 2^-13 .. 2} of token
// column nt, the same power of two for all its channels, which the logit
// multiplies back per column (key_comp).
__device__ __forceinline__ uint32_t key_frag(uint32_t rotated, int nt) {
  return rotated & ((1u << (11 + nt)) | (1u << (27 + nt)));
}
__host__ __device__ constexpr float key_comp(int nt) { return pos_comp(11 + nt); }

// Bits r and r+16 of w as an f16x2 pair {0, 2^bit_exp(r)} with a single AND:
// the word is pre-rotated so that the two bits sit on one fp16 exponent bit
// (positions 10..14 of each half), r5/r10/r31 = w rotated left by 5/10/31.
// The power of two is undone per channel on the accumulator at the end.
__device__ __forceinline__ uint32_t bit_pair_exp(uint32_t w, uint32_t r5, uint32_t r10, uint32_t r31, int r) {
  if (r >= 10 && r <= 14) return w & ((1u << r) | (1u << (r + 16)));
  if (r >= 5 && r <= 9) return r5 & ((1u << (r + 5)) | (1u << (r + 21)));
  if (r <= 4) return r10 & ((1u << (r + 10)) | (1u << (r + 26)));
  return r31 & ((1u << 14) | (1u << 30));
}
// fp16 exponent position of bit r after the rotation, and the factor that
// maps the accumulated 2^e * x back to x.
__host__ __device__ constexpr int bit_pos(int r) {
  return (r >= 10 && r <= 14) ? r : (r >= 5 && r <= 9) ? r + 5 : (r <= 4) ? r + 10 : 14;
}
__host__ __device__ constexpr float bit_comp(int r) { return pos_comp(bit_pos(r)); }

// fp16 high part of two floats (truncated to 11 significant bits, exact in
// fp16) and the fp16 rounding of the remainder.
__device__ __forceinline__ void split_hi_lo(float2 w, uint32_t& hi, uint32_t& lo) {
  const float2 h = make_float2(__uint_as_float(__float_as_uint(w.x) & 0xFFFFE000u),
                               __uint_as_float(__float_as_uint(w.y) & 0xFFFFE000u));
  const float2 l = f2_sub(w, h);
  hi = pack_f16x2(h.x, h.y);
  lo = pack_f16x2(l.x, l.y);
}

// z and s of one group from its bf16 (min, max) word.
template <int BITS>
__device__ __forceinline__ void dequant_params(uint32_t mm, float& z, float& s) {
  const float lo = __uint_as_float(mm << 16), hi = __uint_as_float(mm & 0xFFFF0000u);
  if (BITS == 1) {
    s = (hi - lo) * 0.5f;
    z = fmaf(s, 0.5f, lo);  // (3 min + max) / 4 = min + s / 2
  } else {
    s = (hi - lo) * (1.f / 3.f);
    z = lo;
  }
}

// z and s of four groups from their bf16 (min, max) words, two groups per
// packed instruction (the same roundings as dequant_params).
template <int BITS>
__device__ __forceinline__ void dequant_params4(uint4 mm, float4& z, float4& s) {
  const float2 lo01 = make_float2(__uint_as_float(mm.x << 16), __uint_as_float(mm.y << 16));
  const float2 lo23 = make_float2(__uint_as_float(mm.z << 16), __uint_as_float(mm.w << 16));
  const float2 hi01 = make_float2(__uint_as_float(mm.x & 0xFFFF0000u), __uint_as_float(mm.y & 0xFFFF0000u));
  const float2 hi23 = make_float2(__uint_as_float(mm.z & 0xFFFF0000u), __uint_as_float(mm.w & 0xFFFF0000u));
  constexpr float f = BITS == 1 ? 0.5f : 1.f / 3.f;
  const float2 s01 = f2_mul(f2_sub(hi01, lo01), make_float2(f, f));
  const float2 s23 = f2_mul(f2_sub(hi23, lo23), make_float2(f, f));
  s = make_float4(s01.x, s01.y, s23.x, s23.y);
  if (BITS == 1) {
    const float2 z01 = f2_fma(s01, make_float2(0.5f, 0.5f), lo01);
    const float2 z23 = f2_fma(s23, make_float2(0.5f, 0.5f), lo23);
    z = make_float4(z01.x, z01.y, z23.x, z23.y);
  } else {
    z = make_float4(lo01.x, lo01.y, lo23.x, lo23.y);
  }
}

struct CtaMerge {
  float m[kSlots][kMaxRows];
  float l[kSlots][kMaxRows];
  float o[kSlots][kMaxRows][kMergePitch];
};
// the clustered combine's partial (kMaxRows x kPartStride floats) follows the merge buffer
constexpr int kClusterPartOffset = (int)((sizeof(CtaMerge) + 15) / 16 * 16);

// ------------------------------------------------------------ 16-bit rows
// bf16 tensor-core product D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_16816_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four 8x8 b16 matrices from shared memory; lane l gives the row address of
// matrix l / 8, row l % 8.  .trans delivers each matrix transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(row)));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(row)));
}
// Two floats as bf16x2 (x in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}
// x = l1 + l2 + l3 in bf16 (each the rounding of what the previous ones leave;
// the first two remainders are exact in binary32), for two values at once.
__device__ __forceinline__ void split3_bf16(float2 x, uint32_t& l1, uint32_t& l2, uint32_t& l3) {
  l1 = pack_bf16x2(x.x, x.y);
  const float2 r1 = f2_sub(x, unpack_bf16x2(l1));
  l2 = pack_bf16x2(r1.x, r1.y);
  const float2 r2 = f2_sub(r1, unpack_bf16x2(l2));
  l3 = pack_bf16x2(r2.x, r2.y);
}
constexpr int kRowPitch = 512 + 16;  // bytes per staged 16-bit row (K then V, padded: conflict-free ldmatrix)

// The residual window and the fetched rows of this warp's range, before its
// low-bit groups (whose first stage is already in flight), on the tensor
// cores with exact bf16 operands.  Rows are staged ROWB at a time (a multiple
// of 8) with cp.async into `tail` (the warp's stages after the first and its
// z/s table, free until the low-bit loop starts), kRowPitch bytes apart.
// fill_query() is the CTA-wide fill of sq (it ends with a barrier); the
// positions of the warp's first fetched rows are loaded before it, so that
// both latencies overlap.
//   Logits: D(16 x 8 rows) = A (scaled query, the 8 query rows' three bf16
//   limbs: limbs 1 and 2 as rows 0..7 and 8..15 of one product, limb 3 in a
//   second) x B (the rows' keys, straight from shared memory by ldmatrix);
//   lane (gid, t) then holds query row gid's logits of rows 2t, 2t+1 (and
//   8 + ...) of each 8-row tile: the softmax layout of the low-bit loop.
//   Values: oacc (channels x query rows) += A (V^T, ldmatrix.trans) x B (the
//   probabilities in two bf16 limbs, two products), B being the lane's own
//   probabilities.
// sq is the CTA's scaled query tile [kMaxRows][kTilePitch] (rows 2G.. zero).
// On return (m_run, l_run, oacc) hold the softmax state of the rows in the
// fragment layouts of the low-bit loop (oacc divided by the per-channel powers
// of two that loop multiplies back at its end; l_run this lane's share).
template <bool MERGED, bool TOPK, int ROWB, typename FillQuery>
__device__ __forceinline__ void rows16_prologue(const AttnArgs& a, const float* sq, uint8_t* tail,
                                                FillQuery&& fill_query, float& m_run, float& l_run,
                                                float (&oacc)[8][4]) {
  constexpr int NT = ROWB / 8;  // 8-row tiles per batch
  static_assert(ROWB % 8 == 0 && NT >= 1 && NT <= 2, "batches of 8 or 16 rows");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.y;
  const int G = a.G;

  // rows: residual window [0, r), fetched rows [r, r + kk), then the
  // speculative token's own row (seen by the speculative query rows only)
  const int kk = MERGED ? a.k : 0;
  const int j_self = a.kv_self != nullptr ? a.r + kk : -1;
  const int n_rows = a.r + kk + (a.kv_self != nullptr ? 1 : 0);
  const int n_warps = a.chunks * kWarps;
  const int per_warp = (n_rows + n_warps - 1) / n_warps;
  const int j0 = min(n_rows, (int)(blockIdx.x * kWarps + warp) * per_warp);
  const int j1 = min(n_rows, j0 + per_warp);
  const bool spec_lane = MERGED && a.spec_logits != nullptr && gid >= G && gid < 2 * G;
  float* spec_out = spec_lane ? a.spec_logits + (bh * G + (gid - G)) * (int64_t)a.Lcap : nullptr;
  const bool rowlog_lane = TOPK && MERGED && a.sel_rowlog != nullptr && gid >= G && gid < 2 * G;

  m_run = kNeg;
  l_run = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
  // quantised position of the fetched row of lane (window w0), -1 for the residual window
  auto row_pos = [&](int w0) {
    const int j = w0 + lane;
    return (lane < min(32, j1 - w0) && j >= a.r && j < a.r + kk) ? a.idx[bh * a.k + (j - a.r)] : -1;
  };
  const int pos_first = row_pos(j0);
  fill_query();
  if (j0 >= j1) return;

  // the scaled query's three bf16 limbs, as A fragments: lane row gid, channels 16 kc + 2t (+1, +8, +9)
  const float* qrow = sq + gid * kTilePitch;

  for (int w0 = j0; w0 < j1; w0 += 32) {
    const int nwin = min(32, j1 - w0);
    const int pos = w0 == j0 ? pos_first : row_pos(w0);
    const bool ok = lane < nwin && (w0 + lane < a.r || w0 + lane == j_self || (pos >= 0 && pos < a.nq));
    const uint32_t valid = __ballot_sync(0xFFFFFFFFu, ok);
    for (int b0 = 0; b0 < nwin; b0 += ROWB) {
      const int nb = min(ROWB, nwin - b0);
      for (int i = 0; i < ROWB; ++i) {
        uint8_t* dst = tail + kRowPitch * i + 16 * lane;
        if (i < nb && ((valid >> (b0 + i)) & 1u)) {
          const int j = w0 + b0 + i;
          const uint16_t* row = j < a.r        ? a.resid + (bh * a.resid_cap + j) * 2 * kD
                                : j == j_self ? a.kv_self + bh * 2 * kD
                                              : a.staging + (bh * a.k + (j - a.r)) * 2 * kD;
          cp_async16(dst, row + 8 * lane);
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);  // no stale bits under a zero probability
        }
      }
      cp_async_commit();
      cp_async_wait<0>();  // with the first batch, also the low-bit stages issued before it
      __syncwarp();

      // ---- logits: query rows x the batch's rows ----
      float c12[NT][4], c3[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) c12[nt][0] = c12[nt][1] = c12[nt][2] = c12[nt][3] = c3[nt][0] = c3[nt][1] =
          c3[nt][2] = c3[nt][3] = 0.f;
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        uint32_t a12[4], a3[4];
        {
          const float2 x01 = *reinterpret_cast<const float2*>(qrow + 16 * kc + 2 * t);
          const float2 x89 = *reinterpret_cast<const float2*>(qrow + 16 * kc + 2 * t + 8);
          split3_bf16(x01, a12[0], a12[1], a3[0]);
          split3_bf16(x89, a12[2], a12[3], a3[2]);
          a3[1] = a3[3] = 0u;
        }
        // keys: matrices (tile nt, channels 16kc + 8h) for h = 0, 1; lane l addresses row 8 (l >> 4) + (l & 7)
        uint32_t kb[4];
        ldsm_x4(kb, tail + kRowPitch * (8 * (NT == 2 ? (lane >> 4) : 0) + (lane & 7)) + 2 * (16 * kc + 8 * ((lane >> 3) & 1)));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_16816_bf16(c12[nt], a12, kb[2 * nt], kb[2 * nt + 1]);
          mma_16816_bf16(c3[nt], a3, kb[2 * nt], kb[2 * nt + 1]);
        }
      }
      // lane: query row gid, batch rows 8 nt + 2t + e
      float lg[NT][2];
      int posr[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = 8 * nt + 2 * t + e;
          const float v = (c12[nt][e] + c12[nt][2 + e]) + c3[nt][e];
          const int j = w0 + b0 + i;
          posr[nt][e] = __shfl_sync(0xFFFFFFFFu, pos, (b0 + i) & 31);
          const bool seen = i < nb && ((valid >> ((b0 + i) & 31)) & 1u) && !(j == j_self && gid < G);
          lg[nt][e] = seen ? v : kNeg;
        }
      if (spec_lane || rowlog_lane) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pi = posr[nt][e];
            if (lg[nt][e] != kNeg && pi >= 0) {
              if (spec_lane) spec_out[pi] = lg[nt][e] * CUDART_LN2_F;
              if (TOPK && rowlog_lane)  // fetched row j of this (b, hkv), head gid - G
                a.sel_rowlog[(bh * a.k + (w0 + b0 + 8 * nt + 2 * t + e - a.r)) * 4 + (gid - G)] =
                    lg[nt][e] * CUDART_LN2_F;
            }
          }
      }
      // ---- online softmax (base 2): query row gid's max over the four lanes of the row ----
      float mx = lg[0][0] > lg[0][1] ? lg[0][0] : lg[0][1];
      if (NT == 2) mx = fmaxf(mx, fmaxf(lg[NT - 1][0], lg[NT - 1][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      if (__any_sync(0xFFFFFFFFu, m_new != m_run)) {
        const float alpha = fast_exp2(m_run - m_new);
        const float al_a = __shfl_sync(0xFFFFFFFFu, alpha, (2 * t) * 4);
        const float al_b = __shfl_sync(0xFFFFFFFFu, alpha, (2 * t + 1) * 4);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          oacc[mt][0] *= al_a;
          oacc[mt][1] *= al_b;
          oacc[mt][2] *= al_a;
          oacc[mt][3] *= al_b;
        }
        l_run *= alpha;
        m_run = m_new;
      }
      const float m_use = fmaxf(m_run, 0.5f * kNeg);  // a masked logit gives exactly 0
      uint32_t ph[NT], pl[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float p0 = fast_exp2(lg[nt][0] - m_use), p1 = fast_exp2(lg[nt][1] - m_use);
        l_run += p0 + p1;
        ph[nt] = pack_bf16x2(p0, p1);
        const float2 rem = f2_sub(make_float2(p0, p1), unpack_bf16x2(ph[nt]));
        pl[nt] = pack_bf16x2(rem.x, rem.y);
      }
      // ---- values: oacc += V^T (channels x rows) x P (rows x query rows), P in two bf16 limbs ----
      // B fragment: k = rows 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1), n = query row gid -- this lane's p
      const uint32_t bh0 = ph[0], bh1 = NT == 2 ? ph[NT - 1] : 0u;
      const uint32_t bl0 = pl[0], bl1 = NT == 2 ? pl[NT - 1] : 0u;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        // matrices (rows 8 (l >> 4) .., channels 16 mt + 8 ((l >> 3) & 1)), transposed
        uint32_t va[4];
        ldsm_x4_trans(va, tail + kRowPitch * (8 * (NT == 2 ? (lane >> 4) : 0) + (lane & 7)) + 2 * kD +
                              2 * (16 * mt + 8 * ((lane >> 3) & 1)));
        if (NT == 1) va[2] = va[3] = 0u;  // rows 8..15 do not exist in an 8-row batch
        mma_16816_bf16(oacc[mt], va, bh0, bh1);
        mma_16816_bf16(oacc[mt], va, bl0, bl1);
      }
      __syncwarp();  // the batch's rows are read before the next batch is staged
    }
  }
  // the low-bit loop multiplies its accumulators by per-channel powers of two at its end
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const float c0 = 1.f / bit_comp(2 * mt), c1 = 1.f / bit_comp(2 * mt + 1);
    oacc[mt][0] *= c0;
    oacc[mt][1] *= c0;
    oacc[mt][2] *= c1;
    oacc[mt][3] *= c1;
  }
}

// ------------------------------------------------------------ low-bit CTA
template <int BITS, int GROUP, bool MERGED, bool FETCH, bool TOPK, typename FillQuery>
__device__ __forceinline__ void lowbit_cta(const AttnArgs& a, uint8_t* dyn, const float* sq, CtaMerge& merge,
                                           const uint32_t* s_tmem, FillQuery&& fill_query) {
  using LY = Layout<BITS, GROUP>;
  constexpr int NH = LY::H;  // 32-token halves per record
  constexpr int RB = LY::RB;
  constexpr int KMETA = LY::KMETA;
  constexpr int VCODES = LY::VCODES;
  constexpr int VMETA = LY::VMETA;
  constexpr int STAGE = LY::STAGE;
  constexpr int kStages = LY::STAGES;
  constexpr int WARP_BYTES = LY::WARP_BYTES;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.y;
  const int chunk = blockIdx.x;
  const int G = a.G;
  const bool row_valid = gid < 2 * G;

  uint8_t* stage = dyn + (size_t)warp * WARP_BYTES;
  // per-group z and s: keys [t][kc][z0..3, s0..3], values [t][c16][e][z at slot e over cg0..3,
  // s at channel group e over slot0..3] (the scales transposed so that a B fragment's two tokens
  // sit side by side),
  // each t block padded by one float4 so that the four t rows read together
  // fall in different banks
  float4* kzs = reinterpret_cast<float4*>(stage + kStages * STAGE);
  float4* vzs = kzs + kZsPitch * 4;

  // records (groups of GROUP tokens) of this CTA: groups_per_chunk counts 32-token halves
  const int u_begin = chunk * (a.groups_per_chunk / NH);
  const int u_end = min(a.nq / GROUP, u_begin + a.groups_per_chunk / NH);
  const int n_my = (u_end - u_begin - warp + kWarps - 1) / kWarps;  // records of this warp
  const uint8_t* rec_base = a.records + (bh * a.units_cap) * (int64_t)RB;

  // Pre-fetch rows of this warp: rr = pf_slot + pf_nslots * i, row i on
  // item i * pf_every + pf_ph, at most one per pipeline depth, so that a
  // warp waits on at most one host read at a time.  The phase pf_ph (the
  // warp's slot modulo the spacing) spreads the host reads of neighbouring
  // warps over consecutive items: the warps of the grid advance in step, and
  // reads that they all issue in the same item arrive at the host link as one
  // burst.  (Phase 0 carries its first row on item 0, the first low-bit
  // stage, which the 16-bit-row prologue waits for.)  A carried row is loaded
  // into registers (16 bytes per lane) when its item is issued and stored to
  // the staging buffer when the next one is issued, pf_every items later, so
  // the host read's latency stalls no stage of the record pipeline.  Rows
  // beyond the warp's items are copied after the groups.
  const int pf_nslots = gridDim.x * gridDim.y * kWarps;
  const int pf_slot = (blockIdx.y * gridDim.x + blockIdx.x) * kWarps + warp;
  const int n_pf = (FETCH && a.pf_rows > pf_slot) ? (a.pf_rows - pf_slot + pf_nslots - 1) / pf_nslots : 0;
  const int pf_every = n_pf > 0 ? max(kStages, n_my / n_pf) : 1;
  const int pf_ph = pf_slot % pf_every;
  const int pf_carried = (n_pf > 0 && n_my > pf_ph) ? min(n_pf, 1 + (n_my - 1 - pf_ph) / pf_every) : 0;
  int pf_next = n_pf > 0 ? a.pf_idx[pf_slot] : -1;  // position of the next row to issue
  int pf_next_src = (n_pf > 0 && a.pf_src != nullptr) ? a.pf_src[pf_slot] : -1;  // its previous slot, or -1
  int pf_issue_i = 0, pf_issue_item = pf_ph;         // next carried row on the issue side and its item
  uint4 pf_v = make_uint4(0u, 0u, 0u, 0u);  // the carried row in flight: this lane's 16 bytes
  int pf_rr = -1;                           // its staging row, or -1
  auto pf_store = [&]() {
    if (pf_rr >= 0) reinterpret_cast<uint4*>(a.pf_staging + (int64_t)pf_rr * (2 * kD))[lane] = pf_v;
    pf_rr = -1;
  };

  auto issue = [&](int item) {
    if (item < n_my) {
      const int u = u_begin + warp + item * kWarps;
      const uint8_t* src = rec_base + (int64_t)u * RB;
      uint8_t* dst = stage + (item % kStages) * STAGE;
#pragma unroll
      for (int w = 0; w < RB / 512; ++w) cp_async16(dst + 16 * (lane + 32 * w), src + 16 * (lane + 32 * w));
      // the record's bitmap words (one per 32-token half) into the slot's first words
      if (MERGED && lane < NH) cp_async4(dst + RB + 4 * lane, a.bitmap + bh * a.q_groups_cap + NH * u + lane);
      if constexpr (FETCH) {
        // the row this item carries, if any
        const bool carry = item == pf_issue_item && pf_issue_i < pf_carried;
        const int rr = pf_slot + pf_nslots * pf_issue_i;
        const int n = carry ? pf_next : -1;
        if (carry) {
          pf_store();  // the previous carried row, loaded pf_every items ago
          if (n >= 0 && n < a.pf_ncap) {
            const int sj = pf_next_src;
            const uint16_t* row =
                (sj >= 0 && sj < a.pf_prev_k)
                    ? a.pf_prev + ((int64_t)(rr / a.pf_k) * a.pf_prev_k + sj) * (2 * kD)  // still staged
                    : a.pf_host + ((int64_t)(rr / a.pf_k) * a.pf_ncap + n) * (2 * kD);
            pf_v = reinterpret_cast<const uint4*>(row)[lane];
            pf_rr = rr;
          }
          pf_next = (pf_issue_i + 1 < n_pf) ? a.pf_idx[rr + pf_nslots] : -1;
          pf_next_src = (a.pf_src != nullptr && pf_issue_i + 1 < n_pf) ? a.pf_src[rr + pf_nslots] : -1;
          ++pf_issue_i;
          pf_issue_item = pf_issue_i * pf_every + pf_ph;
        }
      }
    }
    cp_async_commit();
  };

  // the state left by this warp's 16-bit rows, and the scaled query of row
  // gid at this lane's 32 channels, ordered m = 4*kc + 2*h + half <->
  // channel 16*kc + 2*t + 8*h + half (registers at 1 bit, else read from sq)
  float m_run, l_run;
  float oacc[8][4];
  // The first low-bit stage is in flight behind the query fill and the 16-bit
  // rows, which are staged in the other stages and the z/s table (a warp's
  // rows then take one round trip); the rest of the pipeline is issued after.
  issue(0);
  rows16_prologue<MERGED, TOPK, LY::ROWB>(a, sq, stage + STAGE, fill_query, m_run, l_run, oacc);
  // on-chip selection: this warp's TMEM lanes (its 32-lane quarter), read after the CTA barrier of the query fill
  uint32_t tmem_warp = 0;
  if constexpr (TOPK) {
    if (a.sel_onchip) {
      tmem_fence_after_sync();
      tmem_warp = *s_tmem + ((uint32_t)(32 * warp) << 16);
    }
  }
#pragma unroll 1
  for (int s = 1; s < kStages - 1; ++s) issue(s);
  constexpr bool kQvReg = QueryInRegisters<BITS>::value;
  float qv[kQvReg ? 32 : 1];
  if constexpr (kQvReg) {
#pragma unroll
    for (int m = 0; m < 32; m += 2) {
      const float2 v = *reinterpret_cast<const float2*>(sq + gid * kTilePitch + 16 * (m >> 2) + 2 * t + 8 * ((m >> 1) & 1));
      qv[m] = v.x;
      qv[m + 1] = v.y;
    }
  }
  float2 zacc01 = make_float2(0.f, 0.f), zacc23 = make_float2(0.f, 0.f);

  const bool spec_row = row_valid && gid >= G && a.spec_logits != nullptr;
  float* spec_out = spec_row ? a.spec_logits + ((bh * G + (gid - G)) * (int64_t)a.Lcap) : nullptr;

#pragma unroll 1
  for (int it = 0; it < n_my; ++it) {
    issue(it + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const uint8_t* R = stage + (it % kStages) * STAGE;
    const int u = u_begin + warp + it * kWarps;

#pragma unroll 1
    for (int hf = 0; hf < NH; ++hf) {
      const int g = NH * u + hf;  // the 32-token group of this half
      const int zi = kZsPitch * (lane >> 3) + 2 * (lane & 7);
      if (hf == 0) {  // ---- z, s of the record's 128 key groups, 4 per lane (shared by its halves) ----
        float4 z, s;
        dequant_params4<BITS>(*reinterpret_cast<const uint4*>(R + KMETA + 16 * lane), z, s);
        kzs[zi] = z;  // lane covers key entries 4*lane..4*lane+3 = (t = lane/8, kc = lane%8)
        kzs[zi + 1] = s;
      }
      // ---- z, s of the half's 128 value groups (32 tokens x 4 channel groups), 4 per lane ----
      {
        float4 z, s;
        // lane's token, channel groups 0..3 (at g = 64 channel groups 2c, 2c+1 share word c)
        uint4 mm;
        if constexpr (GROUP == 32) {
          mm = *reinterpret_cast<const uint4*>(R + VMETA + 16 * lane);
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(R + VMETA + 256 * hf + 8 * lane);
          mm = make_uint4(w.x, w.x, w.y, w.y);
        }
        dequant_params4<BITS>(mm, z, s);
        vzs[zi] = z;  // value entries: (t, c16, slot) = (lane/8, (lane/4)%2, lane%4), cg 0..3
        {  // scales transposed within the c16 block: entry 4 c16 + cg holds slots 0..3
          float* st = reinterpret_cast<float*>(vzs + kZsPitch * (lane >> 3) + 2 * (lane & 4) + 1);
          const int slot = lane & 3;
          st[slot] = s.x;
          st[8 + slot] = s.y;
          st[16 + slot] = s.z;
          st[24 + slot] = s.w;
        }
      }
      __syncwarp();

      // ---- QK, channel chunk outer: A = q o s (hi/lo), B = key bits ----
      uint32_t kw[4], kw1[4];  // word j: channel pairs 4j .. 4j+3 of the lane's four tokens
      {
        const uint8_t* KC = R + 512 * BITS * hf;  // the half's key code planes
        const uint4 v0 = *reinterpret_cast<const uint4*>(KC + 16 * lane);
        kw[0] = v0.x; kw[1] = v0.y; kw[2] = v0.z; kw[3] = v0.w;
        if (BITS == 2) {
          const uint4 v1 = *reinterpret_cast<const uint4*>(KC + 512 + 16 * lane);
          kw1[0] = v1.x; kw1[1] = v1.y; kw1[2] = v1.z; kw1[3] = v1.w;
        }
      }
      float acc[4][4];
  #pragma unroll
      for (int nt = 0; nt < 4; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      float2 bias2 = make_float2(0.f, 0.f);
  #pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        const float4 z4 = kzs[kZsPitch * t + 2 * kc];
        const float4 s4 = kzs[kZsPitch * t + 2 * kc + 1];
        // query row gid at channels 16kc + 2t + {0, 1} and 16kc + 2t + 8 + {0, 1}
        float2 q01, q23;
        if constexpr (kQvReg) {
          q01 = make_float2(qv[4 * kc], qv[4 * kc + 1]);
          q23 = make_float2(qv[4 * kc + 2], qv[4 * kc + 3]);
        } else {
          q01 = *reinterpret_cast<const float2*>(sq + gid * kTilePitch + 16 * kc + 2 * t);
          q23 = *reinterpret_cast<const float2*>(sq + gid * kTilePitch + 16 * kc + 2 * t + 8);
        }
        bias2 = f2_fma(q01, make_float2(z4.x, z4.y), bias2);
        bias2 = f2_fma(q23, make_float2(z4.z, z4.w), bias2);
        uint32_t af[4];
        split_hi_lo(f2_mul(q01, make_float2(s4.x, s4.y)), af[0], af[1]);
        split_hi_lo(f2_mul(q23, make_float2(s4.z, s4.w)), af[2], af[3]);
        // channel pairs e = 2kc (b0) and 2kc + 1 (b1): word kc/2 rotated by 4i, i = e mod 4
        const int rot = 8 * (kc & 1);
        const uint32_t r0 = __funnelshift_l(kw[kc >> 1], kw[kc >> 1], rot);
        const uint32_t r1 = __funnelshift_l(kw[kc >> 1], kw[kc >> 1], rot + 4);
        if (BITS == 2) {  // high plane: weight 2, carried by doubling A (exact in fp16)
          const uint32_t x0 = __funnelshift_l(kw1[kc >> 1], kw1[kc >> 1], rot);
          const uint32_t x1 = __funnelshift_l(kw1[kc >> 1], kw1[kc >> 1], rot + 4);
          const uint32_t af2[4] = {hadd2_u32(af[0], af[0]), hadd2_u32(af[1], af[1]), hadd2_u32(af[2], af[2]),
                                   hadd2_u32(af[3], af[3])};
  #pragma unroll
          for (int nt = 0; nt < 4; ++nt) mma_16816(acc[nt], af2, key_frag(x0, nt), key_frag(x1, nt));
        }
  #pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma_16816(acc[nt], af, key_frag(r0, nt), key_frag(r1, nt));
      }
      float bias = bias2.x + bias2.y;
      bias += __shfl_xor_sync(0xFFFFFFFFu, bias, 1);
      bias += __shfl_xor_sync(0xFFFFFFFFu, bias, 2);

      // ---- logits, speculative-row output, online softmax (base 2) ----
      // bm: the group's tokens whose 16-bit rows were fetched (same word in every lane)
      const uint32_t bm = MERGED ? reinterpret_cast<const uint32_t*>(R + RB)[hf] : 0u;
      float lg[4][2];
  #pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float2 l = f2_fma(f2_add(make_float2(acc[nt][0], acc[nt][1]), make_float2(acc[nt][2], acc[nt][3])),
                                make_float2(key_comp(nt), key_comp(nt)), make_float2(bias, bias));
        lg[nt][0] = l.x;
        lg[nt][1] = l.y;
      }
      if (TOPK && a.sel_onchip) {
        // the half's speculative logits into TMEM, lane = token, column 4 (NH it + hf) + head: transposed
        // through the half's key-code planes, which are in registers since the QK step began
        float* tx = reinterpret_cast<float*>(const_cast<uint8_t*>(R) + 512 * BITS * hf);  // [token][4]
        if (row_valid && gid >= G) {
  #pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            tx[(8 * nt + 2 * t) * 4 + (gid - G)] = lg[nt][0] * CUDART_LN2_F;
            tx[(8 * nt + 2 * t + 1) * 4 + (gid - G)] = lg[nt][1] * CUDART_LN2_F;
          }
        }
        __syncwarp();
        tmem_st4(tmem_warp + 4 * (NH * it + hf), reinterpret_cast<const float4*>(tx)[lane]);
      }
      if (spec_row) {
        float* dst = spec_out + (int64_t)g * kGroup + 2 * t;
        if (!MERGED || bm == 0u) {  // uniform: most groups have no fetched token
  #pragma unroll
          for (int nt = 0; nt < 4; ++nt)
            *reinterpret_cast<float2*>(dst + 8 * nt) =
                f2_mul(make_float2(lg[nt][0], lg[nt][1]), make_float2(CUDART_LN2_F, CUDART_LN2_F));
        } else {
  #pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const uint32_t mb = (bm >> (8 * nt + 2 * t)) & 3u;
            if (!(mb & 1u)) dst[8 * nt] = lg[nt][0] * CUDART_LN2_F;
            if (!(mb & 2u)) dst[8 * nt + 1] = lg[nt][1] * CUDART_LN2_F;
          }
        }
      }
      if (MERGED && bm != 0u) {  // uniform: most groups have no fetched token
  #pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int tok = 8 * nt + 2 * t;
          if ((bm >> tok) & 1u) lg[nt][0] = kNeg;
          if ((bm >> (tok + 1)) & 1u) lg[nt][1] = kNeg;
        }
      }
      float gmax = fmaxf(fmaxf(fmaxf(lg[0][0], lg[0][1]), fmaxf(lg[1][0], lg[1][1])),
                         fmaxf(fmaxf(lg[2][0], lg[2][1]), fmaxf(lg[3][0], lg[3][1])));
      gmax = fmaxf(gmax, __shfl_xor_sync(0xFFFFFFFFu, gmax, 1));
      gmax = fmaxf(gmax, __shfl_xor_sync(0xFFFFFFFFu, gmax, 2));
      const float m_new = fmaxf(m_run, gmax);
      if (__any_sync(0xFFFFFFFFu, m_new != m_run)) {
        const float alpha = fast_exp2(m_run - m_new);
        const float al_a = __shfl_sync(0xFFFFFFFFu, alpha, (2 * t) * 4);
        const float al_b = __shfl_sync(0xFFFFFFFFu, alpha, (2 * t + 1) * 4);
  #pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          oacc[mt][0] *= al_a;
          oacc[mt][1] *= al_b;
          oacc[mt][2] *= al_a;
          oacc[mt][3] *= al_b;
        }
        l_run *= alpha;
        zacc01 = f2_mul(zacc01, make_float2(alpha, alpha));
        zacc23 = f2_mul(zacc23, make_float2(alpha, alpha));
        m_run = m_new;
      }
      // a masked logit (kNeg) gives exactly 0, also while no token has been seen yet
      const float m_use = fmaxf(m_run, 0.5f * kNeg);
      float p[4][2];
  #pragma unroll
      for (int nt = 0; nt < 4; ++nt)
  #pragma unroll
        for (int e = 0; e < 2; ++e) {
          p[nt][e] = fast_exp2(lg[nt][e] - m_use);
          l_run += p[nt][e];
        }

      // ---- PV: two 16-token chunks; A = value bits, B = p o s ----
      uint32_t vw[4], vw1[4];
      {
        const uint8_t* VC = R + VCODES + 512 * BITS * hf;  // the half's value code planes
        const uint4 v0 = *reinterpret_cast<const uint4*>(VC + 16 * lane);
        vw[0] = v0.x; vw[1] = v0.y; vw[2] = v0.z; vw[3] = v0.w;
        if (BITS == 2) {
          const uint4 v1 = *reinterpret_cast<const uint4*>(VC + 512 + 16 * lane);
          vw1[0] = v1.x; vw1[1] = v1.y; vw1[2] = v1.z; vw1[3] = v1.w;
        }
      }
  #pragma unroll
      for (int c16 = 0; c16 < 2; ++c16) {
        const float ps[4] = {p[2 * c16][0], p[2 * c16][1], p[2 * c16 + 1][0], p[2 * c16 + 1][1]};
        float4 zz[4], ss[4];  // zz[slot] over cg, ss[cg] over slot
  #pragma unroll
        for (int slot = 0; slot < 4; ++slot) {
          zz[slot] = vzs[kZsPitch * t + 2 * (4 * c16 + slot)];
          ss[slot] = vzs[kZsPitch * t + 2 * (4 * c16 + slot) + 1];
          const float2 pp = make_float2(ps[slot], ps[slot]);
          zacc01 = f2_fma(pp, make_float2(zz[slot].x, zz[slot].y), zacc01);
          zacc23 = f2_fma(pp, make_float2(zz[slot].z, zz[slot].w), zacc23);
        }
        uint32_t bfr[4][2];
        {
          const float2 p01 = make_float2(ps[0], ps[1]), p23 = make_float2(ps[2], ps[3]);
          float2 x;
  #pragma unroll
          for (int cg = 0; cg < 4; ++cg) {  // ss[cg]: the scales of slots 0..3 at channel group cg
            x = f2_mul(p01, make_float2(ss[cg].x, ss[cg].y)); bfr[cg][0] = pack_f16x2(x.x, x.y);
            x = f2_mul(p23, make_float2(ss[cg].z, ss[cg].w)); bfr[cg][1] = pack_f16x2(x.x, x.y);
          }
        }
        {
          const uint32_t wa = vw[2 * c16], wb = vw[2 * c16 + 1];
          const uint32_t a5 = __funnelshift_l(wa, wa, 5), a10 = __funnelshift_l(wa, wa, 10),
                         a31 = __funnelshift_l(wa, wa, 31);
          const uint32_t b5 = __funnelshift_l(wb, wb, 5), b10 = __funnelshift_l(wb, wb, 10),
                         b31 = __funnelshift_l(wb, wb, 31);
  #pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t af[4] = {bit_pair_exp(wa, a5, a10, a31, 2 * mt), bit_pair_exp(wa, a5, a10, a31, 2 * mt + 1),
                                    bit_pair_exp(wb, b5, b10, b31, 2 * mt), bit_pair_exp(wb, b5, b10, b31, 2 * mt + 1)};
            mma_16816(oacc[mt], af, bfr[mt >> 1][0], bfr[mt >> 1][1]);
          }
        }
        if (BITS == 2) {  // high plane: weight 2, carried by doubling B
          uint32_t bfr2[4][2];
  #pragma unroll
          for (int cg = 0; cg < 4; ++cg) {
            bfr2[cg][0] = hadd2_u32(bfr[cg][0], bfr[cg][0]);
            bfr2[cg][1] = hadd2_u32(bfr[cg][1], bfr[cg][1]);
          }
          const uint32_t xa = vw1[2 * c16], xb = vw1[2 * c16 + 1];
          const uint32_t a5 = __funnelshift_l(xa, xa, 5), a10 = __funnelshift_l(xa, xa, 10),
                         a31 = __funnelshift_l(xa, xa, 31);
          const uint32_t b5 = __funnelshift_l(xb, xb, 5), b10 = __funnelshift_l(xb, xb, 10),
                         b31 = __funnelshift_l(xb, xb, 31);
  #pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t af[4] = {bit_pair_exp(xa, a5, a10, a31, 2 * mt), bit_pair_exp(xa, a5, a10, a31, 2 * mt + 1),
                                    bit_pair_exp(xb, b5, b10, b31, 2 * mt), bit_pair_exp(xb, b5, b10, b31, 2 * mt + 1)};
            mma_16816(oacc[mt], af, bfr2[mt >> 1][0], bfr2[mt >> 1][1]);
          }
        }
      }
      __syncwarp();  // the half's value table and the stage are read by every lane
    }  // halves
  }
  cp_async_wait<0>();
  if constexpr (FETCH) pf_store();
  // pre-fetch rows this warp's groups did not carry, four host reads in flight at a time
  for (int i0 = pf_carried; i0 < n_pf; i0 += 4) {
    int rr[4];
    int n[4];
    int sj[4];
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      rr[u] = pf_slot + pf_nslots * (i0 + u);
      n[u] = i0 + u < n_pf ? a.pf_idx[rr[u]] : -1;
      sj[u] = (a.pf_src != nullptr && i0 + u < n_pf) ? a.pf_src[rr[u]] : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (n[u] >= 0 && n[u] < a.pf_ncap)
        v[u] = reinterpret_cast<const uint4*>(
            (sj[u] >= 0 && sj[u] < a.pf_prev_k) ? a.pf_prev + ((rr[u] / a.pf_k) * (int64_t)a.pf_prev_k + sj[u]) * (2 * kD)
                                                : a.pf_host + ((rr[u] / a.pf_k) * a.pf_ncap + n[u]) * (2 * kD))[lane];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (n[u] >= 0 && n[u] < a.pf_ncap) reinterpret_cast<uint4*>(a.pf_staging + (int64_t)rr[u] * (2 * kD))[lane] = v[u];
  }
  // undo the powers of two of the value-bit expansion, per channel
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    oacc[mt][0] *= bit_comp(2 * mt);
    oacc[mt][1] *= bit_comp(2 * mt);
    oacc[mt][2] *= bit_comp(2 * mt + 1);
    oacc[mt][3] *= bit_comp(2 * mt + 1);
  }
  __syncthreads();  // the merge buffer overlaps the stages of every warp

  // ---- warp state -> shared memory ----
  l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 1);
  l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 2);
  float zacc[4] = {zacc01.x, zacc01.y, zacc23.x, zacc23.y};
#pragma unroll
  for (int cg = 0; cg < 4; ++cg) {
    zacc[cg] += __shfl_xor_sync(0xFFFFFFFFu, zacc[cg], 1);
    zacc[cg] += __shfl_xor_sync(0xFFFFFFFFu, zacc[cg], 2);
  }
  if (t == 0) {
    merge.m[warp][gid] = m_run;
    merge.l[warp][gid] = l_run;
  }
  // oacc[mt]: (channel 16mt+gid, row 2t), (16mt+gid, 2t+1), (16mt+gid+8, 2t), (16mt+gid+8, 2t+1)
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    merge.o[warp][2 * t][16 * mt + gid] = oacc[mt][0];
    merge.o[warp][2 * t + 1][16 * mt + gid] = oacc[mt][1];
    merge.o[warp][2 * t][16 * mt + gid + 8] = oacc[mt][2];
    merge.o[warp][2 * t + 1][16 * mt + gid + 8] = oacc[mt][3];
  }
  __syncwarp();
  // the p*z term of row gid: zacc[cg] applies to channels 32cg .. 32cg+31
#pragma unroll
  for (int cg = 0; cg < 4; ++cg)
#pragma unroll
    for (int q8 = 0; q8 < 8; ++q8) merge.o[warp][gid][32 * cg + 8 * t + q8] += zacc[cg];
}

// ------------------------------------------------------------ merge + combine

// Output row and log-sum-exp of query row rho of (b, hkv) bh from its merged
// softmax state (max M, sum L, unnormalised output O at channel c).
__device__ __forceinline__ void write_row(const AttnArgs& a, int64_t bh, int rho, float M, float L, float O, int c) {
  const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv), G = a.G;
  const int qi = rho / G, gi = rho % G;
  const int64_t orow = ((int64_t)b * 2 + qi) * a.Hq + hk * G + gi;
  a.out[orow * kD + c] = f32_to_bf16_rne(L > 0.f ? O / L : 0.f);
  if (c == 0 && a.lse != nullptr) a.lse[orow] = L > 0.f ? (M + __log2f(L)) * CUDART_LN2_F : -CUDART_INF_F;
}

// The CTA's partial from its warps' states: per query row the max over the
// slots, then the sum and the output at channel c in slot order.  The rows
// are independent: unrolled, their dependent chains interleave.
__device__ __forceinline__ void cta_merge_rows(const CtaMerge& sm, int rows, int c, float* dst) {
#pragma unroll
  for (int rho = 0; rho < kMaxRows; ++rho) {
    if (rho < rows) {
      float M = kNeg;
#pragma unroll
      for (int w = 0; w < kSlots; ++w) M = fmaxf(M, sm.m[w][rho]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kSlots; ++w) {
        const float f = fast_exp2(sm.m[w][rho] - M);
        L += sm.l[w][rho] * f;
        O += sm.o[w][rho][c] * f;
      }
      float* pr = dst + rho * kPartStride;
      if (c == 0) {
        pr[0] = M;
        pr[1] = L;
      }
      pr[4 + c] = O;
    }
  }
}

// Returns whether this CTA was the last of its (b, hkv) and so combined the
// partials.  part_cap: partials that fit in the CTA's dynamic shared memory
// (which starts with the merge buffer `sm`).
__device__ __forceinline__ bool merge_store_combine(CtaMerge& sm, const AttnArgs& a, int* s_last, float* s_ml,
                                                    float* s_w, int part_cap) {
  __syncthreads();
  const int c = threadIdx.x;  // channel
  const int64_t bh = blockIdx.y;
  const int rows = 2 * a.G;
  const int nparts = a.chunks;
  cta_merge_rows(sm, rows, c, a.part + ((bh * nparts + blockIdx.x) * kMaxRows) * kPartStride);
  // combine_kernel runs after this grid.  A run-time flag on purpose: making
  // it a template branch (so that the partial-only instantiations lose the
  // code below) changed the register allocation of the pre-fetching variant
  // and slowed it by a quarter.
  if (a.ext_combine) return false;
  // last CTA of this (b, hkv) merges every partial.  The barrier orders the
  // CTA's partial before thread 0's fence and ticket (a fence is cumulative
  // over what the barrier ordered before it); the fence after the ticket and
  // the second barrier order the last CTA's reads after it.
  __syncthreads();
  if (c == 0) {
    __threadfence();
    *s_last = (atomicAdd(&a.tickets[bh], 1u) == (unsigned)(nparts - 1));
    __threadfence();
  }
  __syncthreads();
  if (!*s_last) return false;
  const float* base = a.part + (bh * nparts * kMaxRows) * kPartStride;
  if (nparts <= part_cap) {
    // Every partial's used rows into shared memory (the merge buffer and the
    // stages, free now) with one round of copies, then per query row the
    // arithmetic of the clustered combine in the same order, so that both
    // give identical results: thread rho finds row rho's max, sum and the
    // partials' weights (computed once, shared), every thread its channel's
    // output.
    float* sp = reinterpret_cast<float*>(&sm);
    const int per_part = rows * (kPartStride / 4);  // 16-byte pieces of one partial's used rows
    for (int p = 0; p < nparts; ++p)
      for (int e = c; e < per_part; e += kThreads)
        cp_async16(sp + (p * kMaxRows * kPartStride) + 4 * e, base + (int64_t)p * kMaxRows * kPartStride + 4 * e);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    if (c < rows) {
      float M = kNeg, L = 0.f;
      for (int p = 0; p < nparts; ++p) M = fmaxf(M, sp[(p * kMaxRows + c) * kPartStride]);
      for (int p = 0; p < nparts; ++p) {
        const float* pr = sp + (p * kMaxRows + c) * kPartStride;
        const float f = fast_exp2(pr[0] - M);
        L += pr[1] * f;
        s_w[p * kMaxRows + c] = f;
      }
      s_ml[c] = M;
      s_ml[kMaxRows + c] = L;
    }
    __syncthreads();
    float O[kMaxRows];
#pragma unroll
    for (int rho = 0; rho < kMaxRows; ++rho) O[rho] = 0.f;
    for (int p = 0; p < nparts; ++p)
#pragma unroll
      for (int rho = 0; rho < kMaxRows; ++rho)
        if (rho < rows) O[rho] += sp[(p * kMaxRows + rho) * kPartStride + 4 + c] * s_w[p * kMaxRows + rho];
#pragma unroll
    for (int rho = 0; rho < kMaxRows; ++rho)
      if (rho < rows) write_row(a, bh, rho, s_ml[rho], s_ml[kMaxRows + rho], O[rho], c);
    if (c == 0) atomicExch(&a.tickets[bh], 0u);  // ready for the next call on this workspace
    return true;
  }
  // More partials than shared memory holds: two passes over (max, sum) blocks.
  // The (max, sum) words of every partial into shared memory (the merge
  // buffer, free now) in one round trip, 2 * kPCap (p, row) pairs at a time.
  // Then, per query row c: the max and the sum over the partials in partial
  // order (the same arithmetic as the clustered combine, so both give
  // identical results); then every partial's output words, 4 partials' worth
  // of independent loads at a time.
  constexpr int kPCap = kSlots * kMaxRows * kMergePitch / (2 * kMaxRows);  // partials per block
  float* sml = &sm.o[0][0][0];  // [p][row][2]
  float M[kMaxRows], O[kMaxRows];
#pragma unroll
  for (int rho = 0; rho < kMaxRows; ++rho) {
    M[rho] = kNeg;
    O[rho] = 0.f;
  }
  // pass 1: the maxima
  for (int p0 = 0; p0 < nparts; p0 += kPCap) {
    const int np = min(kPCap, nparts - p0);
    for (int i = c; i < np * kMaxRows; i += kThreads) {
      const float* pr = base + ((int64_t)(p0 + i / kMaxRows) * kMaxRows + i % kMaxRows) * kPartStride;
      sml[2 * i] = __ldcg(pr);
      sml[2 * i + 1] = __ldcg(pr + 1);
    }
    __syncthreads();
    if (c < rows) {
      float m = p0 == 0 ? kNeg : s_ml[c];
      for (int p = 0; p < np; ++p) m = fmaxf(m, sml[2 * (p * kMaxRows + c)]);
      s_ml[c] = m;
    }
    __syncthreads();
  }
  if (nparts > kPCap) {  // the maxima are final only now: the sums in a second pass over the blocks
    if (c < rows) s_ml[kMaxRows + c] = 0.f;
    for (int p0 = 0; p0 < nparts; p0 += kPCap) {
      const int np = min(kPCap, nparts - p0);
      __syncthreads();
      for (int i = c; i < np * kMaxRows; i += kThreads) {
        const float* pr = base + ((int64_t)(p0 + i / kMaxRows) * kMaxRows + i % kMaxRows) * kPartStride;
        sml[2 * i] = __ldcg(pr);
        sml[2 * i + 1] = __ldcg(pr + 1);
      }
      __syncthreads();
      if (c < rows) {
        float l = s_ml[kMaxRows + c];
        const float m = s_ml[c];
        for (int p = 0; p < np; ++p) l += sml[2 * (p * kMaxRows + c) + 1] * fast_exp2(sml[2 * (p * kMaxRows + c)] - m);
        s_ml[kMaxRows + c] = l;
      }
    }
  } else if (c < rows) {
    float l = 0.f;
    const float m = s_ml[c];
    for (int p = 0; p < nparts; ++p) l += sml[2 * (p * kMaxRows + c) + 1] * fast_exp2(sml[2 * (p * kMaxRows + c)] - m);
    s_ml[kMaxRows + c] = l;
  }
  __syncthreads();
#pragma unroll
  for (int rho = 0; rho < kMaxRows; ++rho) M[rho] = s_ml[rho];
  for (int p0 = 0; p0 < nparts; p0 += 4) {
    float ov[4][kMaxRows], mv[4][kMaxRows];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int rho = 0; rho < kMaxRows; ++rho) {
        const bool in = p0 + u < nparts && rho < rows;
        const float* pr = base + ((int64_t)(p0 + u) * kMaxRows + rho) * kPartStride;
        ov[u][rho] = in ? __ldcg(pr + 4 + c) : 0.f;
        mv[u][rho] = in ? __ldcg(pr) : kNeg;
      }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int rho = 0; rho < kMaxRows; ++rho)
        if (p0 + u < nparts && rho < rows) O[rho] += ov[u][rho] * fast_exp2(mv[u][rho] - M[rho]);
  }
#pragma unroll
  for (int rho = 0; rho < kMaxRows; ++rho) {
    if (rho >= rows) break;
    write_row(a, bh, rho, M[rho], s_ml[kMaxRows + rho], O[rho], c);
  }
  if (c == 0) atomicExch(&a.tickets[bh], 0u);  // ready for the next call on this workspace
  return true;
}

// ------------------------------------------------------------ fused ArgTopK
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 20000000ull;  // 20 ms: a normal wait is a few microseconds

// ArgTopK(A_{1,:}) at the end of the attention (SpeCache page, Algorithm 3):
// the CTA that combined a (b, hkv) publishes its log-sum-exp; every CTA of the
// (b, hkv) waits for it (bounded: on expiry it sets the fault word and goes
// on), scores its own chunk's positions from the speculative logits it and its
// siblings wrote, S(n) = sum_h 2^(log2e (l_h(n) - lse_h)), and keeps its
// chunk's top-k' (k' = min(k, chunk length), ties to the lower position) as
// candidates in the workspace.  The last CTA of the (b, hkv) to finish (a
// second ticket) selects the final k from the candidates, which lie in
// ascending position, and writes idx and the bitmap.  Every globally selected
// position is among its chunk's candidates.
template <int BITS, int GROUP>
__device__ __forceinline__ void select_epilogue(const AttnArgs& a, uint8_t* dyn, SelShared<kThreads>& sh,
                                                bool combined, int* s_flag, float* s_nlse, uint32_t tmem_base) {
  const int tid = threadIdx.x;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv), G = a.G;
  if (combined) {
    if (tid == 0) {
      __threadfence();  // the log-sum-exp this CTA wrote, then the flag
      atomicExch(&a.ready[bh], 1u);
    }
  } else if (tid == 0) {
    const uint64_t t0 = global_ns();
    while (ld_acquire_gpu(&a.ready[bh]) == 0u) {
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicOr(a.fault, 1u);
        break;
      }
      __nanosleep(200);
    }
  }
  __syncthreads();
  if (tid < G) s_nlse[tid] = -__ldcg(a.lse + ((int64_t)b * 2 + 1) * a.Hq + hk * G + tid) * 1.4426950408889634f;
  __syncthreads();

  // ---- scores of this chunk's positions, then its candidates ----
  const int gpc32 = a.groups_per_chunk * kGroup;
  const int p0 = blockIdx.x * gpc32;
  const int len = max(0, min(a.nq, p0 + gpc32) - p0);  // multiple of 32
  uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
  if (a.sel_onchip) {
    // From TMEM: warp w holds its records' halves, lane = token, column 4 (NH it + hf) + head, the
    // logits as the separate path stores them (natural-log units); the fetched positions' logits are
    // the prologue's, in sel_rowlog, and replace the low-bit ones below.
    constexpr int NH = GROUP / 32;
    const int lane = tid & 31, warp = tid >> 5;
    const int u_begin = blockIdx.x * (a.groups_per_chunk / NH);
    const int u_end = min(a.nq / GROUP, u_begin + a.groups_per_chunk / NH);
    const int n_my = (u_end - u_begin - warp + kWarps - 1) / kWarps;
    const uint32_t tw = tmem_base + ((uint32_t)(32 * warp) << 16);
    for (int it = 0; it < n_my; ++it)
      for (int hf = 0; hf < NH; ++hf) {
        const float4 v = tmem_ld4(tw + 4 * (NH * it + hf));
        const float l[4] = {v.x, v.y, v.z, v.w};
        float sc = 0.f;
        for (int gi = 0; gi < G; ++gi) sc += fast_exp2(fmaf(l[gi], 1.4426950408889634f, s_nlse[gi]));
        const int g = NH * (u_begin + warp + it * kWarps) + hf;
        keys[32 * g + lane - p0] = __float_as_uint(sc);
      }
    // TMEM is released here, before the candidates, by the warp that allocated it
    tmem_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
      tmem_fence_after_sync();
      tmem_dealloc(tmem_base, kTmemCols);
    }
    if (a.k > 0) {
      // the fetched positions in [p0, p0 + len): idx is ascending (then -1 padding)
      const int32_t* ix = a.idx + bh * a.k;
      for (int j = tid; j < a.k; j += kThreads) {
        const int p = ix[j];
        if (p >= p0 && p < p0 + len) {
          const float* lr = a.sel_rowlog + (bh * a.k + j) * 4;
          float sc = 0.f;
          for (int gi = 0; gi < G; ++gi) sc += fast_exp2(fmaf(lr[gi], 1.4426950408889634f, s_nlse[gi]));
          keys[p - p0] = __float_as_uint(sc);
        }
      }
    }
  } else {
    const float* lrow = a.spec_logits + (bh * G) * (int64_t)a.Lcap + p0;
    for (int i = 4 * tid; i < len; i += 4 * kThreads) {
      float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int gi = 0; gi < G; ++gi) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(lrow + (int64_t)gi * a.Lcap + i));
        const float nl = s_nlse[gi];
        sc.x += fast_exp2(fmaf(v.x, 1.4426950408889634f, nl));
        sc.y += fast_exp2(fmaf(v.y, 1.4426950408889634f, nl));
        sc.z += fast_exp2(fmaf(v.z, 1.4426950408889634f, nl));
        sc.w += fast_exp2(fmaf(v.w, 1.4426950408889634f, nl));
      }
      *reinterpret_cast<uint4*>(keys + i) =
          make_uint4(__float_as_uint(sc.x), __float_as_uint(sc.y), __float_as_uint(sc.z), __float_as_uint(sc.w));
    }
  }
  __syncthreads();
  const int kloc = min(a.sel_keff, len);
  if (kloc > 0) {
    uint32_t* wgt = keys + len;
    uint32_t* weq = wgt + (len >> 5);
    uint32_t* cand = a.cand + ((bh * a.chunks + blockIdx.x) * (int64_t)a.cand_cap) * 2;
    uint32_t T, need;
    cta_radix_select<kThreads>(keys, len, (uint32_t)kloc, sh, T, need);
    ordered_take<kThreads>(keys, len, T, need, wgt, weq, sh, [&](int i, uint32_t r) {
      cand[2 * r] = keys[i];
      cand[2 * r + 1] = (uint32_t)(p0 + i);
    });
  }

  // ---- the last CTA of the (b, hkv) merges the chunks' candidates ----
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_flag = (atomicAdd(&a.tickets2[bh], 1u) == (unsigned)(a.chunks - 1));
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  int M = 0;
  for (int c = 0; c < a.chunks; ++c) M += min(a.sel_keff, max(0, min(a.nq, (c + 1) * gpc32) - c * gpc32));
  const int nwq = a.nq >> 5;
  uint32_t* mkey = reinterpret_cast<uint32_t*>(dyn);
  uint32_t* mpos = mkey + M;
  uint32_t* sbm = mpos + M;
  uint32_t* wgt = sbm + nwq;
  uint32_t* weq = wgt + ((M + 31) >> 5);
  for (int c = 0, off = 0; c < a.chunks; ++c) {
    const int cnt = min(a.sel_keff, max(0, min(a.nq, (c + 1) * gpc32) - c * gpc32));
    const uint32_t* cand = a.cand + ((bh * a.chunks + c) * (int64_t)a.cand_cap) * 2;
    for (int i = tid; i < cnt; i += kThreads) {
      const uint2 kv = __ldcg(reinterpret_cast<const uint2*>(cand) + i);
      mkey[off + i] = kv.x;
      mpos[off + i] = kv.y;
    }
    off += cnt;
  }
  for (int w = tid; w < nwq; w += kThreads) sbm[w] = 0u;
  __syncthreads();
  int32_t* out = a.sel_idx + bh * a.sel_k;
  if (a.sel_keff > 0) {
    uint32_t T, need;
    cta_radix_select<kThreads>(mkey, M, (uint32_t)a.sel_keff, sh, T, need);
    ordered_take<kThreads>(mkey, M, T, need, wgt, weq, sh, [&](int i, uint32_t r) {
      const uint32_t p = mpos[i];
      out[r] = (int32_t)p;
      atomicOr(&sbm[p >> 5], 1u << (p & 31u));
    });
  }
  for (int j = a.sel_keff + tid; j < a.sel_k; j += kThreads) out[j] = -1;
  if (a.sel_src != nullptr) {  // where each selected position sat in this launch's idx
    __syncthreads();           // every entry of the selection is written
    for (int r = tid; r < a.sel_k; r += kThreads)
      a.sel_src[bh * a.sel_k + r] = r < a.sel_keff ? find_in_prev(a.idx + bh * a.k, a.k, (uint32_t)out[r]) : -1;
  }
  uint32_t* bm = a.sel_bitmap + bh * a.q_groups_cap;
  for (int w = tid; w < a.q_groups_cap; w += kThreads) bm[w] = w < nwq ? sbm[w] : 0u;
  if (tid == 0) {  // every CTA of this (b, hkv) is past its wait: ready for the next call
    atomicExch(&a.ready[bh], 0u);
    atomicExch(&a.tickets2[bh], 0u);
  }
}

// Clustered combine: when all CTAs of a (b, hkv) form one thread-block
// cluster, each keeps its partial in shared memory and, after a cluster
// barrier, CTA r merges query row r (r, r + chunks, ...) from every CTA's
// partial through distributed shared memory: no partials in global memory,
// no fences, no ticket.
__device__ __forceinline__ void cluster_combine(CtaMerge& sm, const AttnArgs& a, float* cpart) {
  namespace cgx = cooperative_groups;
  cgx::cluster_group cluster = cgx::this_cluster();
  __syncthreads();
  const int c = threadIdx.x;  // channel
  const int rows = 2 * a.G;
  cta_merge_rows(sm, rows, c, cpart);
  cluster.sync();
  const unsigned n = cluster.num_blocks();
  const int64_t bh = blockIdx.y;
  for (int rho = (int)cluster.block_rank(); rho < rows; rho += (int)n) {
    float M = kNeg;
    for (unsigned p = 0; p < n; ++p) M = fmaxf(M, cluster.map_shared_rank(cpart, p)[rho * kPartStride]);
    float L = 0.f, O = 0.f;
#pragma unroll 4
    for (unsigned p = 0; p < n; ++p) {
      const float* pr = cluster.map_shared_rank(cpart, p) + rho * kPartStride;
      const float f = fast_exp2(pr[0] - M);
      L += pr[1] * f;
      O += pr[4 + c] * f;
    }
    write_row(a, bh, rho, M, L, O, c);
  }
  cluster.sync();  // every CTA's partial stays readable until all rows are merged
}

template <int BITS, int GROUP, bool MERGED, bool FETCH, bool TOPK, bool CLUSTER>
__global__ void __launch_bounds__(kThreads, 4) attn_kernel(AttnArgs a) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  __shared__ int s_last;
  __shared__ uint32_t s_tmem;  // TMEM base of the on-chip selection
  static_assert(sizeof(SelShared<kThreads>) <= kMaxRows * kTilePitch * sizeof(float),
                "the selection's shared state reuses the query tile");
  __shared__ float s_ml[2 * kMaxRows];
  __shared__ float s_w[kMaxCluster * kMaxRows];  // the combine's partial weights
  __shared__ __align__(16) float s_q[kMaxRows * kTilePitch];
  CtaMerge& merge = *reinterpret_cast<CtaMerge*>(dyn_smem);
  grid_dependency_sync();  // nothing is read or written before the previous kernel is done
  auto fill_query = [&]() {
    // scaled query rows of this (b, hkv): rho = i * G + gi for token i, head gi
    const int64_t bh = blockIdx.y;
    const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv), G = a.G;
    for (int e = threadIdx.x; e < kMaxRows * kD / 4; e += kThreads) {
      const int rho = e / (kD / 4), c4 = e % (kD / 4);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rho < 2 * G) {
        const int qi = rho / G, gi = rho % G;
        const uint2 qq = reinterpret_cast<const uint2*>(a.q + (((int64_t)b * 2 + qi) * a.Hq + hk * G + gi) * kD)[c4];
        v = make_float4(bf16_to_f32(qq.x & 0xFFFFu) * a.qscale, bf16_to_f32(qq.x >> 16) * a.qscale,
                        bf16_to_f32(qq.y & 0xFFFFu) * a.qscale, bf16_to_f32(qq.y >> 16) * a.qscale);
      }
      *reinterpret_cast<float4*>(s_q + rho * kTilePitch + 4 * c4) = v;
    }
    __syncthreads();
  };
  if constexpr (TOPK) {
    if (a.sel_onchip && threadIdx.x < 32) {  // warp 0 allocates; the query fill's barrier publishes it
      tmem_alloc(&s_tmem, kTmemCols);
      tmem_fence_before_sync();
    }
  }
  lowbit_cta<BITS, GROUP, MERGED, FETCH, TOPK>(a, dyn_smem, s_q, merge, &s_tmem, fill_query);
  if constexpr (CLUSTER) {
    cluster_combine(merge, a, reinterpret_cast<float*>(dyn_smem + kClusterPartOffset));
    return;
  }
  constexpr int kPartCap = Layout<BITS, GROUP>::DYN / (int)(kMaxRows * kPartStride * sizeof(float));
  static_assert(kPartCap <= kMaxCluster, "the combine's weight table holds kMaxCluster partials");
  const bool combined = merge_store_combine(merge, a, &s_last, s_ml, s_w, kPartCap);
  if constexpr (TOPK) {
    __syncthreads();  // the query tile and the merge buffer are free from here on
    select_epilogue<BITS, GROUP>(a, dyn_smem, *reinterpret_cast<SelShared<kThreads>*>(s_q), combined, &s_last, s_ml,
                                 s_tmem);
  }
}

// ---------------------------------------------------------------- per-variant host helpers

// The kernels of one (bit width, group size), as the host code of
// attention.cu sees them.
struct AttnVariant {
  int smem;                                                // dynamic shared memory of one CTA
  int (*resident_ctas)(bool fetch);                        // resident CTAs per SM (occupancy query)
  bool (*cluster_fits)(bool merged, bool fetch, int chunks, int64_t BH);
  // the attention grid (not the combine kernel that may follow it)
  cudaError_t (*launch)(const AttnArgs& a, int64_t BH, cudaStream_t stream, bool merged, bool fetch, bool topk,
                        bool clustered);
};
const AttnVariant& attn_variant_b1g32();
const AttnVariant& attn_variant_b1g64();
const AttnVariant& attn_variant_b2g32();
const AttnVariant& attn_variant_b2g64();

template <int BITS, int GROUP>
struct AttnVariantImpl {
  static constexpr int kSmem = Layout<BITS, GROUP>::DYN;

  // Resident attention CTAs per SM on the current device (occupancy query,
  // cached per device and fetch variant).
  template <bool FETCH>
  static int resident() {
    static int cached[64] = {};
    static unsigned long long configured = 0ull;
    const int dev = spc_host::current_device();
    if (dev >= 0 && dev < 64) {
      const int c = __atomic_load_n(&cached[dev], __ATOMIC_ACQUIRE);
      if (c > 0) return c;
    }
    int n = 0;
    auto* fn = attn_kernel<BITS, GROUP, true, FETCH, false, false>;
    cudaError_t e = spc_host::ensure_smem_limit(configured, fn, kSmem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, kSmem);
    if (e != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 2;
    }
    if (dev >= 0 && dev < 64) __atomic_store_n(&cached[dev], n, __ATOMIC_RELEASE);
    return n;
  }
  static int resident_ctas(bool fetch) { return fetch ? resident<true>() : resident<false>(); }

  template <bool MERGED, bool FETCH, bool TOPK, bool CLUSTER>
  static cudaError_t launch_one(const AttnArgs& a, int64_t BH, cudaStream_t stream) {
    static_assert(sizeof(CtaMerge) <= (size_t)kSmem, "merge buffer fits in the dynamic shared memory");
    static_assert(kClusterPartOffset + kMaxRows * kPartStride * 4 <= kSmem,
                  "the clustered combine's partial fits behind the merge buffer");
    auto* fn = attn_kernel<BITS, GROUP, MERGED, FETCH, TOPK, CLUSTER>;
    static unsigned long long configured = 0ull;  // one per instantiation
    cudaError_t e = spc_host::ensure_smem_limit(configured, fn, kSmem);
    if (e != cudaSuccess) return e;
    // programmatic serialisation: the launch overlaps the previous kernel's tail
    // (the kernel waits for it before touching any data); clustered: the CTAs of
    // a (b, hkv) form one cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.chunks, (unsigned)BH, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)a.chunks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CLUSTER ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, fn, a);
  }

  // Whether the CTAs of every (b, hkv) can form one cluster (at most
  // kMaxCluster CTAs) with all B*Hkv clusters resident at once (occupancy
  // query, cached per device and cluster size).
  template <bool MERGED, bool FETCH>
  static bool fits(int chunks, int64_t BH) {
    if (chunks < 2 || chunks > kMaxCluster) return false;
    static int cached[64][kMaxCluster + 1] = {};  // 0 unknown, else 1 + resident clusters
    static unsigned long long configured = 0ull, nonportable = 0ull;
    const int dev = spc_host::current_device();
    if (dev >= 0 && dev < 64) {
      const int c = __atomic_load_n(&cached[dev][chunks], __ATOMIC_ACQUIRE);
      if (c > 0) return (int64_t)(c - 1) >= BH;
    }
    auto* fn = attn_kernel<BITS, GROUP, MERGED, FETCH, false, true>;
    int n = 0;
    cudaError_t e = spc_host::ensure_smem_limit(configured, fn, kSmem);
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (e == cudaSuccess && chunks > 8 && !(__atomic_load_n(&nonportable, __ATOMIC_ACQUIRE) & bit)) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e == cudaSuccess && bit != 0ull) __atomic_fetch_or(&nonportable, bit, __ATOMIC_ACQ_REL);
    }
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)chunks, (unsigned)BH, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = kSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)chunks;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    if (dev >= 0 && dev < 64) __atomic_store_n(&cached[dev][chunks], n + 1, __ATOMIC_RELEASE);
    return (int64_t)n >= BH;
  }
  static bool cluster_fits(bool merged, bool fetch, int chunks, int64_t BH) {
    return merged ? (fetch ? fits<true, true>(chunks, BH) : fits<true, false>(chunks, BH))
                  : (fetch ? fits<false, true>(chunks, BH) : fits<false, false>(chunks, BH));
  }

  // The attention grid: with the fused selection (its last CTA per (b, hkv)
  // combines; merged only), clustered (the CTAs combine through distributed
  // shared memory), or storing its partials for combine_kernel.
  static cudaError_t launch(const AttnArgs& a, int64_t BH, cudaStream_t stream, bool merged, bool fetch, bool topk,
                            bool clustered) {
    if (topk)
      return fetch ? launch_one<true, true, true, false>(a, BH, stream)
                   : launch_one<true, false, true, false>(a, BH, stream);
    if (merged) {
      if (clustered)
        return fetch ? launch_one<true, true, false, true>(a, BH, stream)
                     : launch_one<true, false, false, true>(a, BH, stream);
      return fetch ? launch_one<true, true, false, false>(a, BH, stream)
                   : launch_one<true, false, false, false>(a, BH, stream);
    }
    if (clustered)
      return fetch ? launch_one<false, true, false, true>(a, BH, stream)
                   : launch_one<false, false, false, true>(a, BH, stream);
    return fetch ? launch_one<false, true, false, false>(a, BH, stream)
                 : launch_one<false, false, false, false>(a, BH, stream);
  }

  static AttnVariant table() { return AttnVariant{kSmem, &resident_ctas, &cluster_fits, &launch}; }
};

}  // namespace spc
