// Attn([T_t, T'_{t+1}], C' U C_kappa): the two-query decode attention of the
// SpeCache page (section 3 "Decoding", Algorithm 3) over the packed low-bit
// copy C', with the fetched 16-bit rows C_kappa used in place of their
// low-bit copies, plus the bf16 residual window.
//
// Work split (flash-decoding style split-K over tokens):
//   * grid (chunks + 1, B*Hkv).  CTAs 0..chunks-1 scan 32-token groups of C';
//     CTA `chunks` handles every 16-bit row (residual window and fetched rows).
//   * each CTA writes one partial (running max, sum, unnormalised output) per
//     query row to the workspace; attn_combine_kernel merges them.
//
// Low-bit tile arithmetic.  With k^ = z + s*b (b the code, z and s per key
// group), the logit of query row q is  sum_c q_c s_c b_c + sum_c q_c z_c.  The
// first term is a 16x8x16 tensor-core product per 8 tokens and 16 channels:
//   A = (q o s) for the 8 query rows (2 tokens x G <= 4 heads), split into an
//       fp16 high part (rows 0..7) and the fp16 residual (rows 8..15), so the
//       speculative logits keep ~22 significant bits;
//   B = the key bits, exact {0, 1} (or {0, 2} for the high plane at 2 bits).
// The value side o = sum_n p_n (z_n + s_n b_n) is the same product with
// A = value bits (channels x tokens) and B = p o s (tokens x query rows); the
// p*z term is accumulated on CUDA cores.  Softmax runs in base 2 with the
// scale folded into q.
#include <math_constants.h>

#include "common.cuh"

namespace spc {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;
constexpr float kNeg = -1e30f;  // finite "minus infinity": keeps max/rescale arithmetic NaN-free
constexpr int kPartStride = 132; // floats per (chunk, row) partial: m, l, pad, pad, o[128]

struct AttnArgs {
  const uint8_t* records;
  const uint16_t* resid;
  const uint16_t* q;
  const int32_t* idx;
  const uint32_t* bitmap;
  const uint16_t* staging;
  float* spec_logits;
  float* ws;
  int32_t k;
  int32_t Hq, Hkv, G, nq, r, q_groups_cap, resid_cap;
  int32_t chunks, groups_per_chunk;
  int32_t Lcap;
  float qscale;  // softmax scale * log2(e)
};

// {bit r, bit r+16} of w as an f16x2 pair of {0, v} (v = 1.0 or 2.0).
template <uint32_t kOne>
__device__ __forceinline__ uint32_t expand_pair(uint32_t w, int r) {
  return ((w >> r) & 0x00010001u) * kOne;
}

// Writes this warp's per-row state to shared memory, then (after a barrier)
// the CTA's merged partial to the workspace.
struct CtaMerge {
  float m[kWarps][kMaxRows];
  float l[kWarps][kMaxRows];
  float o[kWarps][kMaxRows][kD];
};

__device__ void cta_merge_and_store(CtaMerge& sm, const AttnArgs& a, int64_t bh, int chunk) {
  __syncthreads();
  const int c = threadIdx.x;  // channel
  const int rows = 2 * a.G;
  float* part = a.ws + ((bh * (a.chunks + 1) + chunk) * kMaxRows) * kPartStride;
  for (int rho = 0; rho < rows; ++rho) {
    float M = kNeg;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w][rho]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = fast_exp2(sm.m[w][rho] - M);
      L += sm.l[w][rho] * f;
      O += sm.o[w][rho][c] * f;
    }
    float* pr = part + rho * kPartStride;
    if (c == 0) {
      pr[0] = M;
      pr[1] = L;
    }
    pr[4 + c] = O;
  }
}

template <int BITS, bool MERGED>
__global__ void __launch_bounds__(kThreads, 2) attn_lowbit_kernel(AttnArgs a) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  constexpr int RB = 1024 * (BITS + 1);
  constexpr int KMETA = 512 * BITS;
  constexpr int VCODES = KMETA + 512;
  constexpr int VMETA = VCODES + 512 * BITS;
  __shared__ CtaMerge merge;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.y;
  const int chunk = blockIdx.x;
  const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv);
  const int G = a.G;
  const bool row_valid = gid < 2 * G;

  uint8_t* stage = dyn_smem + (size_t)warp * kStages * RB;

  // Scaled query of row gid at this lane's 32 channels, ordered
  // m = 4*kc + 2*h + half  <->  channel 16*kc + 2*t + 8*h + half.
  float qv[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) qv[m] = 0.f;
  if (row_valid) {
    const int i = gid / G, gi = gid % G;
    const uint16_t* qrow = a.q + (((int64_t)b * 2 + i) * a.Hq + hk * G + gi) * kD;
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      const int ch = 16 * (m >> 2) + 2 * t + 8 * ((m >> 1) & 1) + (m & 1);
      qv[m] = bf16_to_f32(qrow[ch]) * a.qscale;
    }
  }

  const int g_begin = chunk * a.groups_per_chunk;
  const int g_end = min(a.nq / kGroup, g_begin + a.groups_per_chunk);
  const int n_my = (g_end - g_begin - warp + kWarps - 1) / kWarps;  // groups of this warp
  const uint8_t* rec_base = a.records + (bh * a.q_groups_cap) * (int64_t)RB;

  auto issue = [&](int item) {
    if (item < n_my) {
      const int g = g_begin + warp + item * kWarps;
      const uint8_t* src = rec_base + (int64_t)g * RB;
      uint8_t* dst = stage + (item % kStages) * RB;
#pragma unroll
      for (int u = 0; u < RB / 512; ++u) cp_async16(dst + 16 * (lane + 32 * u), src + 16 * (lane + 32 * u));
    }
    cp_async_commit();
  };

  float m_run = kNeg, l_run = 0.f;
  float zacc[4] = {0.f, 0.f, 0.f, 0.f};
  float oacc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;

  const bool spec_row = row_valid && gid >= G && a.spec_logits != nullptr;
  float* spec_out = spec_row ? a.spec_logits + ((bh * G + (gid - G)) * (int64_t)a.Lcap) : nullptr;

#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) issue(s);

#pragma unroll 1
  for (int it = 0; it < n_my; ++it) {
    issue(it + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const uint8_t* R = stage + (it % kStages) * RB;
    const int g = g_begin + warp + it * kWarps;

    // ---- key group: A fragments (q o s, hi/lo) and the z bias ----
    uint32_t afr[8][4];
    float bias = 0.f;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      const uint4 mm = *reinterpret_cast<const uint4*>(R + KMETA + 128 * t + 16 * kc);
      const uint32_t mw[4] = {mm.x, mm.y, mm.z, mm.w};
      float wv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = bf16_to_f32(mw[e] & 0xFFFFu), hi = bf16_to_f32(mw[e] >> 16);
        float z, sc;
        if (BITS == 1) {
          z = (3.f * lo + hi) * 0.25f;
          sc = (hi - lo) * 0.5f;
        } else {
          z = lo;
          sc = (hi - lo) * (1.f / 3.f);
        }
        wv[e] = qv[4 * kc + e] * sc;
        bias = fmaf(qv[4 * kc + e], z, bias);
      }
      const uint32_t h01 = pack_f16x2(wv[0], wv[1]);
      const uint32_t h23 = pack_f16x2(wv[2], wv[3]);
      const float2 f01 = unpack_f16x2(h01), f23 = unpack_f16x2(h23);
      afr[kc][0] = h01;
      afr[kc][2] = h23;
      afr[kc][1] = pack_f16x2(wv[0] - f01.x, wv[1] - f01.y);
      afr[kc][3] = pack_f16x2(wv[2] - f23.x, wv[3] - f23.y);
    }
    bias += __shfl_xor_sync(0xFFFFFFFFu, bias, 1);
    bias += __shfl_xor_sync(0xFFFFFFFFu, bias, 2);

    // ---- QK: 4 token tiles of 8 ----
    const uint4 kw0 = *reinterpret_cast<const uint4*>(R + 16 * lane);
    const uint32_t kwords0[4] = {kw0.x, kw0.y, kw0.z, kw0.w};
    uint32_t kwords1[4] = {0u, 0u, 0u, 0u};
    if (BITS == 2) {
      const uint4 kw1 = *reinterpret_cast<const uint4*>(R + 512 + 16 * lane);
      kwords1[0] = kw1.x; kwords1[1] = kw1.y; kwords1[2] = kw1.z; kwords1[3] = kw1.w;
    }
    float lg[4][2];
    const uint32_t bm = MERGED ? a.bitmap[bh * a.q_groups_cap + g] : 0u;
    float gmax = kNeg;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (BITS == 2) {
#pragma unroll
        for (int kc = 0; kc < 8; ++kc)
          mma_16816(acc, afr[kc], expand_pair<0x4000u>(kwords1[nt], 2 * kc),
                    expand_pair<0x4000u>(kwords1[nt], 2 * kc + 1));
      }
#pragma unroll
      for (int kc = 0; kc < 8; ++kc)
        mma_16816(acc, afr[kc], expand_pair<0x3C00u>(kwords0[nt], 2 * kc),
                  expand_pair<0x3C00u>(kwords0[nt], 2 * kc + 1));
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = 8 * nt + 2 * t + e;
        const bool masked = MERGED && ((bm >> tok) & 1u);
        const float l = acc[e] + acc[2 + e] + bias;
        lg[nt][e] = masked ? kNeg : l;
        gmax = fmaxf(gmax, lg[nt][e]);
      }
      if (spec_row) {
        const int tok = 8 * nt + 2 * t;
        float* dst = spec_out + (int64_t)g * kGroup + tok;
        const bool m0 = MERGED && ((bm >> tok) & 1u), m1 = MERGED && ((bm >> (tok + 1)) & 1u);
        if (!m0 && !m1) {
          *reinterpret_cast<float2*>(dst) =
              make_float2(lg[nt][0] * CUDART_LN2_F, lg[nt][1] * CUDART_LN2_F);
        } else {
          if (!m0) dst[0] = lg[nt][0] * CUDART_LN2_F;
          if (!m1) dst[1] = lg[nt][1] * CUDART_LN2_F;
        }
      }
    }

    // ---- online softmax (base 2) ----
    gmax = fmaxf(gmax, __shfl_xor_sync(0xFFFFFFFFu, gmax, 1));
    gmax = fmaxf(gmax, __shfl_xor_sync(0xFFFFFFFFu, gmax, 2));
    const float m_new = fmaxf(m_run, gmax);
    const float alpha = fast_exp2(m_run - m_new);
    if (__any_sync(0xFFFFFFFFu, m_new != m_run)) {
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
#pragma unroll
      for (int cg = 0; cg < 4; ++cg) zacc[cg] *= alpha;
      m_run = m_new;
    }
    float p[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[nt][e] = (lg[nt][e] == kNeg) ? 0.f : fast_exp2(lg[nt][e] - m_run);
        l_run += p[nt][e];
      }

    // ---- PV: two 16-token chunks ----
    const uint4 vw0 = *reinterpret_cast<const uint4*>(R + VCODES + 16 * lane);
    const uint32_t vwords0[4] = {vw0.x, vw0.y, vw0.z, vw0.w};
    uint32_t vwords1[4] = {0u, 0u, 0u, 0u};
    if (BITS == 2) {
      const uint4 vw1 = *reinterpret_cast<const uint4*>(R + VCODES + 512 + 16 * lane);
      vwords1[0] = vw1.x; vwords1[1] = vw1.y; vwords1[2] = vw1.z; vwords1[3] = vw1.w;
    }
#pragma unroll
    for (int c16 = 0; c16 < 2; ++c16) {
      const float ps[4] = {p[2 * c16][0], p[2 * c16][1], p[2 * c16 + 1][0], p[2 * c16 + 1][1]};
      float sv[4][4], zv[4][4];  // [slot][cg]
#pragma unroll
      for (int slot = 0; slot < 4; ++slot) {
        const uint4 mm = *reinterpret_cast<const uint4*>(R + VMETA + 128 * t + 64 * c16 + 16 * slot);
        const uint32_t mw[4] = {mm.x, mm.y, mm.z, mm.w};
#pragma unroll
        for (int cg = 0; cg < 4; ++cg) {
          const float lo = bf16_to_f32(mw[cg] & 0xFFFFu), hi = bf16_to_f32(mw[cg] >> 16);
          if (BITS == 1) {
            zv[slot][cg] = (3.f * lo + hi) * 0.25f;
            sv[slot][cg] = (hi - lo) * 0.5f;
          } else {
            zv[slot][cg] = lo;
            sv[slot][cg] = (hi - lo) * (1.f / 3.f);
          }
        }
      }
      uint32_t bfr[4][2];
#pragma unroll
      for (int cg = 0; cg < 4; ++cg) {
        bfr[cg][0] = pack_f16x2(ps[0] * sv[0][cg], ps[1] * sv[1][cg]);
        bfr[cg][1] = pack_f16x2(ps[2] * sv[2][cg], ps[3] * sv[3][cg]);
        zacc[cg] = fmaf(ps[0], zv[0][cg], zacc[cg]);
        zacc[cg] = fmaf(ps[1], zv[1][cg], zacc[cg]);
        zacc[cg] = fmaf(ps[2], zv[2][cg], zacc[cg]);
        zacc[cg] = fmaf(ps[3], zv[3][cg], zacc[cg]);
      }
      const uint32_t wa = vwords0[2 * c16], wb = vwords0[2 * c16 + 1];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t af[4] = {expand_pair<0x3C00u>(wa, 2 * mt), expand_pair<0x3C00u>(wa, 2 * mt + 1),
                          expand_pair<0x3C00u>(wb, 2 * mt), expand_pair<0x3C00u>(wb, 2 * mt + 1)};
        mma_16816(oacc[mt], af, bfr[mt >> 1][0], bfr[mt >> 1][1]);
      }
      if (BITS == 2) {
        const uint32_t wa1 = vwords1[2 * c16], wb1 = vwords1[2 * c16 + 1];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t af[4] = {expand_pair<0x4000u>(wa1, 2 * mt), expand_pair<0x4000u>(wa1, 2 * mt + 1),
                            expand_pair<0x4000u>(wb1, 2 * mt), expand_pair<0x4000u>(wb1, 2 * mt + 1)};
          mma_16816(oacc[mt], af, bfr[mt >> 1][0], bfr[mt >> 1][1]);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- warp partial -> shared memory ----
  l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 1);
  l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 2);
#pragma unroll
  for (int cg = 0; cg < 4; ++cg) {
    zacc[cg] += __shfl_xor_sync(0xFFFFFFFFu, zacc[cg], 1);
    zacc[cg] += __shfl_xor_sync(0xFFFFFFFFu, zacc[cg], 2);
  }
  if (t == 0) {
    merge.m[warp][gid] = m_run;
    merge.l[warp][gid] = l_run;
  }
  __syncwarp();
  // oacc[mt]: (channel 16mt+gid, row 2t), (16mt+gid, 2t+1), (16mt+gid+8, 2t), (16mt+gid+8, 2t+1)
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    merge.o[warp][2 * t][16 * mt + gid] = oacc[mt][0];
    merge.o[warp][2 * t + 1][16 * mt + gid] = oacc[mt][1];
    merge.o[warp][2 * t][16 * mt + gid + 8] = oacc[mt][2];
    merge.o[warp][2 * t + 1][16 * mt + gid + 8] = oacc[mt][3];
  }
  __syncwarp();
  // add the p*z term of row gid: zacc[cg] applies to channels 32cg .. 32cg+31
#pragma unroll
  for (int cg = 0; cg < 4; ++cg)
#pragma unroll
    for (int q8 = 0; q8 < 8; ++q8) merge.o[warp][gid][32 * cg + 8 * t + q8] += zacc[cg];
  cta_merge_and_store(merge, a, bh, chunk);
}

// CTA `chunks` of each (b, hkv): all 16-bit rows (residual window, then the
// fetched rows) on CUDA cores, one token per lane for the logits and four
// channels per lane for the value product.
__global__ void __launch_bounds__(kThreads) attn_bf16_rows_kernel(AttnArgs a) {
  __shared__ CtaMerge merge;
  __shared__ float qs[kMaxRows][kD];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv);
  const int G = a.G, rows = 2 * G;
  for (int i = threadIdx.x; i < kMaxRows * kD; i += kThreads) {
    const int rho = i / kD, c = i % kD;
    float v = 0.f;
    if (rho < rows) {
      const int qi = rho / G, gi = rho % G;
      v = bf16_to_f32(a.q[(((int64_t)b * 2 + qi) * a.Hq + hk * G + gi) * kD + c]) * a.qscale;
    }
    qs[rho][c] = v;
  }
  __syncthreads();

  const int n_rows = a.r + a.k;
  const int n_batches = (n_rows + 31) / 32;
  float m_run[kMaxRows], l_run[kMaxRows], o[kMaxRows][4];
#pragma unroll
  for (int rho = 0; rho < kMaxRows; ++rho) {
    m_run[rho] = kNeg;
    l_run[rho] = 0.f;
    o[rho][0] = o[rho][1] = o[rho][2] = o[rho][3] = 0.f;
  }
  for (int bt = warp; bt < n_batches; bt += kWarps) {
    const int j = 32 * bt + lane;  // this lane's row for the logits
    const uint16_t* row = nullptr;
    int pos = -1;                   // quantised position of a fetched row
    if (j < a.r) {
      row = a.resid + ((bh * a.resid_cap + j) * 2) * kD;
    } else if (j < n_rows) {
      const int jj = j - a.r;
      pos = a.idx[bh * a.k + jj];
      if (pos >= 0 && pos < a.nq) row = a.staging + ((bh * a.k + jj) * 2) * kD;
    }
    float lg[kMaxRows];
#pragma unroll
    for (int rho = 0; rho < kMaxRows; ++rho) lg[rho] = 0.f;
    if (row != nullptr) {
      const uint4* kr = reinterpret_cast<const uint4*>(row);
#pragma unroll 4
      for (int c8 = 0; c8 < kD / 8; ++c8) {
        const uint4 kk = kr[c8];
        const uint32_t kw[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float k0 = bf16_to_f32(kw[e] & 0xFFFFu), k1 = bf16_to_f32(kw[e] >> 16);
#pragma unroll
          for (int rho = 0; rho < kMaxRows; ++rho)
            lg[rho] = fmaf(qs[rho][8 * c8 + 2 * e + 1], k1, fmaf(qs[rho][8 * c8 + 2 * e], k0, lg[rho]));
        }
      }
    }
    const bool live = row != nullptr;
    if (live && pos >= 0 && a.spec_logits != nullptr) {
      for (int gi = 0; gi < G; ++gi)
        a.spec_logits[(bh * G + gi) * (int64_t)a.Lcap + pos] = lg[G + gi] * CUDART_LN2_F;
    }
    float p[kMaxRows];
#pragma unroll
    for (int rho = 0; rho < kMaxRows; ++rho) {
      float mx = live ? lg[rho] : kNeg;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      const float m_new = fmaxf(m_run[rho], mx);
      const float al = fast_exp2(m_run[rho] - m_new);
      m_run[rho] = m_new;
      p[rho] = live ? fast_exp2(lg[rho] - m_new) : 0.f;
      float ps = p[rho];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, off);
      l_run[rho] = l_run[rho] * al + ps;
      o[rho][0] *= al;
      o[rho][1] *= al;
      o[rho][2] *= al;
      o[rho][3] *= al;
    }
    // value product: lane owns channels 4*lane .. 4*lane+3
    const int nb = min(32, n_rows - 32 * bt);
    for (int jj = 0; jj < nb; ++jj) {
      const int jr = 32 * bt + jj;
      const uint16_t* vrow = nullptr;
      if (jr < a.r) {
        vrow = a.resid + ((bh * a.resid_cap + jr) * 2 + 1) * kD;
      } else {
        const int js = jr - a.r;
        const int pj = a.idx[bh * a.k + js];
        if (pj >= 0 && pj < a.nq) vrow = a.staging + ((bh * a.k + js) * 2 + 1) * kD;
      }
      if (vrow == nullptr) continue;  // uniform across the warp
      const uint2 vv = reinterpret_cast<const uint2*>(vrow)[lane];
      const float v0 = bf16_to_f32(vv.x & 0xFFFFu), v1 = bf16_to_f32(vv.x >> 16);
      const float v2 = bf16_to_f32(vv.y & 0xFFFFu), v3 = bf16_to_f32(vv.y >> 16);
#pragma unroll
      for (int rho = 0; rho < kMaxRows; ++rho) {
        const float pj = __shfl_sync(0xFFFFFFFFu, p[rho], jj);
        o[rho][0] = fmaf(pj, v0, o[rho][0]);
        o[rho][1] = fmaf(pj, v1, o[rho][1]);
        o[rho][2] = fmaf(pj, v2, o[rho][2]);
        o[rho][3] = fmaf(pj, v3, o[rho][3]);
      }
    }
  }
  if (lane < kMaxRows) {
    float mv = 0.f, lv = 0.f;
#pragma unroll
    for (int rho = 0; rho < kMaxRows; ++rho)
      if (rho == lane) {
        mv = m_run[rho];
        lv = l_run[rho];
      }
    merge.m[warp][lane] = mv;
    merge.l[warp][lane] = lv;
  }
#pragma unroll
  for (int rho = 0; rho < kMaxRows; ++rho)
#pragma unroll
    for (int e = 0; e < 4; ++e) merge.o[warp][rho][4 * lane + e] = o[rho][e];
  cta_merge_and_store(merge, a, bh, a.chunks);
}

// Merge the split-K partials of one (b, hkv, query row): o in bf16 and the
// natural-log normaliser.
__global__ void __launch_bounds__(kD) attn_combine_kernel(AttnArgs a, uint16_t* out, float* lse) {
  const int64_t bh = blockIdx.y;
  const int rho = blockIdx.x;
  const int c = threadIdx.x;
  const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv);
  const int G = a.G, qi = rho / G, gi = rho % G;
  const int nparts = a.chunks + 1;
  const float* part = a.ws + (bh * nparts * kMaxRows + rho) * kPartStride;
  float M = kNeg;
  for (int p = 0; p < nparts; ++p) M = fmaxf(M, part[(int64_t)p * kMaxRows * kPartStride]);
  float L = 0.f, O = 0.f;
  for (int p = 0; p < nparts; ++p) {
    const float* pr = part + (int64_t)p * kMaxRows * kPartStride;
    const float f = fast_exp2(pr[0] - M);
    L += pr[1] * f;
    O += pr[4 + c] * f;
  }
  const int64_t orow = ((int64_t)b * 2 + qi) * a.Hq + hk * G + gi;
  out[orow * kD + c] = f32_to_bf16_rne(L > 0.f ? O / L : 0.f);
  if (c == 0 && lse != nullptr) lse[orow] = L > 0.f ? (M + __log2f(L)) * CUDART_LN2_F : -CUDART_INF_F;
}

// ---------------------------------------------------------------- host side

struct AttnPlan {
  int chunks;
  int groups_per_chunk;
};

AttnPlan attn_plan(const spc_dims* d) {
  const int ng = num_quantized(d->N, d->R) / kGroup;
  AttnPlan p{0, 1};
  if (ng == 0) return p;
  const int64_t BH = (int64_t)d->B * d->Hkv;
  const int64_t target = (int64_t)spc_host::sm_count() * 2;  // resident CTAs at 2 per SM
  int64_t chunks = (target + BH - 1) / BH;
  chunks = std::max<int64_t>(1, std::min<int64_t>(chunks, (ng + kWarps - 1) / kWarps));
  p.groups_per_chunk = (int)((ng + chunks - 1) / chunks);
  p.chunks = (ng + p.groups_per_chunk - 1) / p.groups_per_chunk;
  return p;
}

size_t attn_workspace_bytes(const spc_dims* d) {
  const AttnPlan p = attn_plan(d);
  return (size_t)d->B * d->Hkv * (p.chunks + 1) * kMaxRows * kPartStride * sizeof(float);
}

template <int BITS, bool MERGED>
static cudaError_t launch_lowbit(const AttnArgs& a, int64_t BH, cudaStream_t stream) {
  const int smem = kWarps * kStages * 1024 * (BITS + 1);
  auto* fn = attn_lowbit_kernel<BITS, MERGED>;
  static unsigned long long configured = 0ull;  // one per <BITS, MERGED> instantiation
  cudaError_t e = spc_host::ensure_smem_limit(configured, fn, smem);
  if (e != cudaSuccess) return e;
  fn<<<dim3(a.chunks, (unsigned)BH), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

spc_status launch_attention(const spc_dims* d, const void* records, const uint16_t* resid,
                            const uint16_t* q, const int32_t* idx, const uint32_t* bitmap,
                            const uint16_t* staging, int32_t k, uint16_t* o, float* lse,
                            float* spec_logits, void* ws, cudaStream_t stream) {
  const AttnPlan plan = attn_plan(d);
  AttnArgs a;
  a.records = static_cast<const uint8_t*>(records);
  a.resid = resid;
  a.q = q;
  a.idx = idx;
  a.bitmap = bitmap;
  a.staging = staging;
  a.spec_logits = spec_logits;
  a.ws = static_cast<float*>(ws);
  a.k = k;
  a.Hq = d->Hq;
  a.Hkv = d->Hkv;
  a.G = d->Hq / d->Hkv;
  a.nq = num_quantized(d->N, d->R);
  a.r = d->N - a.nq;
  a.q_groups_cap = d->q_groups_cap;
  a.resid_cap = d->resid_cap;
  a.chunks = plan.chunks;
  a.groups_per_chunk = plan.groups_per_chunk;
  a.Lcap = d->q_groups_cap * kGroup;
  a.qscale = d->scale * 1.4426950408889634f;
  const int64_t BH = (int64_t)d->B * d->Hkv;
  const bool merged = k > 0;
  cudaError_t e = cudaSuccess;
  if (a.chunks > 0) {
    if (d->bits == 1)
      e = merged ? launch_lowbit<1, true>(a, BH, stream) : launch_lowbit<1, false>(a, BH, stream);
    else
      e = merged ? launch_lowbit<2, true>(a, BH, stream) : launch_lowbit<2, false>(a, BH, stream);
  }
  if (e == cudaSuccess) {
    attn_bf16_rows_kernel<<<dim3(1, (unsigned)BH), kThreads, 0, stream>>>(a);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    attn_combine_kernel<<<dim3(2 * a.G, (unsigned)BH), kD, 0, stream>>>(a, o, lse);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

}  // namespace spc
