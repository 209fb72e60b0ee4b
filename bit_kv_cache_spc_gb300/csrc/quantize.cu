// Quant: the KIVI-style low-bit copy C' with SpeCache's 1-bit zero point and
// scale (SpeCache page, section 3, "Original KIVI quantisation" and "Improved
// 1-bit quantisation"; keys per channel, values per token, groups of 32).
//
// One CTA of 128 threads quantises 32-token groups of one (b, hkv) at a time:
// 8 KB of keys and 8 KB of values in, one 2 KB (1-bit) or 3 KB (2-bit) record
// out.  A CTA loads a group's tiles (cp.async) and then codes them; the
// other resident CTAs of the SM (one wave of them, 21 KB of shared memory
// each) overlap one another's loads.  Per group: thread c finds key channel c's min/max and
// parameters; then one warp per key token (and per value token pair) codes a
// conflict-free 16-byte block per lane, and one ballot per code word yields a
// packed word: value words in the record's bit order directly (value groups'
// min/max come from two xor-shuffles inside the same pass), key words token-
// major, then rotated into the record's order in one pass over the words.
// The kernel streams HBM: 512 B read and 64/96 B written per token and KV head.
#include <cstddef>

#include "common.cuh"

namespace spc {

// z and s from the group's min and max, in binary32 exactly as written
// (the __f*_rn intrinsics are never contracted into FMA).
__device__ __forceinline__ void quant_params(int bits, float lo, float hi, float& z, float& s) {
  if (bits == 1) {
    z = __fmul_rn(__fadd_rn(__fmul_rn(3.0f, lo), hi), 0.25f);
    s = __fmul_rn(__fsub_rn(hi, lo), 0.5f);
  } else {
    z = lo;
    s = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
  }
}

// The multiplier that stands in for a division by s: the correctly rounded
// reciprocal; 0 when s == 0 (the code is then 0); NaN when 1/s overflows
// binary32 (s below about 2^-128, a subnormal range), so that every quotient
// of such a group is settled by the IEEE division in quant_code.
__device__ __forceinline__ float quant_recip(float s) {
  if (s == 0.0f) return 0.0f;
  const float rs = __frcp_rn(s);
  return isinf(rs) ? __int_as_float(0x7FC00000) : rs;
}

// clamp(rint(fl((x - z) / s)), 0, 2^bits - 1), 0 when s == 0 (rs == 0 then).
// The product with the correctly rounded reciprocal rs is within 1e-6 of the
// IEEE quotient for the quotients that occur (|q| <= 3), so it decides every
// value whose quotient is farther than 1e-5 from a rounding boundary k + 1/2;
// the IEEE division settles the rest, and every product that is not a number
// (a NaN rs, or an infinite x - z times a zero rs).  At 1 bit the code is 1
// exactly when the quotient exceeds 1/2 (1/2 itself rounds to even, 0); a
// quotient that is not a number gets code 0.
template <int BITS>
__device__ __forceinline__ uint32_t quant_code(float x, float z, float s, float rs) {
  const float d = __fsub_rn(x, z);
  float t = __fmul_rn(d, rs);
  if (BITS == 1) {
    if (!(fabsf(__fsub_rn(t, 0.5f)) >= 1e-5f) && s != 0.0f) t = __fdiv_rn(d, s);
    return t > 0.5f ? 1u : 0u;
  } else {
    const float fr = __fsub_rn(t, floorf(t));
    if (!(fabsf(__fsub_rn(fr, 0.5f)) >= 1e-5f) && s != 0.0f) t = __fdiv_rn(d, s);
    return (uint32_t)fminf(fmaxf(rintf(t), 0.0f), 3.0f);  // fmaxf(NaN, 0) = 0
  }
}

// bf16 bit patterns in value order and back: ord increases with the value
// (-0 just below +0, NaN patterns outside every finite and infinite value).
__device__ __forceinline__ uint32_t bf16_ord(uint32_t b) { return (b & 0x8000u) ? (b ^ 0xFFFFu) : (b | 0x8000u); }
__device__ __forceinline__ uint32_t bf16_unord(uint32_t o) { return (o & 0x8000u) ? (o & 0x7FFFu) : (o ^ 0xFFFFu); }

// The smallest bf16 value x of a group's range [lo, hi] whose code
// quant_code<BITS>(x, z, s, rs) is at least `level` (1 .. 2^BITS - 1), as a
// float; NaN when no x of the range reaches it.  quant_code is the code of
// the IEEE quotient fl(fl(x - z) / s), a non-decreasing function of x, so an
// element of the group has code >= level exactly when x >= the threshold (a
// NaN element compares false, code 0, as quant_code gives it).  Checked at
// both ends of the range first (lo's code is not always 0: when 3 min + max
// overflows binary32, z = -inf and every element codes 1), then in the
// bracket (lo, hi]: the bf16 value at the analytic point z + (level - 1/2) s
// and its two neighbours settle it unless binary32 absorbs x - z over a run
// of bf16 values there (tiny x near a zero midpoint), which bisection then
// resolves.
template <int BITS>
__device__ __forceinline__ float code_threshold(float lo, float hi, float z, float s, float rs, uint32_t level) {
  auto ge = [&](uint32_t o) {
    return quant_code<BITS>(__uint_as_float(bf16_unord(o) << 16), z, s, rs) >= level;
  };
  uint32_t a = bf16_ord(__float_as_uint(lo) >> 16), b = bf16_ord(__float_as_uint(hi) >> 16);
  if (!(a <= b) || !ge(b)) return __int_as_float(0x7FC00000);
  if (ge(a)) return __uint_as_float(bf16_unord(a) << 16);
  // invariant: code(a) < level <= code(b)
  const float guess = __fadd_rn(z, __fmul_rn((float)level - 0.5f, s));
  const uint32_t og = min(max(bf16_ord(__float_as_uint(guess) >> 16), a + 1u), b);
  if (ge(og)) {
    b = og;
    if (og - 1u > a) {
      if (!ge(og - 1u)) return __uint_as_float(bf16_unord(og) << 16);
      b = og - 1u;
    }
  } else {
    a = og;
    if (og + 1u < b) {
      if (ge(og + 1u)) return __uint_as_float(bf16_unord(og + 1u) << 16);
      a = og + 1u;
    }
  }
  while (b - a > 1u) {
    const uint32_t m = (a + b) >> 1;
    if (ge(m)) b = m; else a = m;
  }
  return __uint_as_float(bf16_unord(b) << 16);
}

// min/max of bf16 values carried as floats; -0.0 is stored as +0.0.
__device__ __forceinline__ uint32_t bf16_bits_canonical(float f) {
  return f == 0.0f ? 0u : (__float_as_uint(f) >> 16);
}

struct QuantArgs {
  const uint16_t* k;
  const uint16_t* v;
  uint8_t* records;
  int32_t Hkv, N, nq, q_groups_cap, units_cap;
  int64_t total_groups;  // B * Hkv * (nq / group): the kernel's units of work
};

// Shared memory of the quantiser and the append kernel.  The second tile pair
// is last: the g = 32 quantiser codes one 32-token group at a time and
// launches without it (more resident CTAs hide the loads instead).
struct QuantSmem {
  float kt[3][kD];  // per key channel: 1 bit: the code threshold (code_threshold); 2 bits: z, s, 1/s
  uint32_t klohi[kD];
  uint32_t rec[256 * 3];             // the record being assembled (up to 3 KB)
  uint16_t tile[2][2][kGroup * kD];  // [tile][keys, values][token][channel]
};

// Token pair p of a group (tokens 2p, 2p+1) is where value code words
// (a, t = p & 3, j = 2 * (p >> 3) + ((p >> 2) & 1)) take their bits; the
// (min, max) of token n, channel group cg is value-minmax word 32 t' + m with
// t' = (n & 7) >> 1, m = 16 (n >> 4) + 4 (2 ((n & 15) >> 3) + (n & 1)) + cg.
__device__ __forceinline__ int vmeta_word(int n, int cg) {
  const int n16 = n & 15;
  return 32 * ((n16 & 7) >> 1) + 16 * (n >> 4) + 4 * (2 * (n16 >> 3) + (n16 & 1)) + cg;
}
// At g = 64 a half's 64 value-minmax words hold token n's (min, max) of
// channels 64c .. 64c+63 at word 2m + c, where m = 8 ((n >> 1) & 3) +
// 4 (n >> 4) + 2 ((n >> 3) & 1) + (n & 1) is the lane that reads token n.
__device__ __forceinline__ int vmeta64_word(int n, int c) {
  return 2 * (8 * ((n >> 1) & 3) + 4 * (n >> 4) + 2 * ((n >> 3) & 1) + (n & 1)) + c;
}

// Codes one 32-token group from the tiles ks, vs ([token][channel] bf16 in
// shared memory) into its record at dst.  At g = 64 the tiles are half `half`
// of a 64-token group (ks_other the other half's keys) and dst its record:
// this half's code planes go there, with the keys' (min, max) words (written
// by half 0) and this half's value (min, max) words.  Every thread of the
// 128-thread CTA takes part; the tiles may be reused once this returns.
template <int BITS, int GROUP>
__device__ __forceinline__ void code_group(QuantSmem& sm, const uint16_t* ks, const uint16_t* vs,
                                           const uint16_t* ks_other, uint8_t* dst_rec, int half_of_64 = 0) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int rb = 1024 * (BITS + 1);
  constexpr int KMETA = 128 * BITS, VCODES = KMETA + 128, VMETA = VCODES + 128 * BITS;  // in words
  // Lane beta's key channels for word t are base + 2t, base = 16 k + 8 h + half
  // with (half, k, h) = (beta >> 4, (beta >> 1) & 7, beta & 1): all four lie in
  // the 16-byte block at channel 16 k + 8 h, at halves 2t + half.
  const int half = lane >> 4, kk = (lane >> 1) & 7, hh = lane & 1;
  const int kblock = 16 * kk + 8 * hh;

  // ---- key group parameters: thread = channel ----
  {
    const int c = tid;
    float lo = bf16_to_f32(ks[c]), hi = lo;
#pragma unroll 8
    for (int n = 1; n < kGroup; ++n) {
      const float x = bf16_to_f32(ks[n * kD + c]);
      lo = fminf(lo, x);
      hi = fmaxf(hi, x);
    }
    if (GROUP == 64) {  // the group's other 32 tokens
#pragma unroll 8
      for (int n = 0; n < kGroup; ++n) {
        const float x = bf16_to_f32(ks_other[n * kD + c]);
        lo = fminf(lo, x);
        hi = fmaxf(hi, x);
      }
    }
    float z, s;
    quant_params(BITS, lo, hi, z, s);
    const float rs = quant_recip(s);
    if (BITS == 1) {
      sm.kt[0][c] = code_threshold<1>(lo, hi, z, s, rs, 1u);
    } else {  // three thresholds of the dearer 2-bit code cost more than the codes they replace
      sm.kt[0][c] = z;
      sm.kt[1][c] = s;
      sm.kt[2][c] = rs;
    }
    sm.klohi[c] = bf16_bits_canonical(lo) | (bf16_bits_canonical(hi) << 16);
  }
  __syncthreads();

  // ---- key codes: warp per token, one ballot per code word.  At 1 bit a
  // code is one comparison with the channel's threshold, found once per
  // channel for the group's tokens (a value group's 32 elements are spread
  // over 4 lanes, 8 each, and the 2-bit code needs three thresholds: there the
  // per-element quotient costs less) ----
  {
    float T[4][3];  // 1 bit: the channel's threshold; 2 bits: its z, s, 1/s
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int c = kblock + 2 * t + half;
#pragma unroll
      for (int l = 0; l < (BITS == 1 ? 1 : 3); ++l) T[t][l] = sm.kt[l][c];
    }
    for (int n = 8 * warp; n < 8 * warp + 8; ++n) {  // token n = 8 j + a
      const uint4 blk = *reinterpret_cast<const uint4*>(ks + n * kD + kblock);
      const uint32_t wv[4] = {blk.x, blk.y, blk.z, blk.w};  // halves 2t, 2t+1 in word t
      const int j = n >> 3, aa = n & 7;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float x = bf16_to_f32(half ? (wv[t] >> 16) : (wv[t] & 0xFFFFu));
        const uint32_t code = BITS == 1 ? (x >= T[t][0] ? 1u : 0u) : quant_code<BITS>(x, T[t][0], T[t][1], T[t][2]);
        const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, code & 1u);
        const int word = 4 * (4 * aa + t) + j;
        if (BITS == 2) {
          const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, code >> 1);
          if (lane == 1) sm.rec[128 + word] = b1;
        }
        if (lane == 0) sm.rec[word] = b0;
      }
    }
  }

  // ---- value parameters and codes: warp per token pair ----
  for (int p = 4 * warp; p < 4 * warp + 4; ++p) {
    const int n = 2 * p + half;  // this lane's token
    const uint4 blk = *reinterpret_cast<const uint4*>(vs + n * kD + kblock);  // channels kblock .. +7
    const uint32_t wv[4] = {blk.x, blk.y, blk.z, blk.w};
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = bf16_to_f32(wv[e] & 0xFFFFu);
      x[2 * e + 1] = bf16_to_f32(wv[e] >> 16);
    }
    float lo = x[0], hi = x[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) {
      lo = fminf(lo, x[e]);
      hi = fmaxf(hi, x[e]);
    }
    // the 32-channel group cg = kk >> 1 spans the four lanes that differ in bits
    // 0..1, the 64-channel group kk >> 2 the eight that differ in bits 0..2
#pragma unroll
    for (int off = 1; off <= (GROUP == 64 ? 4 : 2); off <<= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
      hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
    }
    float z, s;
    quant_params(BITS, lo, hi, z, s);
    const float rs = quant_recip(s);
    if (GROUP == 32 && (lane & 3) == 0)
      sm.rec[VMETA + vmeta_word(n, kk >> 1)] = bf16_bits_canonical(lo) | (bf16_bits_canonical(hi) << 16);
    if (GROUP == 64 && (lane & 7) == 0)
      sm.rec[VMETA + vmeta64_word(n, kk >> 2)] = bf16_bits_canonical(lo) | (bf16_bits_canonical(hi) << 16);
    const int t = p & 3, j = 2 * (p >> 3) + ((p >> 2) & 1);
#pragma unroll
    for (int aa = 0; aa < 8; ++aa) {  // channel kblock + aa = 16 k + 8 h + a
      const uint32_t code = quant_code<BITS>(x[aa], z, s, rs);
      const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, code & 1u);
      const int word = 4 * (4 * aa + t) + j;
      if (BITS == 2) {
        const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, code >> 1);
        if (lane == 1) sm.rec[VCODES + 128 + word] = b1;
      }
      if (lane == 0) sm.rec[VCODES + word] = b0;
    }
  }
  __syncthreads();  // every key code word of every warp is in place
  // ---- key code words into the record's order ----
  // The ballots give token-major words: word 4L + n (L = 4a + t) holds token
  // 8n + a, bit e + 16h for channel 16 (e >> 1) + 8 (e & 1) + 2t + h.  Record
  // word 4L + j takes bits e = 4j + i (i = 0..3) of the four tokens: bit
  // e + 16h of word n goes to bit (11 + n + 16h - 4i) mod 32, a left rotation
  // by (11 + n - 4j - 5i) mod 32 of the pair (e, e + 16).
  uint32_t kperm[BITS];
  {
    const int L = tid >> 2, j = tid & 3;
#pragma unroll
    for (int p = 0; p < BITS; ++p) {
      uint32_t w = 0u;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const uint32_t src = __funnelshift_r(sm.rec[128 * p + 4 * L + n], sm.rec[128 * p + 4 * L + n], 4 * j);
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // bits i, i + 16 of src are e, e + 16 of the word
          const int rot = (11 + n - 5 * i) & 31;
          w |= __funnelshift_l(src, src, rot) & __funnelshift_l(0x10001u << i, 0x10001u << i, rot);
        }
      }
      kperm[p] = w;
    }
  }
  {
    const int tt = tid >> 5, m = tid & 31;
    const int kc = 16 * (m >> 2) + 2 * tt + 8 * ((m >> 1) & 1) + (m & 1);
    sm.rec[KMETA + tid] = sm.klohi[kc];
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < BITS; ++p) sm.rec[128 * p + tid] = kperm[p];
  __syncthreads();

  // ---- the record out, coalesced ----
  uint4* dst = reinterpret_cast<uint4*>(dst_rec);
  const uint4* src = reinterpret_cast<const uint4*>(sm.rec);
  if constexpr (GROUP == 32) {
    for (int i = tid; i < rb / 16; i += 128) __stcs(dst + i, src[i]);
  } else {  // in 16-byte units: K codes of half h at 32 BITS h, K minmax at 64 BITS, V codes of half h at
            // 64 BITS + 32 + 32 BITS h, V minmax of half h at 128 BITS + 32 + 16 h
    const int h = half_of_64;
    for (int i = tid; i < 32 * BITS; i += 128) __stcs(dst + 32 * BITS * h + i, src[i]);
    if (h == 0)
      for (int i = tid; i < 32; i += 128) __stcs(dst + 64 * BITS + i, src[32 * BITS + i]);
    for (int i = tid; i < 32 * BITS; i += 128) __stcs(dst + 64 * BITS + 32 + 32 * BITS * h + i, src[32 * BITS + 32 + i]);
    for (int i = tid; i < 16; i += 128) __stcs(dst + 128 * BITS + 32 + 16 * h + i, src[64 * BITS + 32 + i]);
  }
  __syncthreads();  // the record buffer is reused by the next group
}

template <int BITS, int GROUP>
__global__ void __launch_bounds__(128) quantize_kernel(QuantArgs a) {
  extern __shared__ __align__(16) uint8_t qsmem[];
  QuantSmem& sm = *reinterpret_cast<QuantSmem*>(qsmem);
  const int tid = threadIdx.x;
  const int ng = a.nq / kGroup;
  constexpr int rb = 1024 * (BITS + 1);
  if constexpr (GROUP == 64) {
    // a 64-token group per iteration: both tile buffers, two records with the
    // group's shared parameters
    const int ng64 = a.nq / 64;
    for (int64_t gi = blockIdx.x; gi < a.total_groups; gi += gridDim.x) {
      const int64_t bh = gi / ng64;
      const int g = (int)(gi % ng64);
      for (int half = 0; half < 2; ++half) {
        const int64_t row0 = bh * a.N + (int64_t)(2 * g + half) * kGroup;
        const uint8_t* ksrc = reinterpret_cast<const uint8_t*>(a.k + row0 * kD);
        const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(a.v + row0 * kD);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          cp_async16(reinterpret_cast<uint8_t*>(sm.tile[half][0]) + 16 * (tid + 128 * r), ksrc + 16 * (tid + 128 * r));
          cp_async16(reinterpret_cast<uint8_t*>(sm.tile[half][1]) + 16 * (tid + 128 * r), vsrc + 16 * (tid + 128 * r));
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      __syncthreads();
      uint8_t* rec = a.records + (bh * a.units_cap + g) * record_bytes(BITS, 64);
      code_group<BITS, 64>(sm, sm.tile[0][0], sm.tile[0][1], sm.tile[1][0], rec, 0);
      code_group<BITS, 64>(sm, sm.tile[1][0], sm.tile[1][1], sm.tile[0][0], rec, 1);  // ends with a barrier: tiles free
    }
    return;
  }

  // g = 32: one group per iteration, loaded into tile 0 and coded
  auto load = [&](int64_t gi, int buf) {
    if (gi < a.total_groups) {
      const int64_t bh = gi / ng;
      const int g = (int)(gi % ng);
      const int64_t row0 = bh * a.N + (int64_t)g * kGroup;
      const uint8_t* ksrc = reinterpret_cast<const uint8_t*>(a.k + row0 * kD);
      const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(a.v + row0 * kD);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        cp_async16(reinterpret_cast<uint8_t*>(sm.tile[buf][0]) + 16 * (tid + 128 * r), ksrc + 16 * (tid + 128 * r));
        cp_async16(reinterpret_cast<uint8_t*>(sm.tile[buf][1]) + 16 * (tid + 128 * r), vsrc + 16 * (tid + 128 * r));
      }
    }
    cp_async_commit();
  };

  for (int64_t gi = blockIdx.x; gi < a.total_groups; gi += gridDim.x) {
    const int buf = 0;
    load(gi, buf);
    cp_async_wait<0>();
    __syncthreads();
    const int64_t bh = gi / ng;
    const int g = (int)(gi % ng);
    code_group<BITS, 32>(sm, sm.tile[buf][0], sm.tile[buf][1], nullptr, a.records + (bh * a.q_groups_cap + g) * (int64_t)rb);
  }
  cp_async_wait<0>();
}

// Residual window: rows N_q .. N-1 of K and V copied into [resid_cap][2][D].
__global__ void resid_copy_kernel(const uint16_t* k, const uint16_t* v, uint16_t* resid, int32_t Hkv,
                                  int32_t N, int32_t nq, int32_t resid_cap, int64_t total_vec) {
  const int r = N - nq;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total_vec;
       i += (int64_t)gridDim.x * blockDim.x) {
    // i enumerates (bh, row j, kv, 16-byte chunk of 16)
    const int chunk = (int)(i & 15);
    const int kv = (int)((i >> 4) & 1);
    const int64_t rest = i >> 5;
    const int j = (int)(rest % r);
    const int64_t bh = rest / r;
    const uint16_t* src = (kv == 0 ? k : v) + ((bh * N + nq + j) * kD);
    uint16_t* dst = resid + ((bh * resid_cap + j) * 2 + kv) * kD;
    reinterpret_cast<uint4*>(dst)[chunk] = __ldcs(reinterpret_cast<const uint4*>(src) + chunk);
  }
}

template <int BITS, int GROUP>
static cudaError_t launch_quantize_bits(const QuantArgs& a, cudaStream_t stream) {
  // g = 32 uses tile 0 only (see QuantSmem)
  const int smem = GROUP == 32 ? (int)offsetof(QuantSmem, tile[1]) : (int)sizeof(QuantSmem);
  static unsigned long long configured = 0ull;
  cudaError_t e = spc_host::ensure_smem_limit(configured, quantize_kernel<BITS, GROUP>, smem);
  if (e != cudaSuccess) return e;
  // One wave of resident CTAs (the kernel strides over the groups): a second,
  // partial wave would start only when the first ends.
  static int resident[64] = {};
  const int dev = spc_host::current_device();
  int per_sm = (dev >= 0 && dev < 64) ? __atomic_load_n(&resident[dev], __ATOMIC_ACQUIRE) : 0;
  if (per_sm <= 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_kernel<BITS, GROUP>, 128, smem) !=
            cudaSuccess ||
        per_sm <= 0) {
      cudaGetLastError();
      per_sm = 1;
    }
    if (dev >= 0 && dev < 64) __atomic_store_n(&resident[dev], per_sm, __ATOMIC_RELEASE);
  }
  const int64_t grid = std::min<int64_t>(a.total_groups, (int64_t)spc_host::sm_count() * per_sm);
  quantize_kernel<BITS, GROUP><<<(unsigned)grid, 128, smem, stream>>>(a);
  return cudaGetLastError();
}

spc_status launch_quantize(const spc_dims* d, const uint16_t* k, const uint16_t* v, void* records,
                           uint16_t* resid, cudaStream_t stream) {
  const int32_t nq = num_quantized(d->N, d->R, d->group);
  const int32_t r = d->N - nq;
  const int64_t BH = (int64_t)d->B * d->Hkv;
  cudaError_t e = cudaSuccess;
  if (nq > 0) {
    QuantArgs a;
    a.k = k;
    a.v = v;
    a.records = static_cast<uint8_t*>(records);
    a.Hkv = d->Hkv;
    a.N = d->N;
    a.nq = nq;
    a.q_groups_cap = d->q_groups_cap;
    a.units_cap = records_cap(d->group, d->q_groups_cap);
    a.total_groups = BH * (nq / d->group);
    if (d->group == 64)
      e = d->bits == 1 ? launch_quantize_bits<1, 64>(a, stream) : launch_quantize_bits<2, 64>(a, stream);
    else
      e = d->bits == 1 ? launch_quantize_bits<1, 32>(a, stream) : launch_quantize_bits<2, 32>(a, stream);
  }
  if (e == cudaSuccess && r > 0) {
    const int64_t total_vec = BH * r * 32;
    const int64_t grid = std::min<int64_t>((total_vec + 255) / 256, (int64_t)spc_host::sm_count() * 8);
    resid_copy_kernel<<<(unsigned)grid, 256, 0, stream>>>(k, v, resid, d->Hkv, d->N, nq, d->resid_cap,
                                                         total_vec);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

// ------------------------------------------------------------ decode-time append
// The new token's K/V joins the cache (SpeCache page, section 3 "Decoding",
// Algorithm 3) and its 16-bit row goes to the host cache (section 3's offload
// of the full-precision cache to CPU memory).  One CTA per (b, hkv): the row
// goes to window row r = N - N_q (and host row N); when N+1 tokens quantise
// one more group, the window's oldest g rows are coded into records N_q/32 ..
// by the same code_group as the prefill, and the window shifts down by g.
struct AppendArgs {
  const uint16_t* k_new;  // [B][Hkv][D]
  const uint16_t* v_new;
  uint8_t* records;
  uint16_t* resid;        // [B][Hkv][resid_cap][2][D]
  uint16_t* host;         // device address of [B][Hkv][n_cap][2][D], or null
  int64_t n_cap;
  int32_t N, nq, r, resid_cap, q_groups_cap, units_cap, flush;
};

template <int BITS, int GROUP>
__global__ void __launch_bounds__(128) append_kernel(AppendArgs a) {
  extern __shared__ __align__(16) uint8_t qsmem[];
  QuantSmem& sm = *reinterpret_cast<QuantSmem*>(qsmem);
  const int tid = threadIdx.x;
  const int64_t bh = blockIdx.x;
  uint4* win = reinterpret_cast<uint4*>(a.resid + bh * a.resid_cap * 2 * kD);  // 32 uint4 per row: K then V
  if (tid < 32) {
    const uint4 v = tid < 16 ? reinterpret_cast<const uint4*>(a.k_new + bh * kD)[tid]
                             : reinterpret_cast<const uint4*>(a.v_new + bh * kD)[tid - 16];
    win[(int64_t)a.r * 32 + tid] = v;
    if (a.host != nullptr) reinterpret_cast<uint4*>(a.host + (bh * a.n_cap + a.N) * 2 * kD)[tid] = v;
  }
  if (!a.flush) return;
  __syncthreads();  // the new row may belong to the group being flushed
  for (int i = tid; i < GROUP * 32; i += 128) {  // window rows 0..g-1 -> [token][channel] tiles of 32 rows
    const int n = i >> 5, q = i & 31, tile = n >> 5, row = n & 31;
    const uint4 v = win[n * 32 + q];
    if (q < 16) reinterpret_cast<uint4*>(sm.tile[tile][0] + row * kD)[q] = v;
    else reinterpret_cast<uint4*>(sm.tile[tile][1] + row * kD)[q - 16] = v;
  }
  __syncthreads();
  uint8_t* rec = a.records + (bh * a.units_cap + a.nq / GROUP) * record_bytes(BITS, GROUP);
  code_group<BITS, GROUP>(sm, sm.tile[0][0], sm.tile[0][1], sm.tile[1][0], rec, 0);
  if (GROUP == 64) code_group<BITS, GROUP>(sm, sm.tile[1][0], sm.tile[1][1], sm.tile[0][0], rec, 1);
  // rows g .. r move to 0 .. r-g, 32 rows at a time: a chunk's sources lie
  // past every destination written before it, and it is read in full before
  // it is written
  const int keep = a.r + 1 - GROUP;
  for (int c0 = 0; c0 < keep; c0 += kGroup) {
    const int rows = min(kGroup, keep - c0);
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = tid + 128 * u, n = i >> 5;
      if (n < rows) v[u] = win[(int64_t)(GROUP + c0 + n) * 32 + (i & 31)];
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = tid + 128 * u, n = i >> 5;
      if (n < rows) win[(int64_t)(c0 + n) * 32 + (i & 31)] = v[u];
    }
    __syncthreads();
  }
}

template <int BITS, int GROUP>
static cudaError_t launch_append_k(const AppendArgs& a, int64_t BH, cudaStream_t stream) {
  const int smem = (int)sizeof(QuantSmem);
  static unsigned long long configured = 0ull;
  cudaError_t e = spc_host::ensure_smem_limit(configured, append_kernel<BITS, GROUP>, smem);
  if (e == cudaSuccess) append_kernel<BITS, GROUP><<<(unsigned)BH, 128, smem, stream>>>(a);
  return e;
}

spc_status launch_append(const spc_dims* d, const uint16_t* k_new, const uint16_t* v_new, void* records,
                         uint16_t* resid, uint16_t* host_dev, int64_t n_cap, cudaStream_t stream) {
  AppendArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.records = static_cast<uint8_t*>(records);
  a.resid = resid;
  a.host = host_dev;
  a.n_cap = n_cap;
  a.N = d->N;
  a.nq = num_quantized(d->N, d->R, d->group);
  a.r = d->N - a.nq;
  a.resid_cap = d->resid_cap;
  a.q_groups_cap = d->q_groups_cap;
  a.units_cap = records_cap(d->group, d->q_groups_cap);
  a.flush = num_quantized(d->N + 1, d->R, d->group) > a.nq ? 1 : 0;
  const int64_t BH = (int64_t)d->B * d->Hkv;
  if (BH == 0) return SPC_OK;
  cudaError_t e;
  if (d->bits == 1)
    e = d->group == 64 ? launch_append_k<1, 64>(a, BH, stream) : launch_append_k<1, 32>(a, BH, stream);
  else
    e = d->group == 64 ? launch_append_k<2, 64>(a, BH, stream) : launch_append_k<2, 32>(a, BH, stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

}  // namespace spc
