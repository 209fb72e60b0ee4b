// Quant: the KIVI-style low-bit copy C' with SpeCache's 1-bit zero point and
// scale (SpeCache page, section 3, "Original KIVI quantisation" and "Improved
// 1-bit quantisation"; keys per channel, values per token, groups of 32).
//
// One CTA of 128 threads quantises one 32-token group of one (b, hkv) at a
// time: 8 KB of keys and 8 KB of values in, one 2 KB (1-bit) or 3 KB (2-bit)
// record out.  The kernel streams HBM: 512 B read and 64/96 B written per
// token and KV head.
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

// clamp(rint(fl((x - z) / s)), 0, cmax), 0 when s == 0.  The product with the
// correctly rounded reciprocal rs is within 1e-6 of the IEEE quotient for the
// quotients that occur (|q| <= 3), so it decides every value whose fractional
// part is farther than 1e-5 from one half; the IEEE division settles the rest.
__device__ __forceinline__ uint32_t quant_code(float x, float z, float s, float rs, float cmax) {
  if (s == 0.0f) return 0u;
  const float d = __fsub_rn(x, z);
  float t = __fmul_rn(d, rs);
  const float fr = __fsub_rn(t, floorf(t));
  if (fabsf(__fsub_rn(fr, 0.5f)) < 1e-5f) t = __fdiv_rn(d, s);
  return (uint32_t)fminf(fmaxf(rintf(t), 0.0f), cmax);
}

// min/max of bf16 values carried as floats; -0.0 is stored as +0.0.
__device__ __forceinline__ uint32_t bf16_bits_canonical(float f) {
  return f == 0.0f ? 0u : (__float_as_uint(f) >> 16);
}

struct QuantArgs {
  const uint16_t* k;
  const uint16_t* v;
  uint8_t* records;
  int32_t Hkv, N, nq, bits, q_groups_cap;
  int64_t total_groups;  // B * Hkv * (nq / 32)
};

__global__ void __launch_bounds__(128) quantize_kernel(QuantArgs a) {
  __shared__ __align__(16) uint16_t ks[kGroup * kD];
  __shared__ uint32_t kmask[2][kD];          // [plane][channel]: bit n = token n
  __shared__ uint32_t klohi[kD];             // [channel]: min | max << 16
  __shared__ uint32_t vmask[2][kGroup][4];   // [plane][token][cg]: bit j = channel 32cg+j
  __shared__ uint32_t vlohi[kGroup][4];      // [token][cg]

  const int tid = threadIdx.x;
  const int ng = a.nq / kGroup;
  const int bits = a.bits;
  const float cmax = (float)((1 << bits) - 1);
  const int64_t rb = record_bytes(bits);

  for (int64_t gi = blockIdx.x; gi < a.total_groups; gi += gridDim.x) {
    const int64_t bh = gi / ng;
    const int g = (int)(gi % ng);
    const int64_t row0 = bh * a.N + (int64_t)g * kGroup;  // first token of the group
    const uint4* ksrc = reinterpret_cast<const uint4*>(a.k + row0 * kD);
    const uint4* vsrc = reinterpret_cast<const uint4*>(a.v + row0 * kD);

    // ---- load: keys to shared memory, values kept in registers ----
    uint4 vreg[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      reinterpret_cast<uint4*>(ks)[tid + 128 * r] = __ldcs(ksrc + tid + 128 * r);
      vreg[r] = __ldcs(vsrc + tid + 128 * r);
    }

    // ---- values: group = (token, 32 channels) = 4 consecutive threads ----
    // thread tid holds, for r = 0..3, token (tid>>4) + 8r, channels
    // 32*cg + 8*sub .. +7 with cg = (tid&15)>>2, sub = tid&3.
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t w[4] = {vreg[r].x, vreg[r].y, vreg[r].z, vreg[r].w};
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = bf16_to_f32(w[e] & 0xFFFFu);
        x[2 * e + 1] = bf16_to_f32(w[e] >> 16);
      }
      float lo = x[0], hi = x[0];
#pragma unroll
      for (int e = 1; e < 8; ++e) {
        lo = fminf(lo, x[e]);
        hi = fmaxf(hi, x[e]);
      }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
        hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
      }
      float z, s;
      quant_params(bits, lo, hi, z, s);
      const float rs = (s != 0.0f) ? __frcp_rn(s) : 0.0f;
      uint32_t m0 = 0, m1 = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t c = quant_code(x[e], z, s, rs, cmax);
        m0 |= (c & 1u) << e;
        m1 |= ((c >> 1) & 1u) << e;
      }
      const int n = (tid >> 4) + 8 * r, cg = (tid & 15) >> 2, sub = tid & 3;
      reinterpret_cast<uint8_t*>(&vmask[0][n][cg])[sub] = (uint8_t)m0;
      reinterpret_cast<uint8_t*>(&vmask[1][n][cg])[sub] = (uint8_t)m1;
      if (sub == 0) vlohi[n][cg] = bf16_bits_canonical(lo) | (bf16_bits_canonical(hi) << 16);
    }
    __syncthreads();

    // ---- keys: group = (32 tokens, channel), thread tid = channel ----
    {
      const int c = tid;
      float lo = bf16_to_f32(ks[c]), hi = lo;
#pragma unroll 8
      for (int n = 1; n < kGroup; ++n) {
        const float x = bf16_to_f32(ks[n * kD + c]);
        lo = fminf(lo, x);
        hi = fmaxf(hi, x);
      }
      float z, s;
      quant_params(bits, lo, hi, z, s);
      const float rs = (s != 0.0f) ? __frcp_rn(s) : 0.0f;
      uint32_t m0 = 0, m1 = 0;
#pragma unroll 8
      for (int n = 0; n < kGroup; ++n) {
        const uint32_t code = quant_code(bf16_to_f32(ks[n * kD + c]), z, s, rs, cmax);
        m0 |= (code & 1u) << n;
        m1 |= ((code >> 1) & 1u) << n;
      }
      kmask[0][c] = m0;
      kmask[1][c] = m1;
      klohi[c] = bf16_bits_canonical(lo) | (bf16_bits_canonical(hi) << 16);
    }
    __syncthreads();

    // ---- scatter into the record layout (spc.h), thread tid = word tid ----
    uint32_t* rec = reinterpret_cast<uint32_t*>(a.records + (bh * a.q_groups_cap + g) * rb);
    const int w = tid, L = w >> 2, j = w & 3, aa = L >> 2, t = L & 3;
    for (int p = 0; p < bits; ++p) {
      uint32_t kw = 0, vw = 0;
      const int kn = 8 * j + aa;
#pragma unroll
      for (int b = 0; b < 32; ++b) {
        const int kc = 16 * ((b & 15) >> 1) + 2 * t + 8 * (b & 1) + (b >> 4);
        kw |= ((kmask[p][kc] >> kn) & 1u) << b;
        const int vn = 16 * (j >> 1) + 8 * (j & 1) + 2 * t + (b >> 4);
        const int vc = 16 * ((b & 15) >> 1) + 8 * (b & 1) + aa;
        vw |= ((vmask[p][vn][vc >> 5] >> (vc & 31)) & 1u) << b;
      }
      __stcs(rec + 128 * p + w, kw);
      __stcs(rec + 128 * (bits + 1) + 128 * p + w, vw);
    }
    {
      const int tt = w >> 5, m = w & 31;
      const int kc = 16 * (m >> 2) + 2 * tt + 8 * ((m >> 1) & 1) + (m & 1);
      __stcs(rec + 128 * bits + w, klohi[kc]);
      const int vn = 16 * (m >> 4) + 8 * ((m >> 3) & 1) + 2 * tt + ((m >> 2) & 1);
      __stcs(rec + 128 * (2 * bits + 1) + w, vlohi[vn][m & 3]);
    }
    __syncthreads();
  }
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

spc_status launch_quantize(const spc_dims* d, const uint16_t* k, const uint16_t* v, void* records,
                           uint16_t* resid, cudaStream_t stream) {
  const int32_t nq = num_quantized(d->N, d->R);
  const int32_t r = d->N - nq;
  const int64_t BH = (int64_t)d->B * d->Hkv;
  if (nq > 0) {
    QuantArgs a;
    a.k = k;
    a.v = v;
    a.records = static_cast<uint8_t*>(records);
    a.Hkv = d->Hkv;
    a.N = d->N;
    a.nq = nq;
    a.bits = d->bits;
    a.q_groups_cap = d->q_groups_cap;
    a.total_groups = BH * (nq / kGroup);
    const int64_t grid = std::min<int64_t>(a.total_groups, (int64_t)spc_host::sm_count() * 12);
    quantize_kernel<<<(unsigned)grid, 128, 0, stream>>>(a);
  }
  if (r > 0) {
    const int64_t total_vec = BH * r * 32;
    const int64_t grid = std::min<int64_t>((total_vec + 255) / 256, (int64_t)spc_host::sm_count() * 8);
    resid_copy_kernel<<<(unsigned)grid, 256, 0, stream>>>(k, v, resid, d->Hkv, d->N, nq, d->resid_cap,
                                                         total_vec);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

}  // namespace spc
