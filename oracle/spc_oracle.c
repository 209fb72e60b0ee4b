/*
 * spc_oracle.c -- plain, slow CPU oracle of the SpeCache decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see spc_oracle.h): used by the tests, smoke() and
 * the benchmark's CPU baseline, never by the product path.
 *
 * Every function follows the SpeCache page ("SpeCache: Speculative Key-Value
 * Caching for Efficient Generation of LLMs", arXiv 2503.16163) step by step:
 *   - quantisation: section 3, "Original KIVI quantisation" (Q(X) = round((X-z)/s),
 *     X' = Q(X)*s + z, z = min X, s = (max X - min X)/(2^B - 1)) and "Improved
 *     1-bit quantisation" (z = (3 min X + max X)/4, s = (max X - min X)/2);
 *   - grouping: keys per channel, values per token (KIVI, as the SemKV page
 *     section 2.1 describes it), group size g = 32 or 64 and a bf16 residual
 *     window (SpeCache page, section 4, software setup; the appendix's LongBench runs
 *     use g = 64);
 *   - attention: O = Attn([T_t, T'_{t+1}], C' U C_kappa) of section 3
 *     ("Decoding") and Algorithm 3, where C' U C_kappa replaces the low-bit rows
 *     C'_kappa by the 16-bit rows C_kappa;
 *   - ArgTopK over the speculative token's attention row (Algorithm 3, and
 *     Algorithm 2 for the pre-decoding step);
 *   - Pre-fetch: an index copy of 16-bit rows (Algorithm 3).
 * Readings where the pages are silent (tie rules, metadata format, GQA
 * summation, residual split) are the ones listed in the design notes and are
 * restated at each function below.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -ffp-contract=off (no contraction, so
 * binary32 steps round exactly as written).
 */
#include "spc_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* The bf16 pattern of a value that is itself a bf16 value (min/max of bf16
 * inputs), with -0.0 stored as +0.0. */
static uint16_t float_to_bf16_exact(float f) {
  if (f == 0.0f) return 0;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

int32_t orc_nq(const orc_dims* d) {
  /* Reading: the quantised part is a whole number of g-token groups and the
   * rest (at least R tokens, fewer than R + g) stays in the bf16 residual
   * window (KIVI keeps a full-precision window of recent tokens, SpeCache page,
   * section 4).  N_q = floor((N-R)/g)*g when N >= R. */
  if (d->N <= d->R) return 0;
  return ((d->N - d->R) / d->group) * d->group;
}

void orc_quant_params(int32_t bits, int32_t mode, float lo, float hi, float* z, float* s) {
  if (bits == 1 && mode == 0) {
    /* Improved 1-bit rule: z = (3 min + max)/4, s = (max - min)/2. */
    *z = (3.0f * lo + hi) * 0.25f;
    *s = (hi - lo) * 0.5f;
  } else if (bits == 1) {
    /* Original KIVI at B = 1: z = min, s = (max - min)/(2^1 - 1). */
    *z = lo;
    *s = hi - lo;
  } else {
    /* Original KIVI at B = 2: z = min, s = (max - min)/(2^2 - 1). */
    *z = lo;
    *s = (hi - lo) / 3.0f;
  }
}

uint8_t orc_quant_code(int32_t bits, float x, float z, float s) {
  /* Q(X) = round((X - z)/s).  Reading: round half to even, then clamp to the
   * code range (at 1 bit (X-z)/s spans [-0.5, 1.5]); a constant group (s = 0)
   * gets code 0, whose dequantised value z is the group's value. */
  if (s == 0.0f) return 0;
  float t = (x - z) / s;
  /* Reading: a quotient that is not a number (an infinite x - z over an
   * infinite s, possible only when the group's range overflows binary32)
   * has no nearest integer; it gets the lower end of the clamp, code 0. */
  if (isnan(t)) return 0;
  float c = rintf(t);
  float cmax = (float)((1 << bits) - 1);
  if (c < 0.0f) c = 0.0f;
  if (c > cmax) c = cmax;
  return (uint8_t)c;
}

double orc_dequant(int32_t bits, int32_t mode, uint16_t lo_b, uint16_t hi_b, int32_t code) {
  /* X' = Q(X) * s + z, evaluated in fp64 from the stored min/max. */
  double lo = (double)bf16_to_float(lo_b), hi = (double)bf16_to_float(hi_b);
  double z, s;
  if (bits == 1 && mode == 0) {
    z = (3.0 * lo + hi) / 4.0;
    s = (hi - lo) / 2.0;
  } else if (bits == 1) {
    z = lo;
    s = hi - lo;
  } else {
    z = lo;
    s = (hi - lo) / 3.0;
  }
  return (double)code * s + z;
}

void orc_quantize(const orc_dims* d, int32_t mode, const uint16_t* K, const uint16_t* V,
                  uint8_t* kcode, uint16_t* kmm, uint8_t* vcode, uint16_t* vmm) {
  const int32_t B = d->B, H = d->Hkv, N = d->N, D = d->D, nq = orc_nq(d);
  const int32_t g_sz = d->group, ng = nq / g_sz, ncg = D / g_sz;
#pragma omp parallel for collapse(2) schedule(static)
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t h = 0; h < H; ++h) {
      const uint16_t* Kbh = K + ((int64_t)(b * H + h) * N) * D;
      const uint16_t* Vbh = V + ((int64_t)(b * H + h) * N) * D;
      /* Keys: one group per (g-token block g, channel c). */
      for (int32_t g = 0; g < ng; ++g) {
        for (int32_t c = 0; c < D; ++c) {
          float lo = bf16_to_float(Kbh[(int64_t)(g_sz * g) * D + c]), hi = lo;
          for (int32_t j = 1; j < g_sz; ++j) {
            float x = bf16_to_float(Kbh[(int64_t)(g_sz * g + j) * D + c]);
            if (x < lo) lo = x;
            if (x > hi) hi = x;
          }
          float z, s;
          orc_quant_params(d->bits, mode, lo, hi, &z, &s);
          int64_t m = (((int64_t)(b * H + h) * ng + g) * D + c) * 2;
          kmm[m] = float_to_bf16_exact(lo);
          kmm[m + 1] = float_to_bf16_exact(hi);
          for (int32_t j = 0; j < g_sz; ++j) {
            int32_t n = g_sz * g + j;
            float x = bf16_to_float(Kbh[(int64_t)n * D + c]);
            kcode[((int64_t)(b * H + h) * nq + n) * D + c] = orc_quant_code(d->bits, x, z, s);
          }
        }
      }
      /* Values: one group per (token n, g-channel block cg). */
      for (int32_t n = 0; n < nq; ++n) {
        for (int32_t cg = 0; cg < ncg; ++cg) {
          float lo = bf16_to_float(Vbh[(int64_t)n * D + g_sz * cg]), hi = lo;
          for (int32_t j = 1; j < g_sz; ++j) {
            float x = bf16_to_float(Vbh[(int64_t)n * D + g_sz * cg + j]);
            if (x < lo) lo = x;
            if (x > hi) hi = x;
          }
          float z, s;
          orc_quant_params(d->bits, mode, lo, hi, &z, &s);
          int64_t m = (((int64_t)(b * H + h) * nq + n) * ncg + cg) * 2;
          vmm[m] = float_to_bf16_exact(lo);
          vmm[m + 1] = float_to_bf16_exact(hi);
          for (int32_t j = 0; j < g_sz; ++j) {
            int32_t c = g_sz * cg + j;
            float x = bf16_to_float(Vbh[(int64_t)n * D + c]);
            vcode[((int64_t)(b * H + h) * nq + n) * D + c] = orc_quant_code(d->bits, x, z, s);
          }
        }
      }
    }
  }
}

int64_t orc_record_bytes(int32_t bits) { return 1024 * (int64_t)(bits + 1); }

int64_t orc_unit_bytes(int32_t bits, int32_t group) {
  return group == 64 ? 2048 * (int64_t)bits + 1024 : orc_record_bytes(bits);
}

int32_t orc_units_cap(int32_t group, int32_t q_groups_cap) {
  return group == 64 ? (q_groups_cap + 1) / 2 : q_groups_cap;
}

/* Code planes of the 32 tokens n0 .. n0+31 of (b, hkv) bh, by the word rule
 * below: kc and vc receive `bits` planes of 128 words each. */
static void pack_code_words(const uint8_t* kcode, const uint8_t* vcode, int64_t bh, int32_t nq, int32_t D,
                            int32_t n0, int32_t bits, uint32_t* kc, uint32_t* vc) {
  for (int32_t p = 0; p < bits; ++p) {
    for (int32_t L = 0; L < 32; ++L) {
      int32_t a = L >> 2, t = L & 3;
      for (int32_t j = 0; j < 4; ++j) {
        uint32_t wk = 0, wv = 0;
        for (int32_t bit = 0; bit < 32; ++bit) {
          int32_t kv = (bit + 21) % 32, kq = kv / 4;
          int32_t ke = 4 * j + (4 - kq % 4) % 4;
          int32_t ktok = 8 * (kv % 4) + a;
          int32_t kch = 16 * (ke >> 1) + 8 * (ke & 1) + 2 * t + ((kq >= 1 && kq <= 4) ? 1 : 0);
          int32_t kcv = kcode[(bh * nq + n0 + ktok) * D + kch];
          wk |= (uint32_t)((kcv >> p) & 1) << bit;
          int32_t vtok = 16 * (j >> 1) + 8 * (j & 1) + 2 * t + (bit >> 4);
          int32_t vch = 16 * ((bit & 15) >> 1) + 8 * (bit & 1) + a;
          int32_t vcv = vcode[(bh * nq + n0 + vtok) * D + vch];
          wv |= (uint32_t)((vcv >> p) & 1) << bit;
        }
        kc[128 * p + 4 * L + j] = wk;
        vc[128 * p + 4 * L + j] = wv;
      }
    }
  }
}

/*
 * The library's byte layout of the low-bit copy (D = 128), written out as a
 * plain index rule.  With g = 32 a record holds one 32-token group and is, in
 * order:
 *   K codes  : `bits` planes of 128 u32 words (plane p holds bit p of each code)
 *   K minmax : 128 u32 words, min in bits 0..15 and max in bits 16..31 (bf16)
 *   V codes  : `bits` planes of 128 u32 words
 *   V minmax : 128 u32 words
 * With L = 4a + t (a in 0..7, t in 0..3), j in 0..3 and bit b in 0..31:
 *   K code word 4L+j, bit b : with v = (b + 21) mod 32, n = v mod 4,
 *                             q = v div 4, i = (4 - q mod 4) mod 4,
 *                             h = 1 if 1 <= q <= 4 else 0, e = 4j + i:
 *                             token 8n + a, channel 16*(e>>1) + 8*(e&1) + 2t + h
 *   K minmax word 32t+m     : channel 16*(m>>2) + 2t + 8*((m>>1)&1) + (m&1)
 *   V code word 4L+j, bit b : token 16*(j>>1) + 8*(j&1) + 2t + (b>>4),
 *                             channel 16*((b&15)>>1) + 8*(b&1) + a
 *   V minmax word 32t+m     : token 16*(m>>4) + 8*((m>>3)&1) + 2t + ((m>>2)&1),
 *                             channel group m&3
 * With g = 64 a record holds one 64-token group, its two 32-token halves
 * H = 0, 1 coded by the same word rules, and each group's (min, max) stored
 * once (48 bytes per token and KV head at 1 bit, 80 at 2 bits):
 *   K codes of half 0, K codes of half 1  (`bits` planes of 128 words each)
 *   K minmax : 128 words, word 32t+m as above, over the 64 tokens
 *   V codes of half 0, V codes of half 1
 *   V minmax : 128 words; word 64H + 2m + c: token 32H + 16*((m>>2)&1) +
 *              8*((m>>1)&1) + 2*(m>>3) + (m&1), channels 64c .. 64c+63
 * Records follow one another, q_groups_cap of them per (b,hkv) at g = 32 and
 * (q_groups_cap + 1) / 2 at g = 64.
 * The residual window is bf16 [resid_cap, 2, D] per (b,hkv): row j holds the
 * key then the value of token N_q + j.
 */
void orc_pack(const orc_dims* d, const uint8_t* kcode, const uint16_t* kmm,
              const uint8_t* vcode, const uint16_t* vmm,
              const uint16_t* K, const uint16_t* V,
              int32_t q_groups_cap, int32_t resid_cap,
              uint8_t* records, uint16_t* resid) {
  const int32_t B = d->B, H = d->Hkv, N = d->N, D = d->D, nq = orc_nq(d), bits = d->bits;
  const int32_t g_sz = d->group, r = N - nq;
  const int32_t kng = nq / g_sz, vncg = D / g_sz;  /* groups of the logical metadata */
  const int64_t UB = orc_unit_bytes(bits, g_sz);
  const int32_t ucap = orc_units_cap(g_sz, q_groups_cap), nu = nq / g_sz;
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t h = 0; h < H; ++h) {
      const int64_t bh = (int64_t)b * H + h;
      for (int32_t u = 0; u < nu; ++u) {
        uint32_t* rec = (uint32_t*)(records + (bh * ucap + u) * UB);
        memset(rec, 0, (size_t)UB);
        if (g_sz == 32) {
          uint32_t* kc = rec;
          uint32_t* kmw = rec + 128 * bits;
          uint32_t* vc = kmw + 128;
          uint32_t* vmw = vc + 128 * bits;
          pack_code_words(kcode, vcode, bh, nq, D, 32 * u, bits, kc, vc);
          for (int32_t t = 0; t < 4; ++t) {
            for (int32_t m = 0; m < 32; ++m) {
              int32_t vtok = 16 * (m >> 4) + 8 * ((m >> 3) & 1) + 2 * t + ((m >> 2) & 1);
              int64_t vm = ((bh * nq + 32 * u + vtok) * vncg + (m & 3)) * 2;
              vmw[32 * t + m] = (uint32_t)vmm[vm] | ((uint32_t)vmm[vm + 1] << 16);
            }
          }
          for (int32_t t = 0; t < 4; ++t) {
            for (int32_t m = 0; m < 32; ++m) {
              int32_t kch = 16 * (m >> 2) + 2 * t + 8 * ((m >> 1) & 1) + (m & 1);
              int64_t km = ((bh * kng + u) * D + kch) * 2;
              kmw[32 * t + m] = (uint32_t)kmm[km] | ((uint32_t)kmm[km + 1] << 16);
            }
          }
        } else {
          uint32_t* kmw = rec + 256 * bits;
          uint32_t* vmw = kmw + 128 + 256 * bits;
          for (int32_t hf = 0; hf < 2; ++hf) {
            pack_code_words(kcode, vcode, bh, nq, D, 64 * u + 32 * hf, bits, rec + 128 * bits * hf,
                            kmw + 128 + 128 * bits * hf);
            for (int32_t m = 0; m < 32; ++m) {
              int32_t vtok = 16 * ((m >> 2) & 1) + 8 * ((m >> 1) & 1) + 2 * (m >> 3) + (m & 1);
              for (int32_t c = 0; c < 2; ++c) {
                int64_t vm = ((bh * nq + 64 * u + 32 * hf + vtok) * vncg + c) * 2;
                vmw[64 * hf + 2 * m + c] = (uint32_t)vmm[vm] | ((uint32_t)vmm[vm + 1] << 16);
              }
            }
          }
          for (int32_t t = 0; t < 4; ++t) {
            for (int32_t m = 0; m < 32; ++m) {
              int32_t kch = 16 * (m >> 2) + 2 * t + 8 * ((m >> 1) & 1) + (m & 1);
              int64_t km = ((bh * kng + u) * D + kch) * 2;
              kmw[32 * t + m] = (uint32_t)kmm[km] | ((uint32_t)kmm[km + 1] << 16);
            }
          }
        }
      }
      for (int32_t j = 0; j < r; ++j) {
        const int64_t src = (bh * N + nq + j) * D;
        uint16_t* dst = resid + ((bh * resid_cap + j) * 2) * D;
        memcpy(dst, K + src, sizeof(uint16_t) * (size_t)D);
        memcpy(dst + D, V + src, sizeof(uint16_t) * (size_t)D);
      }
    }
  }
}

void orc_attention(const orc_dims* d, int32_t mode, const uint16_t* q,
                   const uint8_t* kcode, const uint16_t* kmm,
                   const uint8_t* vcode, const uint16_t* vmm,
                   const uint16_t* K, const uint16_t* V,
                   const int32_t* idx, int32_t k, const uint16_t* kv_self,
                   double* o, double* lse, double* S) {
  const int32_t B = d->B, H = d->Hkv, Hq = d->Hq, N = d->N, D = d->D, nq = orc_nq(d);
  const int32_t G = Hq / H, g_sz = d->group, ng = nq / g_sz, ncg = D / g_sz;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t hk = 0; hk < H; ++hk) {
      const int64_t bh = (int64_t)b * H + hk;
      /* Rows of K and V as this step sees them: C' U C_kappa plus the residual. */
      double* kr = (double*)malloc(sizeof(double) * (size_t)N * D);
      double* vr = (double*)malloc(sizeof(double) * (size_t)N * D);
      char* sel = (char*)calloc((size_t)(nq > 0 ? nq : 1), 1);
      if (idx != NULL) {
        for (int32_t j = 0; j < k; ++j) {
          int32_t n = idx[bh * k + j];
          if (n >= 0 && n < nq) sel[n] = 1;
        }
      }
      for (int32_t n = 0; n < N; ++n) {
        for (int32_t c = 0; c < D; ++c) {
          if (n < nq && !sel[n]) {
            int64_t km = ((bh * ng + n / g_sz) * D + c) * 2;
            int64_t vm = ((bh * nq + n) * ncg + c / g_sz) * 2;
            kr[(int64_t)n * D + c] = orc_dequant(d->bits, mode, kmm[km], kmm[km + 1],
                                                 kcode[(bh * nq + n) * D + c]);
            vr[(int64_t)n * D + c] = orc_dequant(d->bits, mode, vmm[vm], vmm[vm + 1],
                                                 vcode[(bh * nq + n) * D + c]);
          } else {
            kr[(int64_t)n * D + c] = (double)bf16_to_float(K[(bh * N + n) * D + c]);
            vr[(int64_t)n * D + c] = (double)bf16_to_float(V[(bh * N + n) * D + c]);
          }
        }
      }
      double* logit = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
      if (S != NULL)
        for (int32_t n = 0; n < nq; ++n) S[bh * nq + n] = 0.0;
      for (int32_t gi = 0; gi < G; ++gi) {
        const int32_t h = hk * G + gi;
        for (int32_t i = 0; i < 2; ++i) {
          const uint16_t* qv = q + (((int64_t)b * 2 + i) * Hq + h) * D;
          /* The speculative token (i = 1) also sees its own key and value
           * when they are given: Algorithm 3 attends over [K, K_t], and the
           * speculative token comes after T_t, so T_t does not see its row. */
          const uint16_t* self = (kv_self != NULL && i == 1) ? kv_self + bh * 2 * D : NULL;
          double mx = -INFINITY, lself = -INFINITY;
          for (int32_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int32_t c = 0; c < D; ++c)
              acc += (double)bf16_to_float(qv[c]) * kr[(int64_t)n * D + c];
            logit[n] = d->scale * acc;
            if (logit[n] > mx) mx = logit[n];
          }
          if (self != NULL) {
            double acc = 0.0;
            for (int32_t c = 0; c < D; ++c) acc += (double)bf16_to_float(qv[c]) * (double)bf16_to_float(self[c]);
            lself = d->scale * acc;
            if (lself > mx) mx = lself;
          }
          double den = 0.0;
          for (int32_t n = 0; n < N; ++n) den += exp(logit[n] - mx);
          if (self != NULL) den += exp(lself - mx);
          double* ov = o ? o + (((int64_t)b * 2 + i) * Hq + h) * D : NULL;
          if (ov != NULL) {
            for (int32_t c = 0; c < D; ++c) ov[c] = 0.0;
            for (int32_t n = 0; n < N; ++n) {
              double p = exp(logit[n] - mx) / den;
              for (int32_t c = 0; c < D; ++c) ov[c] += p * vr[(int64_t)n * D + c];
            }
            if (self != NULL) {
              double p = exp(lself - mx) / den;
              for (int32_t c = 0; c < D; ++c) ov[c] += p * (double)bf16_to_float(self[D + c]);
            }
          }
          if (lse != NULL)
            lse[((int64_t)b * 2 + i) * Hq + h] = (N > 0 || self != NULL) ? mx + log(den) : -INFINITY;
          /* Reading: the score of position n for ArgTopK is the speculative
           * token's probability summed over the query heads sharing KV head hk. */
          if (S != NULL && i == 1)
            for (int32_t n = 0; n < nq; ++n) S[bh * nq + n] += exp(logit[n] - mx) / den;
        }
      }
      free(logit);
      free(sel);
      free(kr);
      free(vr);
    }
  }
}

typedef struct {
  double s;
  int32_t n;
} scored_pos;

static int by_score_then_index(const void* a, const void* b) {
  const scored_pos* x = (const scored_pos*)a;
  const scored_pos* y = (const scored_pos*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->n < y->n) ? -1 : (x->n > y->n);
}

static int by_int(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x < y) ? -1 : (x > y);
}

void orc_topk(const orc_dims* d, const double* S, int32_t k, int32_t* idx, uint32_t* bitmap) {
  const int32_t B = d->B, H = d->Hkv, nq = orc_nq(d);
  const int32_t nw = (nq + 31) / 32;
  const int32_t keff = k < nq ? k : nq;
#pragma omp parallel for collapse(2) schedule(static)
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t h = 0; h < H; ++h) {
      const int64_t bh = (int64_t)b * H + h;
      scored_pos* all = (scored_pos*)malloc(sizeof(scored_pos) * (size_t)(nq > 0 ? nq : 1));
      for (int32_t n = 0; n < nq; ++n) {
        all[n].s = S[bh * nq + n];
        all[n].n = n;
      }
      qsort(all, (size_t)nq, sizeof(scored_pos), by_score_then_index);
      int32_t* out = idx + bh * k;
      for (int32_t j = 0; j < keff; ++j) out[j] = all[j].n;
      qsort(out, (size_t)keff, sizeof(int32_t), by_int);
      for (int32_t j = keff; j < k; ++j) out[j] = -1;
      if (bitmap != NULL) {
        uint32_t* bm = bitmap + bh * nw;
        for (int32_t w = 0; w < nw; ++w) bm[w] = 0;
        for (int32_t j = 0; j < keff; ++j) bm[out[j] / 32] |= 1u << (out[j] % 32);
      }
      free(all);
    }
  }
}

void orc_gather(const orc_dims* d, const uint16_t* host, int64_t n_cap,
                const int32_t* idx, int32_t k, uint16_t* staging) {
  const int32_t B = d->B, H = d->Hkv, D = d->D;
  for (int32_t b = 0; b < B; ++b)
    for (int32_t h = 0; h < H; ++h) {
      const int64_t bh = (int64_t)b * H + h;
      for (int32_t j = 0; j < k; ++j) {
        int32_t n = idx[bh * k + j];
        if (n < 0) continue;
        memcpy(staging + (bh * k + j) * 2 * D, host + (bh * n_cap + n) * 2 * D,
               sizeof(uint16_t) * 2 * (size_t)D);
      }
    }
}

void orc_append(const orc_dims* d, int32_t q_groups_cap, int32_t resid_cap,
                const uint16_t* k_new, const uint16_t* v_new,
                uint8_t* records, uint16_t* resid, uint16_t* host, int64_t n_cap) {
  const int32_t B = d->B, H = d->Hkv, D = d->D, N = d->N, nq = orc_nq(d), r = N - nq, g_sz = d->group;
  orc_dims next = *d;
  next.N = N + 1;
  const int flush = orc_nq(&next) > nq;
  /* one g-token group of one (b, hkv), quantised and packed on its own */
  orc_dims one = *d;
  one.B = 1;
  one.Hkv = 1;
  one.N = g_sz;
  one.R = 0;
  const int64_t UB = orc_unit_bytes(d->bits, g_sz);
  const int32_t ucap = orc_units_cap(g_sz, q_groups_cap);
  uint16_t* Kg = malloc(sizeof(uint16_t) * (size_t)g_sz * D);
  uint16_t* Vg = malloc(sizeof(uint16_t) * (size_t)g_sz * D);
  uint8_t* kcode = malloc((size_t)g_sz * D);
  uint8_t* vcode = malloc((size_t)g_sz * D);
  uint16_t* kmm = malloc(sizeof(uint16_t) * 2 * (size_t)D);
  uint16_t* vmm = malloc(sizeof(uint16_t) * 2 * (size_t)g_sz * (size_t)(D / g_sz));
  for (int32_t b = 0; b < B; ++b)
    for (int32_t h = 0; h < H; ++h) {
      const int64_t bh = (int64_t)b * H + h;
      uint16_t* win = resid + bh * resid_cap * 2 * D; /* row j: K at win + 2Dj, V at + D */
      memcpy(win + (int64_t)r * 2 * D, k_new + bh * D, sizeof(uint16_t) * (size_t)D);
      memcpy(win + (int64_t)r * 2 * D + D, v_new + bh * D, sizeof(uint16_t) * (size_t)D);
      if (host != NULL) {
        memcpy(host + (bh * n_cap + N) * 2 * D, k_new + bh * D, sizeof(uint16_t) * (size_t)D);
        memcpy(host + (bh * n_cap + N) * 2 * D + D, v_new + bh * D, sizeof(uint16_t) * (size_t)D);
      }
      if (!flush) continue;
      for (int32_t j = 0; j < g_sz; ++j) {
        memcpy(Kg + (int64_t)j * D, win + (int64_t)j * 2 * D, sizeof(uint16_t) * (size_t)D);
        memcpy(Vg + (int64_t)j * D, win + (int64_t)j * 2 * D + D, sizeof(uint16_t) * (size_t)D);
      }
      orc_quantize(&one, 0, Kg, Vg, kcode, kmm, vcode, vmm);
      orc_pack(&one, kcode, kmm, vcode, vmm, Kg, Vg, g_sz / 32, 0,
               records + (bh * ucap + nq / g_sz) * UB, NULL);
      memmove(win, win + (int64_t)g_sz * 2 * D, sizeof(uint16_t) * 2 * (size_t)D * (size_t)(r + 1 - g_sz));
    }
  free(Kg);
  free(Vg);
  free(kcode);
  free(vcode);
  free(kmm);
  free(vmm);
}
