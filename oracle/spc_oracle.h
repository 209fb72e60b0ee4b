/*
 * spc_oracle.h -- plain CPU oracle of the SpeCache decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code: only the tests, the package's smoke() check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library; both only see the same seeded inputs.
 *
 * Source of every definition: "SpeCache: Speculative Key-Value Caching for
 * Efficient Generation of LLMs" (arXiv 2503.16163), page
 * papercache.org/.../specache-speculative-key-value-caching-..., sections 3 and 7.
 * The grouping axes (keys per channel, values per token) follow KIVI as the
 * SemKV page describes it in its section 2.1.
 *
 * Tensors are plain row-major arrays; bf16 values travel as their uint16 bit
 * patterns.  Floating point is fp64 except where a floating-point value
 * decides an integer (the quantisation code), which is taken in binary32
 * exactly as the formulas are written, without fused multiply-add.
 */
#ifndef SPC_ORACLE_H
#define SPC_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct orc_dims {
  int32_t B;      /* batch */
  int32_t Hq;     /* query heads */
  int32_t Hkv;    /* key/value heads; Hq % Hkv == 0, G = Hq / Hkv */
  int32_t D;      /* head dim, multiple of 32 */
  int32_t bits;   /* 1 or 2 */
  int32_t N;      /* visible tokens */
  int32_t R;      /* residual window: N_q = floor(max(N-R,0)/g)*g */
  int32_t group;  /* g, tokens per key group and channels per value group: 32 or 64 */
  double scale;   /* softmax scale applied to q.k */
} orc_dims;

/* Number of quantised tokens N_q and residual tokens r = N - N_q. */
int32_t orc_nq(const orc_dims* d);

/* Zero point and scale of one group from its min/max (binary32).
 * mode 0: SpeCache (1-bit: z=(3min+max)/4, s=(max-min)/2) and KIVI (2-bit:
 * z=min, s=(max-min)/3); mode 1: the original KIVI 1-bit rule z=min,
 * s=max-min, kept only as a sanity flag. */
void orc_quant_params(int32_t bits, int32_t mode, float lo, float hi, float* z, float* s);

/* Quantisation code of one value: clamp(rint((x-z)/s), 0, 2^bits-1); 0 if s==0. */
uint8_t orc_quant_code(int32_t bits, float x, float z, float s);

/* Logical quantisation of one layer (SpeCache page, section 3, "Original KIVI" and
 * "Improved 1-bit" formulas).  Inputs K, V: bf16 [B,Hkv,N,D].  Outputs:
 *   kcode u8  [B,Hkv,N_q,D]          kmm u16 [B,Hkv,N_q/32,D,2]  (min,max bf16)
 *   vcode u8  [B,Hkv,N_q,D]          vmm u16 [B,Hkv,N_q,D/32,2]
 * Keys are grouped per channel over 32 consecutive tokens, values per token
 * over 32 consecutive channels.  -0.0 is stored as +0.0 in min/max. */
void orc_quantize(const orc_dims* d, int32_t mode, const uint16_t* K, const uint16_t* V,
                  uint8_t* kcode, uint16_t* kmm, uint8_t* vcode, uint16_t* vmm);

/* Dequantised value in fp64: code*s + z with z, s from min/max in fp64. */
double orc_dequant(int32_t bits, int32_t mode, uint16_t lo, uint16_t hi, int32_t code);

/* Byte layout of the low-bit copy C' and the residual window as the library
 * stores them (the index rule is spelled out in spc_oracle.c, orc_pack).
 * records: u8 [B,Hkv,orc_units_cap(g, q_groups_cap), orc_unit_bytes(bits, g)]
 * (a record per 32-token group at g = 32, per 64-token group at g = 64);
 * resid: bf16 [B,Hkv,resid_cap,2,D]. */
int64_t orc_record_bytes(int32_t bits);
int64_t orc_unit_bytes(int32_t bits, int32_t group);
int32_t orc_units_cap(int32_t group, int32_t q_groups_cap);
void orc_pack(const orc_dims* d, const uint8_t* kcode, const uint16_t* kmm,
              const uint8_t* vcode, const uint16_t* vmm,
              const uint16_t* K, const uint16_t* V,
              int32_t q_groups_cap, int32_t resid_cap,
              uint8_t* records, uint16_t* resid);

/* Two-query attention over C' U C_kappa (SpeCache page, section 3 decoding, and
 * Algorithm 3).  q: bf16 [B,2,Hq,D] (row 0 the output token T_t, row 1 the
 * speculative token T'_{t+1}).  Position n < N_q uses the dequantised row
 * unless n is listed in idx[b,hkv,0..k-1] (then the original bf16 row of
 * K, V); positions n >= N_q are the bf16 residual rows of K, V.
 * idx may be NULL (k ignored): that is the plain low-bit attention.
 * kv_self: bf16 [B,Hkv,2,D] (key row, value row) or NULL: the speculative
 * token's own row, one more visible row for query row 1 only (Algorithm 3
 * attends over [K, K_t]; T_t precedes the speculative token).
 * Outputs (fp64): o [B,2,Hq,D], lse [B,2,Hq] (natural log of the softmax
 * normaliser of the scaled logits), S [B,Hkv,N_q]: the speculative token's
 * attention probabilities (normalised over every row it sees) summed over
 * the G query heads of the KV head.  Any output pointer may be NULL. */
void orc_attention(const orc_dims* d, int32_t mode, const uint16_t* q,
                   const uint8_t* kcode, const uint16_t* kmm,
                   const uint8_t* vcode, const uint16_t* vmm,
                   const uint16_t* K, const uint16_t* V,
                   const int32_t* idx, int32_t k, const uint16_t* kv_self,
                   double* o, double* lse, double* S);

/* ArgTopK per (b,hkv) over S[b,hkv,0..N_q-1]: the k_eff = min(k,N_q)
 * positions of largest S, ties to the lower index, listed ascending in
 * idx[b,hkv,0..k_eff-1]; idx[b,hkv,j] = -1 for k_eff <= j < k.  bitmap
 * u32 [B,Hkv,ceil(N_q/32)]: bit (n%32) of word n/32 set iff n is selected. */
void orc_topk(const orc_dims* d, const double* S, int32_t k, int32_t* idx, uint32_t* bitmap);

/* Pre-fetch copy: staging[b,h,j,t,:] = host[b,h,idx[b,h,j],t,:] for t in {K,V},
 * j < k with idx >= 0.  host: bf16 [B,Hkv,n_cap,2,D]; staging [B,Hkv,k,2,D]. */
void orc_gather(const orc_dims* d, const uint16_t* host, int64_t n_cap,
                const int32_t* idx, int32_t k, uint16_t* staging);

/* Decode-time append (SpeCache page, section 3 "Decoding", Algorithm 3: the
 * new token's K/V joins the cache; section 3's offload of the 16-bit cache to
 * CPU memory).  d describes the cache before the call (d->N tokens held as
 * records (as orc_pack lays them out for q_groups_cap) and the residual window resid
 * [B,Hkv,resid_cap,2,D], as orc_pack lays them out).  Token N's rows k_new,
 * v_new (bf16 [B,Hkv,D]) go to window row r = N - N_q; when N+1 tokens
 * quantise one more group, the window's oldest 32 rows are quantised as group
 * N_q/32 (orc_quantize on those rows), packed into its record, and dropped
 * from the window (with g = 64: the oldest 64 rows, two records).  host (bf16 [B,Hkv,n_cap,2,D], may be NULL) receives row N. */
void orc_append(const orc_dims* d, int32_t q_groups_cap, int32_t resid_cap,
                const uint16_t* k_new, const uint16_t* v_new,
                uint8_t* records, uint16_t* resid, uint16_t* host, int64_t n_cap);

#ifdef __cplusplus
}
#endif
#endif
