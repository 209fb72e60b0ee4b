/*
 * spc.h -- C ABI of libspc, the GB300 (sm_103a) decode-time hot path of
 * SpeCache ("SpeCache: Speculative Key-Value Caching for Efficient Generation
 * of LLMs", arXiv 2503.16163).
 *
 * The library implements the per-layer primitives the page's Algorithms 1-3
 * name: Quant (section 3), Attn over [T_t, T'_{t+1}] with C' U C_kappa
 * (section 3 "Decoding", Algorithm 3), ArgTopK over the speculative token's
 * attention row (Algorithm 3; Algorithm 2 for the pre-decoding step) and
 * Pre-fetch of the selected 16-bit rows from CPU memory (Algorithm 3).
 *
 * Conventions for every call:
 *   - Pointers are device pointers unless stated otherwise; bf16 values are
 *     passed as their 16-bit patterns (uint16_t).  All tensors are dense,
 *     row-major, and 16-byte aligned.
 *   - The caller owns and allocates every buffer.  The library never
 *     allocates, frees or synchronises; each call enqueues its kernels on the
 *     given stream (NULL = the legacy default stream) and returns.
 *   - Calls are stateless and may be made from several host threads.
 *   - Argument errors return SPC_ERR_INVALID / SPC_ERR_UNSUPPORTED before
 *     anything is launched; a failed launch returns SPC_ERR_CUDA (the CUDA
 *     error is left for cudaGetLastError / spc_last_cuda_error).
 */
#ifndef SPC_H
#define SPC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPC_ABI_VERSION 2

/* A cudaStream_t. */
typedef struct CUstream_st* spc_stream;

typedef enum spc_status {
  SPC_OK = 0,
  SPC_ERR_INVALID = 1,     /* bad argument (null pointer, size, alignment) */
  SPC_ERR_UNSUPPORTED = 2, /* valid shape this build does not handle */
  SPC_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  SPC_ERR_NOT_MAPPED = 4,  /* host pointer is not device-mapped pinned memory */
  SPC_ERR_WORKSPACE = 5,   /* workspace smaller than the size query returns */
  SPC_ERR_TIMEOUT = 6      /* a bounded wait inside a kernel ran out (spc_read_device_status) */
} spc_status;

/*
 * Shape of one layer's cache.  D must be 128 and group g 32 or 64 (the page's
 * group sizes, section 4 and the appendix's LongBench runs).  G = Hq / Hkv
 * query heads share a KV head; this build handles G in {1, 2, 4}.
 * The quantised prefix has N_q = floor(max(N - R, 0) / g) * g tokens and the
 * residual window the last r = N - N_q tokens (KIVI keeps the most recent
 * tokens in 16 bits; SpeCache page, section 4).  Capacities bound the buffers:
 * N_q / 32 <= q_groups_cap and r <= resid_cap.
 */
typedef struct spc_dims {
  int32_t B, Hq, Hkv, D;
  int32_t bits;         /* 1 or 2 */
  int32_t group;        /* g: 32 or 64 */
  int32_t N;            /* visible tokens of this layer */
  int32_t R;            /* residual window target */
  int32_t q_groups_cap; /* 32-token groups the record array can hold per (b,hkv) */
  int32_t resid_cap;    /* residual rows the residual buffer can hold per (b,hkv) */
  float scale;          /* softmax scale applied to q.k, e.g. 1/sqrt(128) */
} spc_dims;

int32_t spc_abi_version(void);
const char* spc_status_string(spc_status s);
/* The cudaError_t of the last SPC_ERR_CUDA on this host thread (0 if none). */
int32_t spc_last_cuda_error(void);

/* N_q of the shape (see spc_dims).  Returns -1 for an invalid shape. */
int32_t spc_num_quantized(const spc_dims* d);

/*
 * Low-bit copy C' of one layer ("records").  Bytes spc_records_bytes(d) in
 * all, row-major [B][Hkv][records per (b, hkv)][record bytes].
 *
 * g = 32: per (b, hkv) q_groups_cap records of 1024*(bits+1) bytes; record g
 * holds tokens 32g .. 32g+31 and is, in order:
 *   K codes  : `bits` planes of 128 u32 words (plane p holds bit p of each code)
 *   K minmax : 128 u32 words, min in bits 0..15 and max in bits 16..31 (bf16)
 *   V codes  : `bits` planes of 128 u32 words
 *   V minmax : 128 u32 words
 * With L = 4a + t (a in 0..7, t in 0..3), j in 0..3 and bit b in 0..31:
 *   K code word 4L+j, bit b : with v = (b + 21) mod 32, n = v mod 4,
 *                             q = v div 4, i = (4 - q mod 4) mod 4,
 *                             h = 1 if 1 <= q <= 4 else 0, e = 4j + i:
 *                             token 8n + a, channel 16*(e>>1) + 8*(e&1) + 2t + h
 *                             (rotated left by 4i, the word holds token 8n + a's
 *                             bits for channels 16*(e>>1) + 8*(e&1) + 2t + {0, 1}
 *                             at bits 11 + n and 27 + n)
 *   K minmax word 32t+m     : channel 16*(m>>2) + 2t + 8*((m>>1)&1) + (m&1)
 *   V code word 4L+j, bit b : token 16*(j>>1) + 8*(j&1) + 2t + (b>>4),
 *                             channel 16*((b&15)>>1) + 8*(b&1) + a
 *   V minmax word 32t+m     : token 16*(m>>4) + 8*((m>>3)&1) + 2t + ((m>>2)&1),
 *                             channel group m&3
 * This is 64 (1-bit) or 96 (2-bit) bytes per token and KV head, 1/8 or 3/16
 * of bf16.
 *
 * g = 64: per (b, hkv) (q_groups_cap + 1) / 2 records of 2048*bits + 1024
 * bytes; record u holds the 64-token group of tokens 64u .. 64u+63 as two
 * halves H = 0, 1 (tokens 64u + 32H ..), each group's metadata stored once:
 *   K codes of half 0, then of half 1 (`bits` planes of 128 words each, the
 *              code word rule above for the half's 32 tokens)
 *   K minmax : 128 words, word 32t+m as above, extremes over the 64 tokens
 *   V codes of half 0, then of half 1 (as above)
 *   V minmax : 128 words; word 64H + 2m + c holds token 32H + 16*((m>>2)&1) +
 *              8*((m>>1)&1) + 2*(m>>3) + (m&1) of the record, channels
 *              64c .. 64c+63
 * This is 48 (1-bit) or 80 (2-bit) bytes per token and KV head.
 *
 * Keys are grouped per channel over g tokens, values per token over g
 * consecutive channels (KIVI's axes).  min/max are the group's exact bf16
 * extremes (-0.0 stored as +0.0); the zero point and scale are derived from
 * them (SpeCache page, section 3): 1-bit z = (3min+max)/4, s = (max-min)/2;
 * 2-bit z = min, s = (max-min)/3.
 */
size_t spc_records_bytes(const spc_dims* d);

/* Residual window: bf16 [B][Hkv][resid_cap][2][D]; row j holds the key then
 * the value of token N_q + j.  The same [.., 2, D] row format is used for the
 * full 16-bit host cache and for the staging buffer of fetched rows. */
size_t spc_resid_bytes(const spc_dims* d);

/*
 * Quant (SpeCache page, section 3; Algorithm 1, K' = Quant(K), V' = Quant(V)).
 * k, v: bf16 [B][Hkv][N][D] (device).  Writes records 0 .. N_q/g-1 of every
 * (b,hkv) and residual rows 0 .. r-1.  Codes are
 *   clamp(rint((x - z) / s), 0, 2^bits - 1), code 0 when s == 0,
 * with z, s and (x - z) / s evaluated in IEEE binary32, round to nearest even,
 * without fused multiply-add.
 */
spc_status spc_quantize_kv(const spc_dims* d, const uint16_t* k, const uint16_t* v,
                           void* records, uint16_t* resid, spc_stream stream);

/* Bytes of device workspace spc_decode_attn2 / spc_merged_attn need for this
 * shape on the current device with at most k_max fetched rows per (b, hkv):
 * control words (three per (b, hkv) and a fault word, padded to 256 bytes)
 * followed by the split-K partials (one per CTA of the attention grid and
 * query row, merged by the call's second kernel unless the CTAs combine in a
 * cluster).  The caller zero-fills a workspace once after allocating it;
 * every call leaves the control words zero again.  Calls that share a
 * workspace must not overlap on the GPU (issue them on one stream, or order
 * them with events).
 * Returns 0 for an invalid shape. */
size_t spc_attn_workspace_bytes(const spc_dims* d, int32_t k_max);

/*
 * Attn([T_t, T'_{t+1}], C') -- the two-query decode attention over the
 * low-bit copy (SpeCache page, section 3 "Decoding"; with no fetched rows this is also
 * the pre-decoding attention of Algorithm 2).
 *   q     : bf16 [B][2][Hq][D]; row 0 is the output token T_t, row 1 the
 *           speculative token T'_{t+1}.  Query head h uses KV head h / G.
 *   kv_self : bf16 [B][Hkv][2][D] (per (b, hkv) the key row, then the value
 *           row) or NULL: the speculative token's own key and value, seen by
 *           the speculative query only (it follows T_t, so T_t does not see
 *           it), as one more visible row that is not a cache position (no
 *           spec_logits entry, never selected; its probability still counts
 *           in the speculative lse).  Algorithm 3 attends over [K, K_t] with
 *           the new tokens' rows; the speculative token's row cannot join the
 *           cache, so it is passed here and dropped after the call.
 *   o     : bf16 [B][2][Hq][D], softmax(scale * q.K^T) V over all N tokens
 *           (and the speculative row's own row for q row 1), keys/values
 *           dequantised from C' for n < N_q, residual rows after.
 *   lse   : fp32 [B][2][Hq] or NULL, natural log of the softmax normaliser.
 *   spec_logits : fp32 [B][Hkv][G][q_groups_cap*32] or NULL: the speculative
 *           token's scaled logits scale*q.k at the quantised positions, the
 *           input of spc_topk_select.
 *   ws    : zero-filled-once device workspace of at least
 *           spc_attn_workspace_bytes(d, 0) bytes (see that function).
 */
spc_status spc_decode_attn2(const spc_dims* d, const void* records, const uint16_t* resid,
                            const uint16_t* q, const uint16_t* kv_self, uint16_t* o, float* lse,
                            float* spec_logits, void* ws, size_t ws_bytes, spc_stream stream);

/*
 * Attn([T_t, T'_{t+1}], C' U C_kappa) (SpeCache page, section 3 "Decoding",
 * Algorithm 3): as spc_decode_attn2, but at the k positions idx[b][hkv][0..k-1]
 * (ascending, < N_q, -1 entries ignored) both the key and the value are the
 * fetched 16-bit rows staging[b][hkv][j] (bf16 [B][Hkv][k][2][D]) instead of
 * the low-bit rows.  bitmap (u32 [B][Hkv][q_groups_cap], bit n%32 of word
 * n/32) must mark exactly the listed positions.  spec_logits at a fetched
 * position holds the logit of the fetched row.  k = 0 is spc_decode_attn2.
 * ws holds at least spc_attn_workspace_bytes(d, k) bytes.
 */
spc_status spc_merged_attn(const spc_dims* d, const void* records, const uint16_t* resid,
                           const uint16_t* q, const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap,
                           const uint16_t* staging, int32_t k, uint16_t* o, float* lse,
                           float* spec_logits, void* ws, size_t ws_bytes, spc_stream stream);

/*
 * Attn([T_t, T'_{t+1}], C' U C_kappa) of one layer together with the
 * Pre-fetch(C_kappa) of another layer (SpeCache page section 3, Algorithm 3:
 * the prefetch runs "in parallel with the following layers' computation").
 * Same as spc_merged_attn, and in the same launch the selected 16-bit rows
 * fetch_idx ([B][Hkv][fetch_k], same B and Hkv) of the pinned, mapped host
 * cache fetch_host_kv ([B][Hkv][fetch_n_cap][2][D], HOST pointer) are copied
 * to fetch_staging ([B][Hkv][fetch_k][2][D]), exactly as spc_host_gather
 * would.  The copy rides on the attention's own load pipeline, so the host
 * link works while the SMs compute; the attention's results are unchanged.
 * fetch_staging must not share a byte with the staging rows this call reads
 * (SPC_ERR_INVALID: the copy would race with the attention's reads).
 * fetch_k = 0 is spc_merged_attn.  SPC_ERR_NOT_MAPPED as spc_host_gather.
 */
spc_status spc_merged_attn_fetch(const spc_dims* d, const void* records, const uint16_t* resid,
                                 const uint16_t* q, const uint16_t* kv_self, const int32_t* idx,
                                 const uint32_t* bitmap,
                                 const uint16_t* staging, int32_t k, uint16_t* o, float* lse, float* spec_logits,
                                 void* ws, size_t ws_bytes, const uint16_t* fetch_host_kv, int64_t fetch_n_cap,
                                 const int32_t* fetch_idx, int32_t fetch_k, uint16_t* fetch_staging,
                                 spc_stream stream);

/*
 * spc_merged_attn_fetch that keeps the rows already staged (SpeCache page,
 * section 3, pre-fetching and offloading during decoding: the 16-bit rows
 * that are not in the new top-k are evicted, so the rows that are stay).
 * Row j of the new selection, fetch_idx[b][hkv][j], is copied from
 * fetch_prev_staging[b][hkv][fetch_src[b][hkv][j]] (device,
 * [B][Hkv][fetch_prev_k][2][D]) when fetch_src[b][hkv][j] >= 0, else from
 * the host cache; fetch_src is what spc_topk_select_prev writes for this
 * selection against the previous one, whose rows fetch_prev_staging holds.
 * fetch_staging is then exactly what spc_merged_attn_fetch writes, with only
 * the new rows read over the host link.  fetch_prev_staging must not share
 * a byte with fetch_staging (16-byte aligned; NULL only with fetch_prev_k = 0, when
 * every row comes from the host).  Everything else as spc_merged_attn_fetch.
 */
spc_status spc_merged_attn_fetch_prev(const spc_dims* d, const void* records, const uint16_t* resid,
                                      const uint16_t* q, const uint16_t* kv_self, const int32_t* idx,
                                      const uint32_t* bitmap, const uint16_t* staging, int32_t k, uint16_t* o,
                                      float* lse, float* spec_logits, void* ws, size_t ws_bytes,
                                      const uint16_t* fetch_host_kv, int64_t fetch_n_cap, const int32_t* fetch_idx,
                                      int32_t fetch_k, uint16_t* fetch_staging, const int32_t* fetch_src,
                                      const uint16_t* fetch_prev_staging, int32_t fetch_prev_k, spc_stream stream);

/*
 * Kernels that spc_decode_attn2 (k = 0), spc_merged_attn (k > 0) or
 * spc_merged_attn_fetch (fetch_k > 0) enqueue for this shape on the current
 * device: 1 when the CTAs of every (b, hkv) form one resident thread-block
 * cluster and combine their split-K partials through distributed shared
 * memory, else 2 (the attention grid stores its partials in the workspace and
 * a second, small kernel merges them).  A host-side query (no launch), for
 * callers that count launches or plan CUDA graphs.  -1 for an invalid shape
 * or a negative count.
 */
int32_t spc_attn_kernel_count(const spc_dims* d, int32_t k, int32_t fetch_k);

/*
 * One decoding step of a layer (SpeCache page, Algorithm 3) in one launch:
 * spc_merged_attn (optionally carrying another layer's Pre-fetch, as
 * spc_merged_attn_fetch) followed by ArgTopK(A_{1,:}), exactly as
 * spc_topk_select(d, spec_logits, lse, next_k, next_idx, next_bitmap) would
 * compute it.  The selection runs at the end of the attention: the CTA that
 * combines a (b, hkv) publishes its log-sum-exp, every CTA of the (b, hkv)
 * waits for it (bounded by a timer; on expiry it sets a fault word, reported
 * by spc_read_device_status) and keeps its chunk's candidates, and the last
 * CTA selects the final next_k.  So the speculative logits are re-read from
 * L2 by the CTAs that wrote them instead of by a second kernel.
 *   next_idx, next_bitmap: outputs as spc_topk_select's; they may be the idx
 *            and bitmap this call reads (every CTA of a (b, hkv) has read them
 *            before any is written).
 *   ws, ws_bytes: at least spc_step_workspace_bytes(d, max(k, next_k)),
 *            zero-filled once (the same contract as spc_attn_workspace_bytes).
 *   lse is required (non-NULL).
 *   spec_logits: as spc_merged_attn's, or NULL to keep the speculative
 *            logits on chip: every CTA then holds its chunk's logits in its
 *            SM's tensor memory (TMEM, 128 of the SM's 512 columns, lane =
 *            token, column = head) from the low-bit loop to its selection, so
 *            they are neither written to nor read back from device memory;
 *            only the fetched rows' logits (k x 4 floats per (b, hkv)) pass
 *            through the workspace.  The selection is identical.  NULL is
 *            accepted when spc_decode_step_on_chip returns 1 for the same
 *            arguments, else the call returns SPC_ERR_UNSUPPORTED.
 *   fetch_*: as spc_merged_attn_fetch; fetch_k = 0 for none.
 * Every CTA of the launch must be resident at once (the attention's grid is
 * one wave of the GPU): if other work holds the SMs for long enough, the
 * waits run out and the selection is wrong (SPC_ERR_TIMEOUT from
 * spc_read_device_status; zero-fill the workspace again before reuse).  When
 * the selection does not fit the attention's shared memory it is launched
 * separately, right after, on the same stream, with the same results.
 */
size_t spc_step_workspace_bytes(const spc_dims* d, int32_t k_max);
/* 1 when spc_decode_step with these arguments can keep the speculative logits
 * on chip (spec_logits == NULL): the selection rides on the attention launch
 * (k > 0) and each warp's 32-token groups need at most 32 x 4 TMEM columns.
 * 0 otherwise, -1 for an invalid shape or a negative count.  A host-side query. */
int32_t spc_decode_step_on_chip(const spc_dims* d, int32_t k, int32_t fetch_k, int32_t next_k);
/* Kernels one spc_decode_step with these arguments enqueues on the current
 * device: 1 when the selection rides on the attention launch, else the
 * attention's (spc_attn_kernel_count) plus the separate top-k.  -1 for an
 * invalid shape or a negative count. */
int32_t spc_decode_step_kernel_count(const spc_dims* d, int32_t k, int32_t fetch_k, int32_t next_k);
spc_status spc_decode_step(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                           const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap, const uint16_t* staging, int32_t k,
                           uint16_t* o, float* lse, float* spec_logits, int32_t next_k, int32_t* next_idx,
                           uint32_t* next_bitmap, void* ws, size_t ws_bytes, const uint16_t* fetch_host_kv,
                           int64_t fetch_n_cap, const int32_t* fetch_idx, int32_t fetch_k,
                           uint16_t* fetch_staging, spc_stream stream);

/*
 * spc_decode_step with the staged rows kept, as spc_merged_attn_fetch_prev
 * and spc_topk_select_prev do separately: the carried pre-fetch copies the
 * rows that fetch_src places in fetch_prev_staging ([B][Hkv][fetch_prev_k][2][D],
 * device) and reads only the others from the host, and the selection also
 * writes next_src ([B][Hkv][next_k]): each selected position's index in idx
 * (this call's own selection, k entries), else -1.  fetch_src is required when
 * fetch_k > 0; fetch_prev_staging must not share a byte with fetch_staging,
 * nor fetch_staging with staging, and next_idx none with idx here (next_src
 * is read against idx after next_idx is written): SPC_ERR_INVALID.
 * Everything else as spc_decode_step; outputs identical to it and to the
 * separate calls.
 */
spc_status spc_decode_step_prev(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                                const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap,
                                const uint16_t* staging, int32_t k, uint16_t* o, float* lse, float* spec_logits,
                                int32_t next_k, int32_t* next_idx, uint32_t* next_bitmap, int32_t* next_src,
                                void* ws, size_t ws_bytes, const uint16_t* fetch_host_kv, int64_t fetch_n_cap,
                                const int32_t* fetch_idx, int32_t fetch_k, uint16_t* fetch_staging,
                                const int32_t* fetch_src, const uint16_t* fetch_prev_staging, int32_t fetch_prev_k,
                                spc_stream stream);

/*
 * Reads and clears the fault word of an attention workspace (ws, laid out for
 * d): SPC_ERR_TIMEOUT if a bounded wait of spc_decode_step ran out since the
 * last read, else SPC_OK.  Synchronises `stream`.
 */
spc_status spc_read_device_status(void* ws, const spc_dims* d, spc_stream stream);

/*
 * spc_merged_attn without a caller-provided workspace.  The SpeCache paper has
 * no counterpart to this call; it exists for callers that cannot allocate
 * device memory (a plug-in running inside a host that owns the device
 * allocator, or a path where cudaMalloc's implicit synchronisation is not
 * allowed).  Same arguments and results as spc_merged_attn minus kv_self
 * (none) and ws/ws_bytes:
 * the workspace is a fixed 8 MiB buffer compiled into the library, which each
 * GPU that uses this call holds until the process exits.  Nothing is
 * allocated.  Argument errors return the statuses spc_merged_attn returns,
 * before anything is enqueued.  The buffer's device address is looked up
 * (cudaGetSymbolAddress) on the first call in each CUDA context and kept for
 * that context (a context made after a device reset gets a fresh lookup), so
 * make that first call before any stream capture.  Shapes whose workspace
 * (spc_attn_workspace_bytes(d, k)) exceeds 8 MiB return SPC_ERR_WORKSPACE.
 * All calls share the buffer: calls that overlap on the GPU race, so issue
 * them in order on one stream.
 */
spc_status spc_merged_attn_noalloc(const spc_dims* d, const void* records, const uint16_t* resid,
                                   const uint16_t* q, const int32_t* idx, const uint32_t* bitmap,
                                   const uint16_t* staging, int32_t k, uint16_t* o, float* lse,
                                   float* spec_logits, spc_stream stream);

/*
 * Offload(C) (SpeCache page, section 3 "Prefilling", Algorithm 1): after a
 * layer's attention the full-precision K and V (device, bf16 [B][Hkv][N][D]
 * each) are copied to the pinned host cache host_kv (HOST pointer, bf16
 * [B][Hkv][n_cap][2][D], rows interleaved K then V; pinned and mapped,
 * otherwise SPC_ERR_NOT_MAPPED; n_cap >= N), so that the device can release
 * them before the next layer.  Rows n < N are written; the copy engines do
 * the work (two strided copies per (b, hkv)), asynchronously on `stream`,
 * typically a copy stream overlapped with the next layer's compute.
 */
spc_status spc_offload_kv(const spc_dims* d, const uint16_t* k, const uint16_t* v, uint16_t* host_kv,
                          int64_t n_cap, spc_stream stream);

/*
 * Decode-time append (SpeCache page, section 3 "Decoding", Algorithm 3: the
 * new token's K/V joins the cache; section 3: the full-precision cache is
 * offloaded to CPU memory).  d describes the cache BEFORE the call: N tokens
 * held as records + resid, as spc_quantize_kv (or earlier appends) left them.
 * Afterwards the cache holds N+1 tokens and the caller advances d->N.
 *   k_new, v_new: bf16 [B][Hkv][D], token N's key and value rows (device).
 *   records, resid: the cache (device), updated in place.
 *   host_kv: HOST pointer to the pinned, mapped full-precision cache
 *            [B][Hkv][n_cap][2][D] (row N is written), or NULL for no
 *            offload; SPC_ERR_NOT_MAPPED if not mapped; n_cap > N.
 * The new row goes to window row r = N - N_q.  When N+1 tokens quantise one
 * more group (N_q' = N_q + g), the window's oldest g rows are quantised
 * into record N_q/g and the window shifts down by g rows; the result is
 * bit-identical to spc_quantize_kv over all N+1 tokens.  Needs
 * resid_cap >= N - N_q + 1 and, at a flush, q_groups_cap >= N_q'/32
 * (SPC_ERR_INVALID otherwise).  One launch on `stream`.
 */
spc_status spc_append_kv(const spc_dims* d, const uint16_t* k_new, const uint16_t* v_new, void* records,
                         uint16_t* resid, uint16_t* host_kv, int64_t n_cap, spc_stream stream);

/*
 * ArgTopK(A_{1,:}) (Algorithm 3): per (b, hkv), the k_eff = min(k, N_q)
 * quantised positions n with the largest score
 *   S(n) = sum over the G query heads h of KV head hkv of
 *          exp(spec_logits[b][hkv][h%G][n] - lse[b][1][h]),
 * i.e. the speculative token's attention probability summed over the group.
 * Ties go to the lower position.  Outputs: idx int32 [B][Hkv][k], ascending,
 * entries k_eff..k-1 set to -1; bitmap u32 [B][Hkv][q_groups_cap] with
 * exactly the selected bits set (words past N_q/32 are zeroed).
 * N_q <= 262144; spec_logits 16-byte aligned (SPC_ERR_INVALID otherwise).
 */
spc_status spc_topk_select(const spc_dims* d, const float* spec_logits, const float* lse,
                           int32_t k, int32_t* idx, uint32_t* bitmap, spc_stream stream);

/*
 * spc_topk_select that also says where each selected position sat in the
 * previous selection, so that a pre-fetch copies only the rows it does not
 * hold yet (spc_merged_attn_fetch_prev):
 *   prev_idx: int32 [B][Hkv][prev_k], the previous selection (ascending,
 *             -1 padded at the end, as spc_topk_select writes it); may be NULL
 *             when prev_k = 0.
 *   src:      int32 [B][Hkv][k] output: src[b][hkv][j] = the index i with
 *             prev_idx[b][hkv][i] == idx[b][hkv][j], else -1 (also for the
 *             -1 entries j >= k_eff).
 * idx and bitmap are exactly spc_topk_select's.  prev_idx must not share a
 * byte with idx (SPC_ERR_INVALID).
 */
spc_status spc_topk_select_prev(const spc_dims* d, const float* spec_logits, const float* lse,
                                int32_t k, int32_t* idx, uint32_t* bitmap, const int32_t* prev_idx,
                                int32_t prev_k, int32_t* src, spc_stream stream);

/*
 * Pre-fetch(C_kappa) (Algorithm 3): copies the selected 16-bit rows from the
 * full-precision cache in CPU memory into HBM,
 *   staging[b][hkv][j][t][:] = host_kv[b][hkv][idx[b][hkv][j]][t][:], t in {K, V},
 * for j < k with idx >= 0 (other staging rows are left untouched).
 *   host_kv : HOST pointer, bf16 [B][Hkv][n_cap][2][D], pinned and mapped
 *             into the device address space (cudaHostAlloc / cudaHostRegister
 *             with mapping); otherwise SPC_ERR_NOT_MAPPED.
 *   max_ctas: bound on the copy kernel's grid (0 = library default), so the
 *             copy can share the GPU with attention running on another stream.
 * Indices must be < n_cap.  The copy is issued on `stream`, typically a side
 * stream ordered after spc_topk_select by an event.
 */
spc_status spc_host_gather(const spc_dims* d, const uint16_t* host_kv, int64_t n_cap,
                           const int32_t* idx, int32_t k, uint16_t* staging, int32_t max_ctas,
                           spc_stream stream);

/*
 * spc_host_gather that keeps the rows already staged (SpeCache page, section
 * 3: the used 16-bit rows outside the new top-k are evicted, the others
 * stay): row j with src[b][hkv][j] >= 0 is copied from
 * prev_staging[b][hkv][src[b][hkv][j]] (device, [B][Hkv][prev_k][2][D]), the
 * others from the host cache.  src is what spc_topk_select_prev writes for
 * idx against the previous selection, whose rows prev_staging holds; staging
 * is then exactly spc_host_gather's.  prev_staging must not share a byte
 * with staging (SPC_ERR_INVALID; 16-byte aligned; NULL only with prev_k = 0).  Everything else as
 * spc_host_gather.
 */
spc_status spc_host_gather_prev(const spc_dims* d, const uint16_t* host_kv, int64_t n_cap,
                                const int32_t* idx, int32_t k, uint16_t* staging, const int32_t* src,
                                const uint16_t* prev_staging, int32_t prev_k, int32_t max_ctas,
                                spc_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* SPC_H */
