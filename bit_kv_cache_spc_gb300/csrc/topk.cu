// ArgTopK(A_{1,:}) of the SpeCache page (Algorithm 3; Algorithm 2 for the
// pre-decoding step): per (b, hkv) the k positions of C' with the largest
// speculative-token attention probability, summed over the G query heads of
// the KV head.
//
// One thread-block cluster (up to 8 CTAs) per (b, hkv) row.  Each CTA turns
// its slice of the row into scores S(n) = sum_h 2^(log2e * (l_h(n) - lse_h))
// held in shared memory as uint32 bit patterns (S >= 0, so integer order is
// float order).  For k up to 2048 the two-level kernel further down selects
// from candidates; for larger k (topk_kernel, next) the cluster runs an
// MSB-first radix select (4 passes of
// 8 bits) for the k-th largest key, summing the CTAs' histograms through
// distributed shared memory.  The ordered compaction works one 32-position
// word at a time: a warp's ballots give the word's bitmap and the in-word
// ranks, and one block-wide scan over the words' counts (plus the lower CTAs'
// totals) gives every selected position its place in the ascending output.
// Ties at the threshold go to the lower position.
#include <cooperative_groups.h>

#include "common.cuh"
#include "select.cuh"

namespace cg = cooperative_groups;

namespace spc {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkMaxSlice = 32768;  // positions per CTA (one 32-position word per thread)

struct TopkArgs {
  const float* logits;  // [BH][G][Lcap]
  const float* lse;     // [B][2][Hq]
  int32_t* idx;         // [BH][k]
  uint32_t* bitmap;     // [BH][q_groups_cap]
  int32_t Hq, Hkv, G, nq, k, keff, Lcap, q_groups_cap;
  int32_t slice;        // positions per CTA, multiple of 32
  // Where each selected position sat in the previous selection (or null):
  // src[j] = the index of idx[j] in prev_idx [BH][prev_k] (ascending, -1
  // padded), else -1.
  const int32_t* prev_idx;
  int32_t prev_k;
  int32_t* src;         // [BH][k]
};

constexpr int kPrevSmem = 2048;  // a previous selection up to this long is searched in shared memory

struct TopkShared {
  uint32_t hist[2][256];  // this CTA's histogram, double-buffered by pass parity
  uint32_t total[256];    // cluster-wide histogram of the current pass
  uint32_t wsum[2][kTopkWarps];
  uint32_t counts[2];     // this CTA's (> threshold, == threshold) counts
  uint32_t prefix, prefix_mask, remaining;
};

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkArgs a) {
  cg::cluster_group cluster = cg::this_cluster();
  grid_dependency_sync();  // nothing is read or written before the previous kernel is done
  extern __shared__ __align__(16) uint32_t keys[];     // [slice]
  __shared__ uint32_t wgt[kTopkMaxSlice / 32];          // per word: count, then exclusive prefix
  __shared__ uint32_t weq[kTopkMaxSlice / 32];
  __shared__ TopkShared sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned rank = cluster.block_rank();
  const unsigned ncta = cluster.num_blocks();
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv);
  const int n0 = (int)rank * a.slice;
  const int len = max(0, min(a.slice, a.nq - n0));  // multiple of 32
  const int nw = len >> 5;
  constexpr float kLog2e = 1.4426950408889634f;

  // ---- scores ----
  float nlse[4];
#pragma unroll
  for (int gi = 0; gi < 4; ++gi)
    nlse[gi] = gi < a.G ? -a.lse[((int64_t)b * 2 + 1) * a.Hq + hk * a.G + gi] * kLog2e : 0.f;
  const float* lrow = a.logits + (bh * a.G) * (int64_t)a.Lcap + n0;
  for (int i = tid; i < len; i += kTopkThreads) {
    float s = 0.f;
    for (int gi = 0; gi < a.G; ++gi) s += fast_exp2(fmaf(__ldcs(lrow + (int64_t)gi * a.Lcap + i), kLog2e, nlse[gi]));
    keys[i] = __float_as_uint(s);
  }
  if (tid == 0) {
    sh.prefix = 0u;
    sh.prefix_mask = 0u;
    sh.remaining = (uint32_t)a.keff;
  }
  __syncthreads();

  // ---- radix select of the keff-th largest key ----
  if (a.keff > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      const int buf = pass & 1;
      for (int j = tid; j < 256; j += kTopkThreads) sh.hist[buf][j] = 0u;
      __syncthreads();
      const uint32_t prefix = sh.prefix, pmask = sh.prefix_mask;
      for (int i0 = 0; i0 < len; i0 += kTopkThreads) {
        const int i = i0 + tid;
        const uint32_t key = i < len ? keys[i] : 0u;
        const bool in = i < len && ((key ^ prefix) & pmask) == 0u;
        const uint32_t active = __ballot_sync(0xFFFFFFFFu, in);
        if (in) {
          const uint32_t bin = (key >> shift) & 255u;
          const uint32_t peers = __match_any_sync(active, bin);
          if ((int)(__ffs(peers) - 1) == lane) atomicAdd(&sh.hist[buf][bin], (uint32_t)__popc(peers));
        }
      }
      cluster.sync();
      for (int j = tid; j < 256; j += kTopkThreads) {
        uint32_t s = 0;
        for (unsigned r = 0; r < ncta; ++r) s += cluster.map_shared_rank(&sh.hist[buf][0], r)[j];
        sh.total[j] = s;
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 8l .. 8l+7; find the bin holding the remaining-th largest
        uint32_t cnt[8], own = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          cnt[e] = sh.total[8 * lane + e];
          own += cnt[e];
        }
        uint32_t above = own;  // inclusive suffix sum over lanes >= this one
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, above, off);
          if (lane + off < 32) above += v;
        }
        above -= own;  // keys in the bins of higher lanes
        const uint32_t rem = sh.remaining;
        if (above < rem && rem <= above + own) {
          uint32_t acc = above;
          for (int e = 7; e >= 0; --e) {
            if (acc + cnt[e] >= rem) {
              sh.prefix = prefix | ((uint32_t)(8 * lane + e) << shift);
              sh.prefix_mask = pmask | (255u << shift);
              sh.remaining = rem - acc;
              break;
            }
            acc += cnt[e];
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- ordered compaction, one 32-position word per warp step ----
  const uint32_t T = sh.prefix;
  const uint32_t need = sh.remaining;  // keys == T to take, lowest positions first
  const bool any = a.keff > 0;
  for (int w = warp; w < nw; w += kTopkWarps) {
    const uint32_t key = keys[32 * w + lane];
    const uint32_t bgt = __ballot_sync(0xFFFFFFFFu, any && key > T);
    const uint32_t beq = __ballot_sync(0xFFFFFFFFu, any && key == T);
    if (lane == 0) {
      wgt[w] = __popc(bgt);
      weq[w] = __popc(beq);
    }
  }
  __syncthreads();
  // exclusive scan of the word counts (one word per thread)
  {
    const uint32_t g = tid < nw ? wgt[tid] : 0u, e = tid < nw ? weq[tid] : 0u;
    uint32_t ig = g, ie = e;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t vg = __shfl_up_sync(0xFFFFFFFFu, ig, off), ve = __shfl_up_sync(0xFFFFFFFFu, ie, off);
      if (lane >= off) {
        ig += vg;
        ie += ve;
      }
    }
    if (lane == 31) {
      sh.wsum[0][warp] = ig;
      sh.wsum[1][warp] = ie;
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t sg = sh.wsum[0][lane], se = sh.wsum[1][lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t vg = __shfl_up_sync(0xFFFFFFFFu, sg, off), ve = __shfl_up_sync(0xFFFFFFFFu, se, off);
        if (lane >= off) {
          sg += vg;
          se += ve;
        }
      }
      sh.wsum[0][lane] = sg;  // inclusive over warps
      sh.wsum[1][lane] = se;
      if (lane == 31) {
        sh.counts[0] = sg;
        sh.counts[1] = se;
      }
    }
    __syncthreads();
    const uint32_t wg0 = warp > 0 ? sh.wsum[0][warp - 1] : 0u, we0 = warp > 0 ? sh.wsum[1][warp - 1] : 0u;
    if (tid < nw) {
      wgt[tid] = wg0 + ig - g;
      weq[tid] = we0 + ie - e;
    }
  }
  cluster.sync();
  uint32_t base_gt = 0, base_eq = 0;
  for (unsigned r = 0; r < rank; ++r) {
    const uint32_t* pc = cluster.map_shared_rank(&sh.counts[0], r);
    base_gt += pc[0];
    base_eq += pc[1];
  }

  int32_t* out = a.idx + bh * a.k;
  uint32_t* bm = a.bitmap + bh * a.q_groups_cap;
  const uint32_t below = (1u << lane) - 1u;
  for (int w = warp; w < nw; w += kTopkWarps) {
    const uint32_t key = keys[32 * w + lane];
    const bool gt = any && key > T, eq = any && key == T;
    const uint32_t bgt = __ballot_sync(0xFFFFFFFFu, gt), beq = __ballot_sync(0xFFFFFFFFu, eq);
    const uint32_t eq_before = base_eq + weq[w] + __popc(beq & below);
    const bool sel = gt || (eq && eq_before < need);
    const uint32_t pos = base_gt + wgt[w] + __popc(bgt & below) + min(eq_before, need);
    if (sel && pos < (uint32_t)a.keff) {
      out[pos] = n0 + 32 * w + lane;
      if (a.src != nullptr)
        a.src[bh * a.k + pos] = find_in_prev(a.prev_idx + bh * a.prev_k, a.prev_k, (uint32_t)(n0 + 32 * w + lane));
    }
    const uint32_t bsel = __ballot_sync(0xFFFFFFFFu, sel);
    if (lane == 0) bm[(n0 >> 5) + w] = bsel;
  }
  if (rank == 0) {
    for (int j = a.keff + tid; j < a.k; j += kTopkThreads) {
      out[j] = -1;
      if (a.src != nullptr) a.src[bh * a.k + j] = -1;
    }
    for (int w = (a.nq >> 5) + tid; w < a.q_groups_cap; w += kTopkThreads) bm[w] = 0u;
  }
  cluster.sync();  // peers may still read this CTA's counters
}

// ------------------------------------------------------------ k <= kMaxCand
// Two-level selection for the usual small k (top 1% of a few ten thousand
// positions).  Every CTA of the cluster keeps candidates of its slice, in
// ascending position, in shared memory; after one cluster barrier the leader
// CTA selects the final k_eff from the concatenated candidates (already in
// ascending position) and writes idx and the bitmap.  The candidates are
//   * when few enough: every key whose top 12 bits (the bin) are at least
//     those of the k_eff-th largest key of the row, which one histogram pass
//     per CTA and the sum of the cluster's histograms through distributed
//     shared memory find (the bin's lower bound is a threshold no selected key
//     is below);
//   * otherwise: the slice's own top-k' (k' = min(k_eff, slice length), ties
//     to the lower position) from a CTA-local radix select.  Every globally
//     selected position is among them (fewer than k_eff positions of the
//     slice precede it in the order key desc, position asc).
constexpr int kMaxCand = 2048;
constexpr int kBinShift = 19;                  // bin = key >> 19: 8 exponent and 4 mantissa bits
constexpr int kBins = 1 << (31 - kBinShift);   // keys are scores >= 0: bit 31 is clear
constexpr int kTopBytes = kBins / 32;          // values of the key's top byte
// A key's bin; a key with bit 31 set (only a NaN score could have it) counts
// in the top bin, as it counts above every other key in the selection.
__device__ __forceinline__ uint32_t key_bin(uint32_t key) { return min(key >> kBinShift, (uint32_t)kBins - 1u); }
constexpr int kSmallBin = kTopkThreads / 4;    // bins up to this size are ranked by counting

// two CTAs of 1024 threads per SM (32 registers), so a cluster per (b, hkv) row fits one wave
__global__ void __launch_bounds__(kTopkThreads, 2) topk_two_level_kernel(TopkArgs a) {
  cg::cluster_group cluster = cg::this_cluster();
  grid_dependency_sync();  // nothing is read or written before the previous kernel is done
  extern __shared__ __align__(16) uint32_t dyn[];  // keys[slice]; the leader then reuses it for the merge
  __shared__ uint32_t wgt[kTopkMaxSlice / 32];
  __shared__ uint32_t weq[kTopkMaxSlice / 32];
  __shared__ uint32_t ckey[kMaxCand], cpos[kMaxCand];  // this CTA's candidates, ascending position
  __shared__ SelShared<kTopkThreads> sh;
  __shared__ __align__(16) uint32_t hist[kBins];  // this CTA's bin counts
  __shared__ uint32_t s_count;      // candidates kept by this CTA
  __shared__ __align__(16) uint32_t htop[kTopBytes];  // this CTA's counts per top byte
  __shared__ uint32_t s_tn[2];                         // the leader's threshold and its tie count
  __shared__ uint32_t s_bin[4];     // the k_eff-th largest key's bin; keys at or above it; keys above its
                                    // top byte; keys in it
  __shared__ float s_nlse[4];       // -lse * log2(e) of the speculative row of each head of the group
  __shared__ int32_t s_prev[kPrevSmem];  // the leader's copy of the previous selection (src output)

  const int tid = threadIdx.x;
  const unsigned rank = cluster.block_rank();
  const unsigned ncta = cluster.num_blocks();
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv);
  const int n0 = (int)rank * a.slice;
  const int len = max(0, min(a.slice, a.nq - n0));  // multiple of 32
  constexpr float kLog2e = 1.4426950408889634f;
  uint32_t* keys = dyn;

  // ---- scores, four positions per thread and round, the round's loads issued up front ----
  if (tid < 4) s_nlse[tid] = tid < a.G ? -a.lse[((int64_t)b * 2 + 1) * a.Hq + hk * a.G + tid] * kLog2e : 0.f;
  // the previous selection, for the src output: copied by the leader now, read at its end
  if (a.src != nullptr && a.prev_k <= kPrevSmem && rank == 0) {
    for (int j = tid; j < a.prev_k; j += kTopkThreads) cp_async4(&s_prev[j], a.prev_idx + bh * a.prev_k + j);
    cp_async_commit();
  }
  for (int j = tid; j < kBins; j += kTopkThreads) hist[j] = 0u;
  if (tid == 0) s_count = 0u;
  __syncthreads();
  const float* lrow = a.logits + (bh * a.G) * (int64_t)a.Lcap + n0;
  for (int i = 4 * tid; i < len; i += 4 * kTopkThreads) {
    float4 v[4];
#pragma unroll
    for (int gi = 0; gi < 4; ++gi)
      v[gi] = gi < a.G ? __ldcs(reinterpret_cast<const float4*>(lrow + (int64_t)gi * a.Lcap + i))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      if (gi < a.G) {
        const float nl = s_nlse[gi];
        sc.x += fast_exp2(fmaf(v[gi].x, kLog2e, nl));
        sc.y += fast_exp2(fmaf(v[gi].y, kLog2e, nl));
        sc.z += fast_exp2(fmaf(v[gi].z, kLog2e, nl));
        sc.w += fast_exp2(fmaf(v[gi].w, kLog2e, nl));
      }
    }
    *reinterpret_cast<uint4*>(keys + i) =
        make_uint4(__float_as_uint(sc.x), __float_as_uint(sc.y), __float_as_uint(sc.z), __float_as_uint(sc.w));
    atomicAdd(&hist[key_bin(__float_as_uint(sc.x))], 1u);  // this slice's bin counts
    atomicAdd(&hist[key_bin(__float_as_uint(sc.y))], 1u);
    atomicAdd(&hist[key_bin(__float_as_uint(sc.z))], 1u);
    atomicAdd(&hist[key_bin(__float_as_uint(sc.w))], 1u);
  }
  __syncthreads();
  if (tid < kTopBytes) {  // this slice's count per top byte (32 bins each)
    const uint4* h4 = reinterpret_cast<const uint4*>(hist + 32 * tid);
    uint32_t t = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 h = h4[j];
      t += h.x + h.y + h.z + h.w;
    }
    htop[tid] = t;
  }
  cluster.sync();  // every CTA's keys, bin and top-byte counts are complete

  // ---- the bin of the k_eff-th largest key of the row (counts summed over the cluster), in warp 0:
  // first its top byte from the per-byte counts, then the bin among that byte's 32 ----
  const int lane = tid & 31, warp = tid >> 5;
  if (a.keff > 0 && warp == 0) {
    const uint32_t keff = (uint32_t)a.keff;
    uint32_t c[4] = {0u, 0u, 0u, 0u};  // lane l: top bytes 4l .. 4l+3
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (r < (int)ncta) {
        const uint4 h = reinterpret_cast<const uint4*>(cluster.map_shared_rank(htop, (unsigned)r))[lane];
        c[0] += h.x;
        c[1] += h.y;
        c[2] += h.z;
        c[3] += h.w;
      }
    }
    const uint32_t own = c[0] + c[1] + c[2] + c[3];
    uint32_t suf = own;  // inclusive suffix sum over the lanes >= this one
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, suf, off);
      if (lane + off < 32) suf += v;
    }
    uint32_t above = suf - own;  // keys with a top byte above 4l+3
    int top = -1;
    uint32_t above_top = 0u;
    if (above < keff && keff <= above + own) {
      for (int j = 3; j >= 0; --j) {
        if (above + c[j] >= keff) {
          top = 4 * lane + j;
          above_top = above;
          break;
        }
        above += c[j];
      }
    }
    const int src = __ffs(__ballot_sync(0xFFFFFFFFu, top >= 0)) - 1;
    top = __shfl_sync(0xFFFFFFFFu, top, src);
    above_top = __shfl_sync(0xFFFFFFFFu, above_top, src);
    // lane l: bin 32 top + l
    uint32_t cb = 0u;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < (int)ncta) cb += cluster.map_shared_rank(hist, (unsigned)r)[32 * top + lane];
    uint32_t sb = cb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, sb, off);
      if (lane + off < 32) sb += v;
    }
    const uint32_t ab = above_top + sb - cb;  // keys in bins above 32 top + l
    if (ab < keff && keff <= ab + cb) {
      s_bin[0] = (uint32_t)(32 * top + lane);
      s_bin[1] = ab + cb;
      s_bin[2] = above_top;
      s_bin[3] = cb;
    }
  }
  __syncthreads();

  // ---- this slice's candidates ----
  const uint32_t kloc = (uint32_t)min(a.keff, len);
  if (a.keff > 0 && s_bin[1] <= (uint32_t)kMaxCand) {  // the same decision in every CTA of the cluster
    // every key at or above the bin's lower bound; warp w compacts words
    // w*per .. w*per+per-1 in order: ballots first (kept in wgt), then the
    // warp's offset from the lower warps' counts
    const uint32_t lower = s_bin[0] << kBinShift;
    const int nw = len >> 5, per = (nw + kTopkWarps - 1) / kTopkWarps;
    const int w0 = min(nw, warp * per), w1 = min(nw, w0 + per);
    uint32_t cnt = 0u;
#pragma unroll 4
    for (int w = w0; w < w1; ++w) {
      const uint32_t bits = __ballot_sync(0xFFFFFFFFu, keys[32 * w + lane] >= lower);
      if (lane == 0) wgt[w] = bits;
      cnt += __popc(bits);
    }
    if (lane == 0) sh.wsum[0][warp] = cnt;
    __syncthreads();
    uint32_t off = lane < warp ? sh.wsum[0][lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xFFFFFFFFu, off, o);
    if (warp == kTopkWarps - 1 && lane == 0) s_count = off + cnt;
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll 4
    for (int w = w0; w < w1; ++w) {
      const uint32_t bits = wgt[w];
      if ((bits >> lane) & 1u) {
        const uint32_t r = off + __popc(bits & below);
        ckey[r] = keys[32 * w + lane];
        cpos[r] = (uint32_t)(n0 + 32 * w + lane);
      }
      off += __popc(bits);
    }
  } else if (kloc > 0) {
    uint32_t T, need;
    cta_radix_select(keys, len, kloc, sh, T, need);
    ordered_take(keys, len, T, need, wgt, weq, sh, [&](int i, uint32_t r) {
      ckey[r] = keys[i];
      cpos[r] = (uint32_t)(n0 + i);
    });
    if (tid == 0) s_count = kloc;
  }
  cluster.sync();

  // ---- merge in the leader: the candidates of every CTA, in rank (= position) order ----
  __shared__ uint32_t s_off[9];  // candidate offsets of the ranks, then the total
  const bool filtered = a.keff > 0 && s_bin[1] <= (uint32_t)kMaxCand;
  uint32_t M = 0;
  uint32_t* mkey = dyn;
  if (rank == 0) {
    if (tid < (int)ncta) wgt[tid] = *cluster.map_shared_rank(&s_count, (unsigned)tid);
    __syncthreads();
    if (tid == 0) {
      uint32_t o = 0;
      for (unsigned r = 0; r < ncta; ++r) {
        s_off[r] = o;
        o += wgt[r];
      }
      s_off[ncta] = o;
    }
    __syncthreads();
    M = s_off[ncta];
    uint32_t* mpos = dyn + M;
    for (uint32_t i = tid; i < M; i += kTopkThreads) {
      unsigned r = 0;
      while (i >= s_off[r + 1]) ++r;
      mkey[i] = cluster.map_shared_rank(ckey, r)[i - s_off[r]];
      mpos[i] = cluster.map_shared_rank(cpos, r)[i - s_off[r]];
    }
  }
  cluster.sync();  // the leader has read every CTA's candidates: the others are done
  if (a.src != nullptr && a.prev_k <= kPrevSmem && rank == 0) {
    cp_async_wait<0>();  // this thread's copies of the previous selection (issued at the start)
    __syncthreads();     // and every other thread's
  }
  if (rank == 0) {
    uint32_t* mpos = dyn + M;
    uint32_t* sbm = dyn + 2 * M;  // bitmap of the selection, one word per 32 quantised positions
    const int nwq = a.nq >> 5;
    for (int w = tid; w < nwq; w += kTopkThreads) sbm[w] = 0u;
    __syncthreads();
    int32_t* out = a.idx + bh * a.k;
    if (a.keff > 0) {
      uint32_t T, need;
      if (filtered && s_bin[3] <= (uint32_t)kSmallBin) {
        // the threshold bin's keys ranked by counting (key desc, position asc):
        // the (k_eff - keys above the bin)-th is T; need = its rank among equal keys + 1
        const uint32_t bstar = s_bin[0], r = (uint32_t)a.keff - (s_bin[1] - s_bin[3]);
        uint32_t* bk = wgt;  // the bin's keys and positions (free here)
        uint32_t* bp = weq;
        const int lane = tid & 31;
        if (tid == 0) sh.sel[0] = 0u;
        __syncthreads();
        for (uint32_t i0 = 0; i0 < M; i0 += kTopkThreads) {  // append, one atomic per warp
          const uint32_t i = i0 + tid;
          const bool in = i < M && key_bin(mkey[i]) == bstar;
          const uint32_t bal = __ballot_sync(0xFFFFFFFFu, in);
          uint32_t base = 0u;
          if (lane == 0 && bal != 0u) base = atomicAdd(&sh.sel[0], (uint32_t)__popc(bal));
          base = __shfl_sync(0xFFFFFFFFu, base, 0);
          if (in) {
            const uint32_t u = base + __popc(bal & ((1u << lane) - 1u));
            bk[u] = mkey[i];
            bp[u] = mpos[i];
          }
        }
        __syncthreads();
        // four threads per key: each counts a quarter of the bin, then the four sums
        const uint32_t nb = sh.sel[0], u = (uint32_t)tid >> 2, part = (uint32_t)tid & 3u;
        const uint32_t ku = u < nb ? bk[u] : 0u, pu = u < nb ? bp[u] : 0u;
        uint32_t gt = 0u, eq_before = 0u;
        if (u < nb) {
          for (uint32_t v = part; v < nb; v += 4u) {
            const uint32_t kv = bk[v];
            gt += kv > ku;
            eq_before += kv == ku && bp[v] < pu;
          }
        }
        gt += __shfl_xor_sync(0xFFFFFFFFu, gt, 1);
        gt += __shfl_xor_sync(0xFFFFFFFFu, gt, 2);
        eq_before += __shfl_xor_sync(0xFFFFFFFFu, eq_before, 1);
        eq_before += __shfl_xor_sync(0xFFFFFFFFu, eq_before, 2);
        if (u < nb && part == 0u && gt + eq_before == r - 1u) {
          s_tn[0] = ku;
          s_tn[1] = r - gt;  // keys equal to T that are selected
        }
        __syncthreads();
        T = s_tn[0];
        need = s_tn[1];
      } else if (filtered && (s_bin[0] >> 5) < (uint32_t)kTopBytes - 1u) {
        // the threshold's top byte is the bin's; keys above that byte are all selected
        cta_radix_select(mkey, (int)M, (uint32_t)a.keff - s_bin[2], sh, T, need, (int)(s_bin[0] >> 5));
      } else {
        cta_radix_select(mkey, (int)M, (uint32_t)a.keff, sh, T, need);
      }
      ordered_take(mkey, (int)M, T, need, wgt, weq, sh, [&](int i, uint32_t r) {
        const uint32_t p = mpos[i];
        out[r] = (int32_t)p;
        atomicOr(&sbm[p >> 5], 1u << (p & 31u));
      });
      if (a.src != nullptr) {  // the selected positions' previous slots (ordered_take ends with a barrier)
        for (int r = tid; r < a.keff; r += kTopkThreads) {
          const uint32_t p = (uint32_t)out[r];
          a.src[bh * a.k + r] = a.prev_k <= kPrevSmem ? find_in_prev(s_prev, a.prev_k, p)
                                                      : find_in_prev(a.prev_idx + bh * a.prev_k, a.prev_k, p);
        }
      }
    }
    for (int j = a.keff + tid; j < a.k; j += kTopkThreads) {
      out[j] = -1;
      if (a.src != nullptr) a.src[bh * a.k + j] = -1;
    }
    uint32_t* bm = a.bitmap + bh * a.q_groups_cap;
    for (int w = tid; w < a.q_groups_cap; w += kTopkThreads) bm[w] = w < nwq ? sbm[w] : 0u;
  }
}

spc_status launch_topk(const spc_dims* d, const float* logits, const float* lse, int32_t k, int32_t* idx,
                       uint32_t* bitmap, cudaStream_t stream, const int32_t* prev_idx, int32_t prev_k, int32_t* src) {
  TopkArgs a;
  a.logits = logits;
  a.lse = lse;
  a.idx = idx;
  a.bitmap = bitmap;
  a.prev_idx = src != nullptr ? prev_idx : nullptr;
  a.prev_k = src != nullptr ? prev_k : 0;
  a.src = src;
  a.Hq = d->Hq;
  a.Hkv = d->Hkv;
  a.G = d->Hq / d->Hkv;
  a.nq = num_quantized(d->N, d->R, d->group);
  a.k = k;
  a.keff = std::min(k, a.nq);
  a.Lcap = d->q_groups_cap * kGroup;
  a.q_groups_cap = d->q_groups_cap;
  // about 8192 positions (8 per thread) per CTA, at most 8 CTAs per cluster
  const int ncta = std::max(1, std::min(8, (a.nq + 8191) / 8192));
  a.slice = std::max(32, ((a.nq + ncta - 1) / ncta + 31) / 32 * 32);
  if (a.slice > kTopkMaxSlice) return SPC_ERR_UNSUPPORTED;
  const int64_t BH = (int64_t)d->B * d->Hkv;
  // two-level selection when every CTA's candidates fit (k <= kMaxCand) and the
  // leader's merge buffers (keys, positions, bitmap) fit in its dynamic memory
  const size_t merge_words = 2 * (size_t)ncta * std::min(a.keff, a.slice) + (size_t)(a.nq >> 5);
  const bool two_level = a.keff <= kMaxCand && merge_words <= (size_t)kTopkMaxSlice;
  const size_t smem = std::max((size_t)a.slice, two_level ? merge_words : (size_t)0) * sizeof(uint32_t);
  auto* fn = two_level ? topk_two_level_kernel : topk_kernel;
  static unsigned long long configured_radix = 0ull, configured_two = 0ull;
  cudaError_t e = spc_host::ensure_smem_limit(two_level ? configured_two : configured_radix, fn,
                                              kTopkMaxSlice * (int)sizeof(uint32_t));
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncta, (unsigned)BH, 1);
    cfg.blockDim = dim3(kTopkThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic serialisation: the launch overlaps the previous kernel's
    // tail (the kernel waits for it before touching any data)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, fn, a);
  }
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

}  // namespace spc
