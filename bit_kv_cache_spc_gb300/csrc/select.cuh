// Exact CTA-wide selection of the k largest uint32 keys (scores >= 0 held as
// their float bit patterns, so integer order is float order), with ties going
// to the lower index.  Shared by the top-k kernel (1024 threads) and the
// selection that ends the fused decode attention (128 threads).
#pragma once

#include "common.cuh"

namespace spc {

// Index of position p in the ascending row prev[0..n), whose -1 padding at
// the end counts as larger than every position (unsigned order), or -1.
// prev is in global or shared memory.
template <typename T>
__device__ __forceinline__ int32_t find_in_prev(const T* prev, int n, uint32_t p) {
  int lo = 0, hi = n;  // the first entry >= p
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((uint32_t)prev[mid] < p)
      lo = mid + 1;
    else
      hi = mid;
  }
  return (lo < n && (uint32_t)prev[lo] == p) ? lo : -1;
}

template <int THREADS>
struct __align__(16) SelShared {
  uint32_t hist[4][256];  // four sub-histograms (warp & 3) to spread atomic contention
  uint32_t wsum[2][THREADS / 32];
  uint32_t sel[2];        // digit search result: prefix, remaining
};

// The kth largest (1 <= kth <= n) of keys[0..n): T, and how many keys equal
// to T belong to the top kth (the other kth - need are > T).  MSB-first radix
// select, 4 passes of 8 bits.  A caller that knows T's top byte (top8 >= 0)
// and that kth counts from the largest key with that top byte (none of keys
// with a larger top byte is among keys) skips the first pass.
template <int THREADS>
__device__ __forceinline__ void cta_radix_select(const uint32_t* keys, int n, uint32_t kth, SelShared<THREADS>& sh,
                                                 uint32_t& T, uint32_t& need, int top8 = -1) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0u, pmask = 0u, rem = kth;
  int pass0 = 0;
  if (top8 >= 0) {
    prefix = (uint32_t)top8 << 24;
    pmask = 0xFF000000u;
    pass0 = 1;
  }
  for (int pass = pass0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int j = tid; j < 4 * 256; j += THREADS) (&sh.hist[0][0])[j] = 0u;
    __syncthreads();
    uint32_t* h = sh.hist[warp & 3];
    for (int i = tid; i < n; i += THREADS) {
      const uint32_t key = keys[i];
      if (((key ^ prefix) & pmask) == 0u) atomicAdd(&h[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 8l .. 8l+7; find the bin holding the rem-th largest
      uint32_t cnt[8], own = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int bin = 8 * lane + e;
        cnt[e] = sh.hist[0][bin] + sh.hist[1][bin] + sh.hist[2][bin] + sh.hist[3][bin];
        own += cnt[e];
      }
      uint32_t above = own;  // inclusive suffix sum over lanes >= this one
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, above, off);
        if (lane + off < 32) above += v;
      }
      above -= own;
      if (above < rem && rem <= above + own) {
        uint32_t acc = above;
        for (int e = 7; e >= 0; --e) {
          if (acc + cnt[e] >= rem) {
            sh.sel[0] = prefix | ((uint32_t)(8 * lane + e) << shift);
            sh.sel[1] = rem - acc;
            break;
          }
          acc += cnt[e];
        }
      }
    }
    __syncthreads();
    prefix = sh.sel[0];
    rem = sh.sel[1];
    pmask |= 255u << shift;
  }
  T = prefix;
  need = rem;
}

// Ordered take over keys[0..n): element i is taken if keys[i] > T, or
// keys[i] == T and fewer than `need` elements equal to T precede it;
// emit(i, rank) is called for each taken element with its rank among the
// taken ones (ranks follow i).  wgt, weq: one word each per 32 elements.
template <int THREADS, typename Emit>
__device__ __forceinline__ void ordered_take(const uint32_t* keys, int n, uint32_t T, uint32_t need,
                                             uint32_t* wgt, uint32_t* weq, SelShared<THREADS>& sh, Emit&& emit) {
  constexpr int kWarpsT = THREADS / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = (n + 31) >> 5;
  for (int w = warp; w < nw; w += kWarpsT) {
    const int i = 32 * w + lane;
    const uint32_t key = i < n ? keys[i] : 0u;
    const uint32_t bgt = __ballot_sync(0xFFFFFFFFu, i < n && key > T);
    const uint32_t beq = __ballot_sync(0xFFFFFFFFu, i < n && key == T);
    if (lane == 0) {
      wgt[w] = __popc(bgt);
      weq[w] = __popc(beq);
    }
  }
  __syncthreads();
  {  // exclusive scan of the word counts: thread t owns words t*per .. t*per+per-1
    const int per = (nw + THREADS - 1) / THREADS;
    const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
    uint32_t g = 0u, e = 0u;
    for (int w = w0; w < w1; ++w) {
      g += wgt[w];
      e += weq[w];
    }
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
      uint32_t sg = lane < kWarpsT ? sh.wsum[0][lane] : 0u, se = lane < kWarpsT ? sh.wsum[1][lane] : 0u;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t vg = __shfl_up_sync(0xFFFFFFFFu, sg, off), ve = __shfl_up_sync(0xFFFFFFFFu, se, off);
        if (lane >= off) {
          sg += vg;
          se += ve;
        }
      }
      if (lane < kWarpsT) {
        sh.wsum[0][lane] = sg;
        sh.wsum[1][lane] = se;
      }
    }
    __syncthreads();
    uint32_t rg = (warp > 0 ? sh.wsum[0][warp - 1] : 0u) + ig - g;
    uint32_t re = (warp > 0 ? sh.wsum[1][warp - 1] : 0u) + ie - e;
    for (int w = w0; w < w1; ++w) {
      const uint32_t cg = wgt[w], ce = weq[w];
      wgt[w] = rg;
      weq[w] = re;
      rg += cg;
      re += ce;
    }
  }
  __syncthreads();
  const uint32_t below = (1u << lane) - 1u;
  for (int w = warp; w < nw; w += kWarpsT) {
    const int i = 32 * w + lane;
    const uint32_t key = i < n ? keys[i] : 0u;
    const bool gt = i < n && key > T, eq = i < n && key == T;
    const uint32_t bgt = __ballot_sync(0xFFFFFFFFu, gt), beq = __ballot_sync(0xFFFFFFFFu, eq);
    const uint32_t eq_before = weq[w] + __popc(beq & below);
    if (gt || (eq && eq_before < need)) emit(i, wgt[w] + __popc(bgt & below) + min(eq_before, need));
  }
  __syncthreads();
}

}  // namespace spc
