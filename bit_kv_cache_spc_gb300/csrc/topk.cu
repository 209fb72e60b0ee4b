// ArgTopK(A_{1,:}) of the SpeCache page (Algorithm 3; Algorithm 2 for the
// pre-decoding step): per (b, hkv) the k positions of C' with the largest
// speculative-token attention probability, summed over the G query heads of
// the KV head.
//
// One thread-block cluster per (b, hkv) row.  Each CTA of the cluster turns
// its slice of the row into scores S(n) = sum_h exp(l_h(n) - lse_h) held in
// shared memory as uint32 bit patterns (S >= 0, so integer order is float
// order), then the cluster runs an MSB-first radix select (4 passes of 8 bits)
// for the k-th largest key, summing the CTAs' histograms through distributed
// shared memory.  A final ordered compaction writes the selected positions in
// ascending order (ties at the threshold go to the lower position) and the
// selection bitmap.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace spc {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

struct TopkArgs {
  const float* logits;  // [BH][G][Lcap]
  const float* lse;     // [B][2][Hq]
  int32_t* idx;         // [BH][k]
  uint32_t* bitmap;     // [BH][q_groups_cap]
  int32_t Hq, Hkv, G, nq, k, keff, Lcap, q_groups_cap;
  int32_t slice;        // positions per CTA, multiple of 32
};

struct TopkShared {
  uint32_t hist[2][256];     // this CTA's histogram, double-buffered by pass parity
  uint32_t total[256];       // cluster-wide histogram of the current pass
  uint32_t warp_cnt[2][kTopkWarps];
  uint32_t counts[2];        // this CTA's (> threshold, == threshold) counts
  uint32_t prefix, prefix_mask, remaining;
};

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkArgs a) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ TopkShared sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned rank = cluster.block_rank();
  const unsigned ncta = cluster.num_blocks();
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.Hkv), hk = (int)(bh % a.Hkv);
  const int n0 = (int)rank * a.slice;
  const int len = max(0, min(a.slice, a.nq - n0));

  // ---- scores ----
  float lse_h[4];
#pragma unroll
  for (int gi = 0; gi < 4; ++gi)
    lse_h[gi] = gi < a.G ? a.lse[((int64_t)b * 2 + 1) * a.Hq + hk * a.G + gi] : 0.f;
  const float* lrow = a.logits + (bh * a.G) * (int64_t)a.Lcap + n0;
  for (int i = tid; i < len; i += kTopkThreads) {
    float s = 0.f;
    for (int gi = 0; gi < a.G; ++gi) s += expf(lrow[(int64_t)gi * a.Lcap + i] - lse_h[gi]);
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
        const bool in = i < len && ((keys[i < len ? i : 0] ^ prefix) & pmask) == 0u;
        const uint32_t active = __ballot_sync(0xFFFFFFFFu, in);
        if (in) {
          const uint32_t bin = (keys[i] >> shift) & 255u;
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
        uint32_t above = 0;  // keys in the bins of higher lanes
        for (int l2 = 0; l2 < 32; ++l2) {
          const uint32_t v = __shfl_sync(0xFFFFFFFFu, own, l2);
          if (l2 > lane) above += v;
        }
        const uint32_t rem = sh.remaining;
        const bool mine = above < rem && rem <= above + own;
        if (mine) {
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

  // ---- ordered compaction ----
  const uint32_t T = sh.prefix;
  const uint32_t need = sh.remaining;  // keys == T to take, lowest positions first
  const bool any = a.keff > 0;
  uint32_t my_gt = 0, my_eq = 0;
  if (any) {
    for (int i = tid; i < len; i += kTopkThreads) {
      my_gt += keys[i] > T;
      my_eq += keys[i] == T;
    }
  }
  for (int off = 16; off > 0; off >>= 1) {
    my_gt += __shfl_xor_sync(0xFFFFFFFFu, my_gt, off);
    my_eq += __shfl_xor_sync(0xFFFFFFFFu, my_eq, off);
  }
  if (lane == 0) {
    sh.warp_cnt[0][warp] = my_gt;
    sh.warp_cnt[1][warp] = my_eq;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t g = 0, e = 0;
    for (int w = 0; w < kTopkWarps; ++w) {
      g += sh.warp_cnt[0][w];
      e += sh.warp_cnt[1][w];
    }
    sh.counts[0] = g;
    sh.counts[1] = e;
  }
  cluster.sync();
  uint32_t base_gt = 0, base_eq = 0;
  for (unsigned r = 0; r < rank; ++r) {
    const uint32_t* pc = cluster.map_shared_rank(&sh.counts[0], r);
    base_gt += pc[0];
    base_eq += pc[1];
  }
  __syncthreads();

  int32_t* out = a.idx + bh * a.k;
  uint32_t* bm = a.bitmap + bh * a.q_groups_cap;
  uint32_t run_gt = base_gt, run_eq = base_eq;
  for (int i0 = 0; i0 < len; i0 += kTopkThreads) {
    const int i = i0 + tid;
    const uint32_t key = i < len ? keys[i] : 0u;
    const bool gt = any && i < len && key > T;
    const bool eq = any && i < len && key == T;
    const uint32_t bgt = __ballot_sync(0xFFFFFFFFu, gt), beq = __ballot_sync(0xFFFFFFFFu, eq);
    const uint32_t below = (1u << lane) - 1u;
    if (lane == 0) {
      sh.warp_cnt[0][warp] = __popc(bgt);
      sh.warp_cnt[1][warp] = __popc(beq);
    }
    __syncthreads();
    uint32_t wgt = 0, weq = 0, tgt = 0, teq = 0;
    for (int w = 0; w < kTopkWarps; ++w) {
      const uint32_t cg_ = sh.warp_cnt[0][w], ce = sh.warp_cnt[1][w];
      if (w < warp) {
        wgt += cg_;
        weq += ce;
      }
      tgt += cg_;
      teq += ce;
    }
    const uint32_t gt_before = run_gt + wgt + __popc(bgt & below);
    const uint32_t eq_before = run_eq + weq + __popc(beq & below);
    const bool sel = gt || (eq && eq_before < need);
    const uint32_t bsel = __ballot_sync(0xFFFFFFFFu, sel);
    const uint32_t pos = gt_before + min(eq_before, need);
    if (sel && pos < (uint32_t)a.keff) out[pos] = n0 + i;
    if (lane == 0 && i0 + 32 * warp < len) bm[(n0 + i0 + 32 * warp) >> 5] = bsel;
    run_gt += tgt;
    run_eq += teq;
    __syncthreads();
  }
  if (rank == 0) {
    for (int j = a.keff + tid; j < a.k; j += kTopkThreads) out[j] = -1;
    for (int w = (a.nq >> 5) + tid; w < a.q_groups_cap; w += kTopkThreads) bm[w] = 0u;
  }
  cluster.sync();  // peers may still read this CTA's counters
}

spc_status launch_topk(const spc_dims* d, const float* logits, const float* lse, int32_t k, int32_t* idx,
                       uint32_t* bitmap, cudaStream_t stream) {
  TopkArgs a;
  a.logits = logits;
  a.lse = lse;
  a.idx = idx;
  a.bitmap = bitmap;
  a.Hq = d->Hq;
  a.Hkv = d->Hkv;
  a.G = d->Hq / d->Hkv;
  a.nq = num_quantized(d->N, d->R);
  a.k = k;
  a.keff = std::min(k, a.nq);
  a.Lcap = d->q_groups_cap * kGroup;
  a.q_groups_cap = d->q_groups_cap;
  int ncta = std::max(1, std::min(8, (a.nq + 16383) / 16384));
  a.slice = std::max(32, ((a.nq + ncta - 1) / ncta + 31) / 32 * 32);
  if (a.slice > 32768) return SPC_ERR_UNSUPPORTED;
  const int64_t BH = (int64_t)d->B * d->Hkv;
  const size_t smem = (size_t)a.slice * sizeof(uint32_t);
  static unsigned long long configured = 0ull;
  cudaError_t e = spc_host::ensure_smem_limit(configured, topk_kernel, 32768 * (int)sizeof(uint32_t));
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncta, (unsigned)BH, 1);
    cfg.blockDim = dim3(kTopkThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_kernel, a);
  }
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

}  // namespace spc
