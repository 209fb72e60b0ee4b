// Host side of the attention entry points: the work split, the workspace
// layout and the launch sequence (the attention grid of the shape's (bit
// width, group size) variant, then combine_kernel unless the CTAs combine in a
// cluster or in the fused selection).  The kernels themselves are in
// attention.cuh, instantiated per variant in attn_b{1,2}g{32,64}.cu.
#include <algorithm>

#include "attention.cuh"

namespace spc {

// ------------------------------------------------------------ combine kernel
// Query row blockIdx.x of (b, hkv) blockIdx.y from the partials that every
// CTA of the attention grid before it stored, in partial order and with the
// arithmetic of the in-kernel combines (so every path gives identical
// results): M = the maximum of the partials' maxima, w_p = 2^(m_p - M), then
// L = sum of l_p w_p and the output at channel threadIdx.x = sum of o_p w_p,
// both as sequential multiply-adds over p.  kThreads threads, 2 * chunks
// floats of dynamic shared memory.
__global__ void __launch_bounds__(kThreads) combine_kernel(AttnArgs a) {
  extern __shared__ float s_cw[];  // [nparts] weights (first the maxima), [nparts] sums
  __shared__ float s_red[kWarps];
  __shared__ float s_L;
  grid_dependency_sync();  // the attention grid's partials are complete and visible
  const int rho = blockIdx.x, c = threadIdx.x;
  const int64_t bh = blockIdx.y;
  const int nparts = a.chunks;
  const float* base = a.part + (bh * nparts * kMaxRows + rho) * kPartStride;
  constexpr int64_t kStep = (int64_t)kMaxRows * kPartStride;  // from one partial's row to the next's
  float* s_w = s_cw;
  float* s_l = s_cw + nparts;
  float m_loc = kNeg;
  for (int p = c; p < nparts; p += kThreads) {
    const float m = __ldcg(base + p * kStep);
    s_w[p] = m;
    s_l[p] = __ldcg(base + p * kStep + 1);
    m_loc = fmaxf(m_loc, m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m_loc = fmaxf(m_loc, __shfl_xor_sync(0xFFFFFFFFu, m_loc, o));
  if ((c & 31) == 0) s_red[c >> 5] = m_loc;
  __syncthreads();
  float M = s_red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_red[w]);
  for (int p = c; p < nparts; p += kThreads) s_w[p] = fast_exp2(s_w[p] - M);
  __syncthreads();
  if (c == 0) {
    float L = 0.f;
    for (int p = 0; p < nparts; ++p) L += s_l[p] * s_w[p];
    s_L = L;
  }
  float O = 0.f;  // 16 partials' loads in flight at a time
  for (int p0 = 0; p0 < nparts; p0 += 16) {
    float ov[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) ov[u] = p0 + u < nparts ? __ldcg(base + (p0 + u) * kStep + 4 + c) : 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (p0 + u < nparts) O += ov[u] * s_w[p0 + u];
  }
  __syncthreads();
  write_row(a, bh, rho, M, s_L, O, c);
}

// ---------------------------------------------------------------- host side

static cudaError_t launch_combine(const AttnArgs& a, int64_t BH, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * a.G), (unsigned)BH, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 2 * sizeof(float) * (size_t)a.chunks;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

static const AttnVariant& variant(const spc_dims* d) {
  if (d->bits == 1) return d->group == 64 ? attn_variant_b1g64() : attn_variant_b1g32();
  return d->group == 64 ? attn_variant_b2g64() : attn_variant_b2g32();
}

struct AttnPlan {
  int chunks;
  int groups_per_chunk;  // 32-token groups per CTA (a multiple of the record's halves)
};

// One wave of resident CTAs over B*Hkv, at least four records (one per warp)
// each.  The 16-bit rows ride on the same CTAs, whatever their number.
static AttnPlan attn_plan(const spc_dims* d, bool fetch) {
  const int nh = d->group / kGroup;  // 32-token halves per record
  const int nu = num_quantized(d->N, d->R, d->group) / d->group;
  const int64_t BH = (int64_t)d->B * d->Hkv;
  AttnPlan p{1, nh};
  if (nu > 0) {
    const int64_t slots = (int64_t)spc_host::sm_count() * variant(d).resident_ctas(fetch);
    int64_t chunks = std::max<int64_t>(1, slots / BH);
    chunks = std::min<int64_t>(chunks, (nu + kWarps - 1) / kWarps);
    // A short row goes to at most kMaxCluster CTAs, whose partials then
    // combine in one cluster (one kernel instead of two), when each CTA then
    // holds at most 32 groups of 32 tokens: measured faster there (batch 1-4
    // at 4K-16K tokens), slower with more groups per CTA.
    if (chunks > kMaxCluster && ((int64_t)nu * nh + kMaxCluster - 1) / kMaxCluster <= 32) chunks = kMaxCluster;
    const int upc = (int)((nu + chunks - 1) / chunks);
    p.chunks = (nu + upc - 1) / upc;
    p.groups_per_chunk = upc * nh;
  }
  return p;
}

static size_t part_floats(const spc_dims* d, const AttnPlan& p) {
  return (size_t)d->B * d->Hkv * p.chunks * kMaxRows * kPartStride;
}

// Workspace: control words first (a fixed place, whatever k is): tickets
// [BH], ready [BH], tickets2 [BH] and the fault word; then the partials from a
// 256-byte boundary; then, for spc_decode_step, the chunks' candidates.
static size_t control_bytes(const spc_dims* d) {
  return ((((size_t)3 * d->B * d->Hkv + 1) * sizeof(uint32_t) + 255) / 256) * 256;
}

static size_t parts_bytes(const spc_dims* d) {
  return std::max(part_floats(d, attn_plan(d, false)), part_floats(d, attn_plan(d, true))) * sizeof(float);
}

// candidates kept per chunk: min(k, N_q, the chunk's positions)
static int cand_cap(const spc_dims* d, const AttnPlan& p, int32_t k) {
  return std::max(0, std::min(std::min(k, num_quantized(d->N, d->R, d->group)), p.groups_per_chunk * kGroup));
}

static size_t cand_bytes(const spc_dims* d, int32_t k_max) {
  size_t best = 0;
  for (bool fetch : {false, true}) {
    const AttnPlan p = attn_plan(d, fetch);
    best = std::max(best, (size_t)d->B * d->Hkv * p.chunks * cand_cap(d, p, k_max) * 2 * sizeof(uint32_t));
  }
  return best;
}

size_t attn_workspace_bytes(const spc_dims* d, int32_t k_max) {
  (void)k_max;  // the partials do not depend on the number of fetched rows
  return control_bytes(d) + parts_bytes(d);
}

// the fetched rows' speculative logits of the on-chip selection: [BH][k][4] floats
static size_t rowlog_bytes(const spc_dims* d, int32_t k_max) {
  return (size_t)d->B * d->Hkv * std::max(k_max, 0) * 4 * sizeof(float);
}

size_t step_workspace_bytes(const spc_dims* d, int32_t k_max) {
  return control_bytes(d) + parts_bytes(d) + cand_bytes(d, k_max) + rowlog_bytes(d, k_max);
}

// The clustered combine, when every (b, hkv)'s CTAs fit one cluster and all
// clusters are resident in one wave.
static bool use_cluster(const spc_dims* d, bool merged, bool fetch, int chunks, int64_t BH) {
  return variant(d).cluster_fits(merged, fetch, chunks, BH);
}

// The fused selection works in the attention's dynamic shared memory: a
// chunk's keys and word counts, then the leader's merge of every chunk's
// candidates and the bitmap.
static bool select_fits(const spc_dims* d, const AttnPlan& p, int32_t k_sel) {
  const int64_t words = variant(d).smem / 4;
  const int64_t nq = num_quantized(d->N, d->R, d->group);
  const int64_t len = (int64_t)p.groups_per_chunk * kGroup;
  const int64_t M = (int64_t)p.chunks * cand_cap(d, p, k_sel);
  return nq > 0 && len + 2 * (len / 32) <= words && 2 * M + nq / 32 + 2 * ((M + 31) / 32) <= words;
}

// The fused selection keeps the speculative logits of every warp's records in
// its TMEM lanes: 4 columns (heads) per 32-token half, kTmemCols per CTA.
static bool onchip_fits(const spc_dims* d, const AttnPlan& p) {
  const int nh = d->group / kGroup;
  const int units_per_warp = (p.groups_per_chunk / nh + kWarps - 1) / kWarps;
  return 4 * nh * units_per_warp <= (int)kTmemCols;
}

// Whether spc_decode_step can keep the speculative logits on chip (spec_logits == nullptr).
bool step_onchip(const spc_dims* d, int32_t k, int32_t fetch_k, int32_t next_k) {
  const bool fetch = (int64_t)d->B * d->Hkv * fetch_k > 0;
  const AttnPlan plan = attn_plan(d, fetch);
  return k > 0 && select_fits(d, plan, next_k) && onchip_fits(d, plan);
}

spc_status launch_attention(const spc_dims* d, const void* records, const uint16_t* resid,
                            const uint16_t* q, const uint16_t* kv_self, const int32_t* idx,
                            const uint32_t* bitmap, const uint16_t* staging, int32_t k, uint16_t* o, float* lse,
                            float* spec_logits, void* ws, cudaStream_t stream, const PrefetchJob* pf,
                            const SelectJob* sel, bool* sel_done) {
  const bool fetch = pf != nullptr && pf->host_dev != nullptr && (int64_t)d->B * d->Hkv * pf->k > 0;
  const AttnPlan plan = attn_plan(d, fetch);
  const int64_t BH = (int64_t)d->B * d->Hkv;
  const bool merged = k > 0;
  const bool topk = sel != nullptr && merged && lse != nullptr && select_fits(d, plan, sel->k) &&
                    (spec_logits != nullptr || onchip_fits(d, plan));
  if (sel_done != nullptr) *sel_done = topk;
  AttnArgs a;
  a.records = static_cast<const uint8_t*>(records);
  a.resid = resid;
  a.q = q;
  a.kv_self = kv_self;
  a.idx = idx;
  a.bitmap = bitmap;
  a.staging = staging;
  a.spec_logits = spec_logits;
  uint32_t* control = static_cast<uint32_t*>(ws);
  a.tickets = control;
  a.ready = control + BH;
  a.tickets2 = control + 2 * BH;
  a.fault = control + 3 * BH;
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + control_bytes(d));
  a.cand = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + control_bytes(d) + parts_bytes(d));
  a.out = o;
  a.lse = lse;
  a.k = k;
  a.Hq = d->Hq;
  a.Hkv = d->Hkv;
  a.G = d->Hq / d->Hkv;
  a.nq = num_quantized(d->N, d->R, d->group);
  a.r = d->N - a.nq;
  a.q_groups_cap = d->q_groups_cap;
  a.units_cap = d->group == 64 ? (d->q_groups_cap + 1) / 2 : d->q_groups_cap;
  a.resid_cap = d->resid_cap;
  a.chunks = plan.chunks;
  a.groups_per_chunk = plan.groups_per_chunk;
  a.Lcap = d->q_groups_cap * kGroup;
  a.qscale = d->scale * 1.4426950408889634f;
  a.pf_host = fetch ? pf->host_dev : nullptr;
  a.pf_idx = pf ? pf->idx : nullptr;
  a.pf_staging = pf ? pf->staging : nullptr;
  a.pf_ncap = pf ? pf->n_cap : 0;
  a.pf_k = pf ? pf->k : 0;
  a.pf_rows = pf ? (int32_t)((int64_t)d->B * d->Hkv * pf->k) : 0;
  a.pf_src = fetch ? pf->src : nullptr;
  a.pf_prev = fetch ? pf->prev : nullptr;
  a.pf_prev_k = fetch ? pf->prev_k : 0;
  a.sel_idx = topk ? sel->idx : nullptr;
  a.sel_src = topk ? sel->src : nullptr;
  a.sel_bitmap = topk ? sel->bitmap : nullptr;
  a.sel_k = topk ? sel->k : 0;
  a.sel_keff = topk ? std::min(sel->k, a.nq) : 0;
  a.cand_cap = topk ? cand_cap(d, plan, sel->k) : 0;
  a.sel_onchip = topk && spec_logits == nullptr ? 1 : 0;
  a.sel_rowlog = a.sel_onchip ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + control_bytes(d) + parts_bytes(d) +
                                                         cand_bytes(d, std::max(k, sel->k)))
                              : nullptr;
  const bool clustered = !topk && use_cluster(d, merged, fetch, a.chunks, BH);
  a.ext_combine = !topk && !clustered;
  cudaError_t e = variant(d).launch(a, BH, stream, merged, fetch, topk, clustered);
  if (e == cudaSuccess && a.ext_combine) e = launch_combine(a, BH, stream);
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

// Kernels that launch_attention enqueues without a fused selection: the
// attention grid, then combine_kernel unless the CTAs combine in a cluster.
int attn_kernel_count(const spc_dims* d, int32_t k, int32_t fetch_k) {
  const int64_t BH = (int64_t)d->B * d->Hkv;
  const bool fetch = BH * fetch_k > 0;
  const AttnPlan plan = attn_plan(d, fetch);
  return use_cluster(d, k > 0, fetch, plan.chunks, BH) ? 1 : 2;
}

// Kernels of one spc_decode_step: one when the selection rides on the
// attention launch, else the attention's and the separate top-k.
int step_kernel_count(const spc_dims* d, int32_t k, int32_t fetch_k, int32_t next_k) {
  const bool fetch = (int64_t)d->B * d->Hkv * fetch_k > 0;
  if (k > 0 && select_fits(d, attn_plan(d, fetch), next_k)) return 1;
  return attn_kernel_count(d, k, fetch_k) + ((d->q_groups_cap == 0 && next_k == 0) ? 0 : 1);
}

}  // namespace spc
