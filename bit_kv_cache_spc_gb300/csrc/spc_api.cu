// extern "C" entry points of libspc (declared in include/spc.h): argument
// validation, then one launch sequence per call on the caller's stream.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace spc {
spc_status launch_quantize(const spc_dims*, const uint16_t*, const uint16_t*, void*, uint16_t*, cudaStream_t);
size_t attn_workspace_bytes(const spc_dims*, int32_t);
spc_status launch_attention(const spc_dims*, const void*, const uint16_t*, const uint16_t*, const uint16_t*,
                            const int32_t*, const uint32_t*, const uint16_t*, int32_t, uint16_t*, float*, float*,
                            void*, cudaStream_t, const PrefetchJob*, const SelectJob*, bool*);
size_t step_workspace_bytes(const spc_dims*, int32_t);
int attn_kernel_count(const spc_dims*, int32_t, int32_t);
int step_kernel_count(const spc_dims*, int32_t, int32_t, int32_t);
bool step_onchip(const spc_dims*, int32_t, int32_t, int32_t);
spc_status launch_topk(const spc_dims*, const float*, const float*, int32_t, int32_t*, uint32_t*, cudaStream_t,
                       const int32_t* prev_idx = nullptr, int32_t prev_k = 0, int32_t* src = nullptr);
spc_status launch_host_gather(const spc_dims*, const uint16_t*, int64_t, const int32_t*, int32_t, uint16_t*,
                              int32_t, cudaStream_t, const int32_t* src = nullptr, const uint16_t* prev = nullptr,
                              int32_t prev_k = 0);
spc_status launch_append(const spc_dims*, const uint16_t*, const uint16_t*, void*, uint16_t*, uint16_t*, int64_t,
                         cudaStream_t);
}  // namespace spc

namespace spc_host {

static thread_local int32_t g_last_cuda_error = 0;

void set_cuda_error(cudaError_t e) { g_last_cuda_error = (int32_t)e; }

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

}  // namespace spc_host

namespace {

using spc_host::aligned16;

// Shape checks shared by every call.
spc_status check_dims(const spc_dims* d) {
  if (d == nullptr) return SPC_ERR_INVALID;
  if (d->B <= 0 || d->Hq <= 0 || d->Hkv <= 0 || d->D <= 0 || d->N < 0 || d->R < 0 || d->q_groups_cap < 0 ||
      d->resid_cap < 0)
    return SPC_ERR_INVALID;
  if (d->Hq % d->Hkv != 0) return SPC_ERR_INVALID;
  if (d->bits != 1 && d->bits != 2) return SPC_ERR_INVALID;
  if (!(std::isfinite(d->scale) && d->scale > 0.f)) return SPC_ERR_INVALID;
  const int G = d->Hq / d->Hkv;
  if (d->D != spc::kD || (d->group != 32 && d->group != 64)) return SPC_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4) return SPC_ERR_UNSUPPORTED;
  const int32_t nq = spc::num_quantized(d->N, d->R, d->group);
  if (nq / spc::kGroup > d->q_groups_cap) return SPC_ERR_INVALID;
  if (d->N - nq > d->resid_cap) return SPC_ERR_INVALID;
  return SPC_OK;
}

// Device address of a pinned, mapped host buffer, or SPC_ERR_NOT_MAPPED.
spc_status mapped_device_pointer(const void* host, const void** dev) {
  cudaPointerAttributes attr;
  const cudaError_t e = cudaPointerGetAttributes(&attr, host);
  if (e != cudaSuccess) {
    cudaGetLastError();  // the failed query leaves no sticky error; clear it
    return SPC_ERR_NOT_MAPPED;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return SPC_ERR_NOT_MAPPED;
  *dev = attr.devicePointer;
  return SPC_OK;
}

}  // namespace

namespace spc_host {

// Argument checks of every attention entry point other than those of its
// workspace, in the order they apply; nothing is launched or enqueued.
spc_status check_attn_args(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                           const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap,
                           const uint16_t* staging, int32_t k, const uint16_t* o, const float* lse,
                           const float* spec_logits) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  const int32_t nq = spc::num_quantized(d->N, d->R, d->group);
  if (q == nullptr || o == nullptr) return SPC_ERR_INVALID;
  if (nq > 0 && records == nullptr) return SPC_ERR_INVALID;
  if (d->N - nq > 0 && resid == nullptr) return SPC_ERR_INVALID;
  if (!aligned16(records) || !aligned16(resid) || !aligned16(q) || !aligned16(kv_self) || !aligned16(o) ||
      !aligned16(lse) || !aligned16(spec_logits))
    return SPC_ERR_INVALID;
  if (k < 0 || k > (1 << 24)) return SPC_ERR_INVALID;
  if (k > 0) {
    if (idx == nullptr || bitmap == nullptr || staging == nullptr || !aligned16(staging)) return SPC_ERR_INVALID;
  }
  return SPC_OK;
}

}  // namespace spc_host

namespace {

// [a, a + na) and [b, b + nb) share a byte
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}
// bytes of a [B][Hkv][k][2][D] bf16 staging buffer
size_t staging_bytes(const spc_dims* d, int64_t k) { return (size_t)d->B * d->Hkv * (size_t)k * 2 * d->D * 2; }
// A carried pre-fetch writes fetch_staging while the attention reads staging
// (k rows) and, with kept rows, copies from prev (prev_k rows): a shared byte
// would race.
bool fetch_buffers_overlap(const spc_dims* d, const uint16_t* staging, int32_t k, const uint16_t* fetch_staging,
                           int32_t fetch_k, const uint16_t* prev, int32_t prev_k) {
  const size_t out = staging_bytes(d, fetch_k);
  return (k > 0 && overlap(staging, staging_bytes(d, k), fetch_staging, out)) ||
         (prev_k > 0 && overlap(prev, staging_bytes(d, prev_k), fetch_staging, out));
}

spc_status attn_common(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                       const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap, const uint16_t* staging, int32_t k,
                       uint16_t* o, float* lse, float* spec_logits, void* ws, size_t ws_bytes,
                       spc_stream stream, const spc::PrefetchJob* pf = nullptr,
                       const spc::SelectJob* sel = nullptr, bool* sel_done = nullptr) {
  spc_status st = spc_host::check_attn_args(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse,
                                            spec_logits);
  if (st != SPC_OK) return st;
  if (ws == nullptr || !aligned16(ws)) return SPC_ERR_INVALID;
  const size_t need = sel != nullptr ? spc::step_workspace_bytes(d, std::max(k, sel->k))
                                     : spc::attn_workspace_bytes(d, k);
  if (ws_bytes < need) return SPC_ERR_WORKSPACE;
  return spc::launch_attention(d, records, resid, q, kv_self, k > 0 ? idx : nullptr, k > 0 ? bitmap : nullptr,
                               k > 0 ? staging : nullptr, k, o, lse, spec_logits, ws,
                               reinterpret_cast<cudaStream_t>(stream), pf, sel, sel_done);
}

}  // namespace

extern "C" {

int32_t spc_abi_version(void) { return SPC_ABI_VERSION; }

const char* spc_status_string(spc_status s) {
  switch (s) {
    case SPC_OK: return "ok";
    case SPC_ERR_INVALID: return "invalid argument";
    case SPC_ERR_UNSUPPORTED: return "unsupported shape";
    case SPC_ERR_CUDA: return "CUDA error";
    case SPC_ERR_NOT_MAPPED: return "host pointer is not mapped pinned memory";
    case SPC_ERR_WORKSPACE: return "workspace too small";
    case SPC_ERR_TIMEOUT: return "a kernel's bounded wait ran out (see spc_read_device_status)";
  }
  return "unknown status";
}

int32_t spc_last_cuda_error(void) { return spc_host::g_last_cuda_error; }

int32_t spc_num_quantized(const spc_dims* d) {
  if (check_dims(d) == SPC_ERR_INVALID) return -1;
  return spc::num_quantized(d->N, d->R, d->group);
}

size_t spc_records_bytes(const spc_dims* d) {
  if (d == nullptr || d->B <= 0 || d->Hkv <= 0 || d->q_groups_cap < 0 || (d->bits != 1 && d->bits != 2) ||
      (d->group != 32 && d->group != 64))
    return 0;
  return (size_t)d->B * d->Hkv * spc::records_cap(d->group, d->q_groups_cap) *
         (size_t)spc::record_bytes(d->bits, d->group);
}

size_t spc_resid_bytes(const spc_dims* d) {
  if (d == nullptr || d->B <= 0 || d->Hkv <= 0 || d->resid_cap < 0 || d->D <= 0) return 0;
  return (size_t)d->B * d->Hkv * d->resid_cap * 2 * d->D * sizeof(uint16_t);
}

spc_status spc_quantize_kv(const spc_dims* d, const uint16_t* k, const uint16_t* v, void* records,
                           uint16_t* resid, spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  const int32_t nq = spc::num_quantized(d->N, d->R, d->group);
  if (d->N > 0 && (k == nullptr || v == nullptr)) return SPC_ERR_INVALID;
  if (nq > 0 && records == nullptr) return SPC_ERR_INVALID;
  if (d->N - nq > 0 && resid == nullptr) return SPC_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(records) || !aligned16(resid)) return SPC_ERR_INVALID;
  return spc::launch_quantize(d, k, v, records, resid, reinterpret_cast<cudaStream_t>(stream));
}

spc_status spc_offload_kv(const spc_dims* d, const uint16_t* k, const uint16_t* v, uint16_t* host_kv,
                          int64_t n_cap, spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  if (d->N == 0) return SPC_OK;
  if (k == nullptr || v == nullptr || host_kv == nullptr || n_cap < d->N) return SPC_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(host_kv)) return SPC_ERR_INVALID;
  const void* host_dev = nullptr;
  st = mapped_device_pointer(host_kv, &host_dev);  // pinned host memory: the copy engines reach it directly
  if (st != SPC_OK) return st;
  const size_t row = (size_t)spc::kD * sizeof(uint16_t);  // 256 bytes
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // rows (b, hkv, n) of K go to host rows (b, hkv, n) at byte 0, of V at byte 256:
  // one strided copy of all B*Hkv*N rows when n_cap == N, else one per (b, hkv)
  // run of N rows (the host runs are n_cap rows apart)
  const int64_t BH = (int64_t)d->B * d->Hkv;
  const int64_t runs = n_cap == d->N ? 1 : BH;
  const size_t height = (size_t)(n_cap == d->N ? BH * d->N : d->N);
  for (int64_t bh = 0; bh < runs; ++bh) {
    for (int kv = 0; kv < 2; ++kv) {
      const uint16_t* src = (kv == 0 ? k : v) + bh * (int64_t)d->N * spc::kD;
      uint16_t* dst = host_kv + (bh * n_cap * 2 + kv) * spc::kD;
      const cudaError_t e = cudaMemcpy2DAsync(dst, 2 * row, src, row, row, height, cudaMemcpyDeviceToHost, s);
      if (e != cudaSuccess) {
        spc_host::set_cuda_error(e);
        return SPC_ERR_CUDA;
      }
    }
  }
  return SPC_OK;
}

spc_status spc_append_kv(const spc_dims* d, const uint16_t* k_new, const uint16_t* v_new, void* records,
                         uint16_t* resid, uint16_t* host_kv, int64_t n_cap, spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  if (d->N >= (1 << 30)) return SPC_ERR_INVALID;
  const int32_t nq = spc::num_quantized(d->N, d->R, d->group);
  const int32_t nq1 = spc::num_quantized(d->N + 1, d->R, d->group);
  if (k_new == nullptr || v_new == nullptr || resid == nullptr) return SPC_ERR_INVALID;
  if (d->N - nq + 1 > d->resid_cap) return SPC_ERR_INVALID;  // room for the new row
  if (nq1 > nq && (records == nullptr || nq1 / spc::kGroup > d->q_groups_cap)) return SPC_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(records) || !aligned16(resid) || !aligned16(host_kv))
    return SPC_ERR_INVALID;
  const void* host_dev = nullptr;
  if (host_kv != nullptr) {
    if (n_cap <= d->N) return SPC_ERR_INVALID;
    st = mapped_device_pointer(host_kv, &host_dev);
    if (st != SPC_OK) return st;
  }
  return spc::launch_append(d, k_new, v_new, records, resid, static_cast<uint16_t*>(const_cast<void*>(host_dev)),
                            n_cap, reinterpret_cast<cudaStream_t>(stream));
}

size_t spc_attn_workspace_bytes(const spc_dims* d, int32_t k_max) {
  if (check_dims(d) != SPC_OK || k_max < 0 || k_max > (1 << 24)) return 0;
  return spc::attn_workspace_bytes(d, k_max);
}

spc_status spc_decode_attn2(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                            const uint16_t* kv_self, uint16_t* o, float* lse, float* spec_logits, void* ws,
                            size_t ws_bytes, spc_stream stream) {
  return attn_common(d, records, resid, q, kv_self, nullptr, nullptr, nullptr, 0, o, lse, spec_logits, ws,
                     ws_bytes, stream);
}

spc_status spc_merged_attn(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                           const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap,
                           const uint16_t* staging, int32_t k, uint16_t* o, float* lse, float* spec_logits,
                           void* ws, size_t ws_bytes, spc_stream stream) {
  return attn_common(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse, spec_logits, ws, ws_bytes,
                     stream);
}

spc_status spc_merged_attn_fetch(const spc_dims* d, const void* records, const uint16_t* resid,
                                 const uint16_t* q, const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap,
                                 const uint16_t* staging, int32_t k, uint16_t* o, float* lse, float* spec_logits,
                                 void* ws, size_t ws_bytes, const uint16_t* fetch_host_kv, int64_t fetch_n_cap,
                                 const int32_t* fetch_idx, int32_t fetch_k, uint16_t* fetch_staging,
                                 spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  if (fetch_k < 0 || fetch_k > (1 << 24) || fetch_n_cap < 0) return SPC_ERR_INVALID;
  if (fetch_k == 0)
    return attn_common(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse, spec_logits, ws, ws_bytes,
                       stream);
  if (fetch_host_kv == nullptr || fetch_idx == nullptr || fetch_staging == nullptr) return SPC_ERR_INVALID;
  if (!aligned16(fetch_host_kv) || !aligned16(fetch_staging)) return SPC_ERR_INVALID;
  if (fetch_buffers_overlap(d, staging, k, fetch_staging, fetch_k, nullptr, 0)) return SPC_ERR_INVALID;
  const void* dev = nullptr;
  st = mapped_device_pointer(fetch_host_kv, &dev);
  if (st != SPC_OK) return st;
  spc::PrefetchJob job{static_cast<const uint16_t*>(dev), fetch_n_cap, fetch_idx, fetch_k, fetch_staging};
  return attn_common(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse, spec_logits, ws, ws_bytes,
                     stream, &job);
}

spc_status spc_merged_attn_fetch_prev(const spc_dims* d, const void* records, const uint16_t* resid,
                                      const uint16_t* q, const uint16_t* kv_self, const int32_t* idx,
                                      const uint32_t* bitmap, const uint16_t* staging, int32_t k, uint16_t* o,
                                      float* lse, float* spec_logits, void* ws, size_t ws_bytes,
                                      const uint16_t* fetch_host_kv, int64_t fetch_n_cap, const int32_t* fetch_idx,
                                      int32_t fetch_k, uint16_t* fetch_staging, const int32_t* fetch_src,
                                      const uint16_t* fetch_prev_staging, int32_t fetch_prev_k, spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  if (fetch_k < 0 || fetch_k > (1 << 24) || fetch_n_cap < 0 || fetch_prev_k < 0 || fetch_prev_k > (1 << 24))
    return SPC_ERR_INVALID;
  if (fetch_k == 0)
    return attn_common(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse, spec_logits, ws, ws_bytes,
                       stream);
  if (fetch_host_kv == nullptr || fetch_idx == nullptr || fetch_staging == nullptr || fetch_src == nullptr)
    return SPC_ERR_INVALID;
  if (!aligned16(fetch_host_kv) || !aligned16(fetch_staging)) return SPC_ERR_INVALID;
  if (fetch_prev_k > 0 && (fetch_prev_staging == nullptr || !aligned16(fetch_prev_staging)))
    return SPC_ERR_INVALID;
  if (fetch_buffers_overlap(d, staging, k, fetch_staging, fetch_k, fetch_prev_staging, fetch_prev_k))
    return SPC_ERR_INVALID;
  const void* dev = nullptr;
  st = mapped_device_pointer(fetch_host_kv, &dev);
  if (st != SPC_OK) return st;
  spc::PrefetchJob job{static_cast<const uint16_t*>(dev), fetch_n_cap, fetch_idx, fetch_k, fetch_staging,
                       fetch_src, fetch_prev_k > 0 ? fetch_prev_staging : nullptr, fetch_prev_k};
  return attn_common(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse, spec_logits, ws, ws_bytes,
                     stream, &job);
}

int32_t spc_attn_kernel_count(const spc_dims* d, int32_t k, int32_t fetch_k) {
  if (check_dims(d) != SPC_OK || k < 0 || k > (1 << 24) || fetch_k < 0 || fetch_k > (1 << 24)) return -1;
  return spc::attn_kernel_count(d, k, fetch_k);
}

int32_t spc_decode_step_kernel_count(const spc_dims* d, int32_t k, int32_t fetch_k, int32_t next_k) {
  if (check_dims(d) != SPC_OK || k < 0 || k > (1 << 24) || fetch_k < 0 || fetch_k > (1 << 24) || next_k < 0 ||
      next_k > (1 << 24))
    return -1;
  return spc::step_kernel_count(d, k, fetch_k, next_k);
}

int32_t spc_decode_step_on_chip(const spc_dims* d, int32_t k, int32_t fetch_k, int32_t next_k) {
  if (check_dims(d) != SPC_OK || k < 0 || k > (1 << 24) || fetch_k < 0 || fetch_k > (1 << 24) || next_k < 0 ||
      next_k > (1 << 24))
    return -1;
  return spc::step_onchip(d, k, fetch_k, next_k) ? 1 : 0;
}

size_t spc_step_workspace_bytes(const spc_dims* d, int32_t k_max) {
  if (check_dims(d) != SPC_OK || k_max < 0 || k_max > (1 << 24)) return 0;
  return spc::step_workspace_bytes(d, k_max);
}

// spc_decode_step and spc_decode_step_prev: with next_src, the pre-fetch keeps
// the rows already staged (fetch_src, fetch_prev) and the selection reports
// each position's index in idx.
static spc_status decode_step(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                              const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap,
                              const uint16_t* staging, int32_t k, uint16_t* o, float* lse, float* spec_logits,
                              int32_t next_k, int32_t* next_idx, uint32_t* next_bitmap, int32_t* next_src, void* ws,
                              size_t ws_bytes, const uint16_t* fetch_host_kv, int64_t fetch_n_cap,
                              const int32_t* fetch_idx, int32_t fetch_k, uint16_t* fetch_staging,
                              const int32_t* fetch_src, const uint16_t* fetch_prev, int32_t fetch_prev_k,
                              bool keep, spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  const int32_t nq = spc::num_quantized(d->N, d->R, d->group);
  if (next_k < 0 || next_k > (1 << 24)) return SPC_ERR_INVALID;
  if (next_bitmap == nullptr || (next_k > 0 && next_idx == nullptr)) return SPC_ERR_INVALID;
  if (keep && next_k > 0 &&
      (next_src == nullptr || (k > 0 && overlap(next_idx, (size_t)d->B * d->Hkv * next_k * 4, idx,
                                                  (size_t)d->B * d->Hkv * k * 4))))
    return SPC_ERR_INVALID;
  if (nq > 0 && lse == nullptr) return SPC_ERR_INVALID;
  if (nq > 262144) return SPC_ERR_UNSUPPORTED;
  // without a logits buffer the selection must ride on the attention with the logits on chip
  if (nq > 0 && spec_logits == nullptr &&
      (fetch_k < 0 || fetch_k > (1 << 24) || k < 0 || k > (1 << 24) || !spc::step_onchip(d, k, fetch_k, next_k)))
    return SPC_ERR_UNSUPPORTED;
  spc::PrefetchJob job{nullptr, fetch_n_cap, fetch_idx, fetch_k, fetch_staging};
  const spc::PrefetchJob* pf = nullptr;
  if (fetch_k != 0) {
    if (fetch_k < 0 || fetch_k > (1 << 24) || fetch_n_cap < 0) return SPC_ERR_INVALID;
    if (fetch_host_kv == nullptr || fetch_idx == nullptr || fetch_staging == nullptr) return SPC_ERR_INVALID;
    if (!aligned16(fetch_host_kv) || !aligned16(fetch_staging)) return SPC_ERR_INVALID;
    if (keep) {
      if (fetch_src == nullptr || fetch_prev_k < 0 || fetch_prev_k > (1 << 24)) return SPC_ERR_INVALID;
      if (fetch_prev_k > 0 && (fetch_prev == nullptr || !aligned16(fetch_prev))) return SPC_ERR_INVALID;
      job.src = fetch_src;
      job.prev = fetch_prev_k > 0 ? fetch_prev : nullptr;
      job.prev_k = fetch_prev_k;
    }
    if (fetch_buffers_overlap(d, staging, k, fetch_staging, fetch_k, job.prev, job.prev_k)) return SPC_ERR_INVALID;
    const void* dev = nullptr;
    st = mapped_device_pointer(fetch_host_kv, &dev);
    if (st != SPC_OK) return st;
    job.host_dev = static_cast<const uint16_t*>(dev);
    pf = &job;
  }
  spc::SelectJob sel{next_idx, next_bitmap, next_k, keep && next_k > 0 ? next_src : nullptr};
  bool fused = false;
  st = attn_common(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse, spec_logits, ws, ws_bytes,
                   stream, pf, &sel, &fused);
  if (st != SPC_OK || fused) return st;
  // the selection could not ride on this attention launch: its own launch, right after
  if (d->q_groups_cap == 0 && next_k == 0) return SPC_OK;
  return spc::launch_topk(d, spec_logits, lse, next_k, next_idx, next_bitmap, reinterpret_cast<cudaStream_t>(stream),
                          idx, k, keep && next_k > 0 ? next_src : nullptr);
}

spc_status spc_decode_step(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                           const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap, const uint16_t* staging, int32_t k,
                           uint16_t* o, float* lse, float* spec_logits, int32_t next_k, int32_t* next_idx,
                           uint32_t* next_bitmap, void* ws, size_t ws_bytes, const uint16_t* fetch_host_kv,
                           int64_t fetch_n_cap, const int32_t* fetch_idx, int32_t fetch_k,
                           uint16_t* fetch_staging, spc_stream stream) {
  return decode_step(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse, spec_logits, next_k, next_idx,
                     next_bitmap, nullptr, ws, ws_bytes, fetch_host_kv, fetch_n_cap, fetch_idx, fetch_k,
                     fetch_staging, nullptr, nullptr, 0, false, stream);
}

spc_status spc_decode_step_prev(const spc_dims* d, const void* records, const uint16_t* resid, const uint16_t* q,
                                const uint16_t* kv_self, const int32_t* idx, const uint32_t* bitmap,
                                const uint16_t* staging, int32_t k, uint16_t* o, float* lse, float* spec_logits,
                                int32_t next_k, int32_t* next_idx, uint32_t* next_bitmap, int32_t* next_src,
                                void* ws, size_t ws_bytes, const uint16_t* fetch_host_kv, int64_t fetch_n_cap,
                                const int32_t* fetch_idx, int32_t fetch_k, uint16_t* fetch_staging,
                                const int32_t* fetch_src, const uint16_t* fetch_prev_staging, int32_t fetch_prev_k,
                                spc_stream stream) {
  return decode_step(d, records, resid, q, kv_self, idx, bitmap, staging, k, o, lse, spec_logits, next_k, next_idx,
                     next_bitmap, next_src, ws, ws_bytes, fetch_host_kv, fetch_n_cap, fetch_idx, fetch_k,
                     fetch_staging, fetch_src, fetch_prev_staging, fetch_prev_k, true, stream);
}

spc_status spc_read_device_status(void* ws, const spc_dims* d, spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  if (ws == nullptr) return SPC_ERR_INVALID;
  uint32_t* fault = static_cast<uint32_t*>(ws) + 3 * (int64_t)d->B * d->Hkv;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, fault, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && v != 0u) e = cudaMemsetAsync(fault, 0, sizeof(v), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return v != 0u ? SPC_ERR_TIMEOUT : SPC_OK;
}

// The arguments of both top-k entry points; SPC_OK when they are valid.
static spc_status check_topk_args(const spc_dims* d, const float* spec_logits, const float* lse, int32_t k,
                                  const int32_t* idx, const uint32_t* bitmap) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  const int32_t nq = spc::num_quantized(d->N, d->R, d->group);
  if (k < 0 || k > (1 << 24)) return SPC_ERR_INVALID;
  if (bitmap == nullptr || (k > 0 && idx == nullptr)) return SPC_ERR_INVALID;
  if (nq > 0 && (spec_logits == nullptr || lse == nullptr)) return SPC_ERR_INVALID;
  if (nq > 0 && !aligned16(spec_logits)) return SPC_ERR_INVALID;  // read in 16-byte pieces
  if (nq > 262144) return SPC_ERR_UNSUPPORTED;
  return SPC_OK;
}

spc_status spc_topk_select(const spc_dims* d, const float* spec_logits, const float* lse, int32_t k,
                           int32_t* idx, uint32_t* bitmap, spc_stream stream) {
  const spc_status st = check_topk_args(d, spec_logits, lse, k, idx, bitmap);
  if (st != SPC_OK) return st;
  if (d->q_groups_cap == 0 && k == 0) return SPC_OK;
  return spc::launch_topk(d, spec_logits, lse, k, idx, bitmap, reinterpret_cast<cudaStream_t>(stream));
}

spc_status spc_topk_select_prev(const spc_dims* d, const float* spec_logits, const float* lse, int32_t k,
                                int32_t* idx, uint32_t* bitmap, const int32_t* prev_idx, int32_t prev_k,
                                int32_t* src, spc_stream stream) {
  const spc_status st = check_topk_args(d, spec_logits, lse, k, idx, bitmap);
  if (st != SPC_OK) return st;
  if (prev_k < 0 || prev_k > (1 << 24)) return SPC_ERR_INVALID;
  if (k > 0 && (src == nullptr ||
                (prev_k > 0 && (prev_idx == nullptr || overlap(prev_idx, (size_t)d->B * d->Hkv * prev_k * 4, idx,
                                                               (size_t)d->B * d->Hkv * k * 4)))))
    return SPC_ERR_INVALID;
  if (d->q_groups_cap == 0 && k == 0) return SPC_OK;
  return spc::launch_topk(d, spec_logits, lse, k, idx, bitmap, reinterpret_cast<cudaStream_t>(stream), prev_idx,
                          prev_k, k > 0 ? src : nullptr);
}

spc_status spc_host_gather(const spc_dims* d, const uint16_t* host_kv, int64_t n_cap, const int32_t* idx,
                           int32_t k, uint16_t* staging, int32_t max_ctas, spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  if (k < 0 || n_cap < 0 || max_ctas < 0) return SPC_ERR_INVALID;
  if (k == 0) return SPC_OK;
  if (host_kv == nullptr || idx == nullptr || staging == nullptr) return SPC_ERR_INVALID;
  if (!aligned16(host_kv) || !aligned16(staging)) return SPC_ERR_INVALID;
  const void* dev = nullptr;
  st = mapped_device_pointer(host_kv, &dev);
  if (st != SPC_OK) return st;
  return spc::launch_host_gather(d, static_cast<const uint16_t*>(dev), n_cap, idx, k, staging, max_ctas,
                                 reinterpret_cast<cudaStream_t>(stream));
}


spc_status spc_host_gather_prev(const spc_dims* d, const uint16_t* host_kv, int64_t n_cap, const int32_t* idx,
                                int32_t k, uint16_t* staging, const int32_t* src, const uint16_t* prev_staging,
                                int32_t prev_k, int32_t max_ctas, spc_stream stream) {
  spc_status st = check_dims(d);
  if (st != SPC_OK) return st;
  if (k < 0 || n_cap < 0 || max_ctas < 0 || prev_k < 0 || prev_k > (1 << 24)) return SPC_ERR_INVALID;
  if (k == 0) return SPC_OK;
  if (host_kv == nullptr || idx == nullptr || staging == nullptr || src == nullptr) return SPC_ERR_INVALID;
  if (!aligned16(host_kv) || !aligned16(staging)) return SPC_ERR_INVALID;
  if (prev_k > 0 && (prev_staging == nullptr || !aligned16(prev_staging) ||
                     overlap(prev_staging, staging_bytes(d, prev_k), staging, staging_bytes(d, k))))
    return SPC_ERR_INVALID;
  const void* dev = nullptr;
  st = mapped_device_pointer(host_kv, &dev);
  if (st != SPC_OK) return st;
  return spc::launch_host_gather(d, static_cast<const uint16_t*>(dev), n_cap, idx, k, staging, max_ctas,
                                 reinterpret_cast<cudaStream_t>(stream), src,
                                 prev_k > 0 ? prev_staging : nullptr, prev_k);
}

}  // extern "C"
