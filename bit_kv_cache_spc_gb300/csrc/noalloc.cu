// spc_merged_attn_noalloc: the merged two-query attention for callers that
// cannot allocate device memory.
//
// spc_merged_attn needs a caller-provided device workspace (split-K partials
// and per-(b, hkv) tickets).  Some callers have no way to get one: code that
// runs inside a host that owns the device allocator (an inference server's
// plug-in, a custom-call hook of another framework, a real-time path where
// cudaMalloc's implicit synchronisation is not allowed).  This entry point
// takes the workspace from a fixed buffer compiled into the library instead,
// and allocates nothing: no cudaMalloc, no cudaFree, no allocating library
// routine.
//
// The buffer is a file-scope __device__ array of kNoAllocScratchBytes.  Each
// GPU on which this entry point is used holds it from then until the process
// exits.  All calls share it, so calls that overlap on the GPU (different
// streams without ordering, or several host threads) race and corrupt each
// other's results; issue them in order on one stream.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace spc {
size_t attn_workspace_bytes(const spc_dims*, int32_t);
}
namespace spc_host {
spc_status check_attn_args(const spc_dims*, const void*, const uint16_t*, const uint16_t*, const uint16_t*,
                           const int32_t*, const uint32_t*, const uint16_t*, int32_t, const uint16_t*, const float*,
                           const float*);
}

namespace {

// 8 MiB: enough for every shape this library is sized for on GB300 (the
// 32-layer LLaMA-3-8B step at 32K context needs about 2.5 MB per call).
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// The unique id of the calling thread's current CUDA context (ids are never
// reused within a process), through the driver entry points that the runtime
// hands out; false when there is no current context or no such entry point.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();  // a failed query leaves no error behind
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return false;
  return get_id(c, id) == CUDA_SUCCESS;
}

// Device address of the buffer in the current context.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress: once per context (the module, and so the buffer, is
// loaded per context; a context created after a device reset gets a new id
// and a fresh lookup), or on every call when the context id is unavailable.
cudaError_t scratch_address(void** out) {
  static std::mutex mu;
  struct Entry {
    unsigned long long ctx;
    void* addr;
  };
  static Entry cache[16] = {};
  static int n_cached = 0, next_slot = 0;
  unsigned long long id = 0;
  bool have_id = current_context_id(&id);
  if (have_id) {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cached; ++i)
      if (cache[i].ctx == id) {
        *out = cache[i].addr;
        return cudaSuccess;
      }
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (!have_id) have_id = current_context_id(&id);  // the lookup made the primary context current
  if (have_id) {
    std::lock_guard<std::mutex> lock(mu);
    cache[next_slot] = Entry{id, p};
    next_slot = (next_slot + 1) % 16;
    if (n_cached < 16) ++n_cached;
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" spc_status spc_merged_attn_noalloc(const spc_dims* d, const void* records, const uint16_t* resid,
                                              const uint16_t* q, const int32_t* idx, const uint32_t* bitmap,
                                              const uint16_t* staging, int32_t k, uint16_t* o, float* lse,
                                              float* spec_logits, spc_stream stream) {
  // the statuses spc_merged_attn would return, before anything is enqueued
  spc_status st = spc_host::check_attn_args(d, records, resid, q, nullptr, idx, bitmap, staging, k, o, lse,
                                            spec_logits);
  if (st != SPC_OK) return st;
  if (spc::attn_workspace_bytes(d, k) > kNoAllocScratchBytes) return SPC_ERR_WORKSPACE;  // beyond the buffer
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  // The buffer keeps the previous call's contents.  The attention kernel's
  // ticket words (one uint32 per (b, hkv), at the start of the workspace)
  // must start at zero; clear them on the call's stream.
  const size_t tickets = (size_t)d->B * d->Hkv * sizeof(uint32_t);
  e = cudaMemsetAsync(ws, 0, tickets, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return spc_merged_attn(d, records, resid, q, nullptr, idx, bitmap, staging, k, o, lse, spec_logits, ws,
                         kNoAllocScratchBytes, stream);
}
