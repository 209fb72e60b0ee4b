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
#include <mutex>

#include "common.cuh"

namespace spc {
size_t attn_workspace_bytes(const spc_dims*, int32_t);
}

namespace {

// 8 MiB: enough for every shape this library is sized for on GB300 (the
// 32-layer LLaMA-3-8B step at 32K context needs about 2.5 MB per call).
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the buffer on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" spc_status spc_merged_attn_noalloc(const spc_dims* d, const void* records, const uint16_t* resid,
                                              const uint16_t* q, const int32_t* idx, const uint32_t* bitmap,
                                              const uint16_t* staging, int32_t k, uint16_t* o, float* lse,
                                              float* spec_logits, spc_stream stream) {
  const size_t need = spc_attn_workspace_bytes(d, k < 0 ? 0 : k);
  if (need == 0) return SPC_ERR_INVALID;               // invalid shape
  if (need > kNoAllocScratchBytes) return SPC_ERR_WORKSPACE;  // beyond the built-in buffer
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
