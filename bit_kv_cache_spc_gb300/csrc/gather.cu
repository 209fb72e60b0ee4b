// Pre-fetch(C_kappa) of the SpeCache page (Algorithm 3): the selected 16-bit
// key/value rows are copied from the full-precision cache in CPU memory into
// an HBM staging buffer.  On GB300 the host cache is pinned, device-mapped
// Grace memory reached over NVLink-C2C, so the copy is a kernel that loads
// the 512-byte rows directly (zero-copy) rather than one DMA call per
// scattered row: one warp moves one row with 16-byte loads per lane, and each
// warp keeps kRowsInFlight rows outstanding to cover the link latency.
#include "common.cuh"

namespace spc {

constexpr int kRowsInFlight = 4;

__global__ void __launch_bounds__(256) host_gather_kernel(const uint4* __restrict__ host, int64_t n_cap,
                                                           const int32_t* __restrict__ idx, int32_t k,
                                                           uint4* __restrict__ staging, int64_t total_rows) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int64_t base = w0 * kRowsInFlight; base < total_rows; base += warps * kRowsInFlight) {
    uint4 v[kRowsInFlight];
    int64_t dst[kRowsInFlight];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int64_t row = base + u;  // row = bh * k + j
      dst[u] = -1;
      if (row < total_rows) {
        const int32_t n = idx[row];
        if (n >= 0 && n < n_cap) {  // out-of-range positions are skipped, never read
          const int64_t bh = row / k;
          v[u] = host[(bh * n_cap + n) * 32 + lane];  // 512 B = 32 x 16 B: K row then V row
          dst[u] = row * 32 + lane;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u)
      if (dst[u] >= 0) staging[dst[u]] = v[u];
  }
}

spc_status launch_host_gather(const spc_dims* d, const uint16_t* host_dev, int64_t n_cap, const int32_t* idx,
                              int32_t k, uint16_t* staging, int32_t max_ctas, cudaStream_t stream) {
  const int64_t total_rows = (int64_t)d->B * d->Hkv * k;
  if (total_rows == 0) return SPC_OK;
  const int64_t need = (total_rows + 8 * kRowsInFlight - 1) / (8 * kRowsInFlight);
  int64_t grid = std::min<int64_t>(need, (int64_t)spc_host::sm_count() * 4);
  if (max_ctas > 0) grid = std::min<int64_t>(grid, max_ctas);
  host_gather_kernel<<<(unsigned)grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(host_dev), n_cap, idx, k,
                                                          reinterpret_cast<uint4*>(staging), total_rows);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

}  // namespace spc
