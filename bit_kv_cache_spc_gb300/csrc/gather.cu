// Pre-fetch(C_kappa) of the SpeCache page (Algorithm 3): the selected 16-bit
// key/value rows are copied from the full-precision cache in CPU memory into
// an HBM staging buffer.  On GB300 the host cache is pinned, device-mapped
// Grace memory reached over NVLink-C2C, so the copy is a kernel that loads
// the 512-byte rows directly (zero-copy) rather than one DMA call per
// scattered row.  Each warp streams its rows through a ring of kRing
// shared-memory slots with cp.async (one 16-byte piece per lane and row), so
// kRing - 1 rows per warp are in flight over the link; the oldest row is
// written to the staging buffer once its copy group has landed.  A few CTAs
// therefore keep the link busy, which lets the gather run beside other
// kernels on a second stream.
#include "common.cuh"

namespace spc {

constexpr int kGatherWarps = 4;
constexpr int kRing = 16;  // row slots per warp (512 bytes each)

// With src (else null), a row whose src entry is >= 0 is still staged from
// the previous selection: it is copied from prev ([B][Hkv][prev_k][2][D],
// device) at that slot instead of from the host.
__global__ void __launch_bounds__(32 * kGatherWarps) host_gather_kernel(const uint16_t* __restrict__ host,
                                                                         int64_t n_cap,
                                                                         const int32_t* __restrict__ idx, int32_t k,
                                                                         uint4* __restrict__ staging,
                                                                         int64_t total_rows,
                                                                         const int32_t* __restrict__ src,
                                                                         const uint16_t* __restrict__ prev,
                                                                         int32_t prev_k) {
  __shared__ __align__(16) uint4 ring[kGatherWarps][kRing][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n_warps = (int64_t)gridDim.x * kGatherWarps;
  const int64_t w0 = (int64_t)blockIdx.x * kGatherWarps + warp;
  const int64_t my_rows = w0 < total_rows ? (total_rows - w0 + n_warps - 1) / n_warps : 0;  // rows w0 + n_warps * i
  uint4(*slots)[32] = ring[warp];

  // Positions of rows 32w .. 32w+31 of this warp (one per lane) for the window
  // being issued (pos) and the next one (pos_next, loaded a window ahead so
  // that its latency hides behind 32 rows of copies).  An out-of-range
  // position is skipped, never read.
  auto load_pos = [&](int64_t i0) -> int32_t {
    int32_t n = -1;
    if (i0 + lane < my_rows) {
      n = idx[w0 + n_warps * (i0 + lane)];
      if (n < 0 || n >= n_cap) n = -1;
    }
    return n;
  };
  // the rows' previous slots (-1: read from the host), loaded with their positions
  auto load_src = [&](int64_t i0) -> int32_t {
    int32_t sj = -1;
    if (src != nullptr && i0 + lane < my_rows) {
      sj = src[w0 + n_warps * (i0 + lane)];
      if (sj >= prev_k) sj = -1;
    }
    return sj;
  };
  int32_t pos = load_pos(0), pos_next = load_pos(32);
  int32_t sj_w = load_src(0), sj_next = load_src(32);
  uint32_t live = __ballot_sync(0xFFFFFFFFu, pos >= 0);
  uint32_t slot_live = 0u;  // per ring slot: the row in it is copied

  auto issue = [&](int64_t i) {
    if (i < my_rows) {
      const int u = (int)(i & 31);
      if (u == 0 && i > 0) {  // next window
        pos = pos_next;
        pos_next = load_pos(i + 32);
        sj_w = sj_next;
        sj_next = load_src(i + 32);
        live = __ballot_sync(0xFFFFFFFFu, pos >= 0);
      }
      const int n = __shfl_sync(0xFFFFFFFFu, pos, u);
      const int sj = __shfl_sync(0xFFFFFFFFu, sj_w, u);
      const uint32_t bit = 1u << (i % kRing);
      if ((live >> u) & 1u) {
        const int64_t row = w0 + n_warps * i;
        const uint16_t* from = sj >= 0 ? prev + ((row / k) * prev_k + sj) * (2 * kD)  // still staged
                                       : host + ((row / k) * n_cap + n) * (2 * kD);
        cp_async16(&slots[i % kRing][lane], from + 8 * lane);
        slot_live |= bit;
      } else {
        slot_live &= ~bit;
      }
    }
    cp_async_commit();
  };

  for (int64_t i = 0; i < kRing - 1; ++i) issue(i);
  for (int64_t i = 0; i < my_rows; ++i) {
    issue(i + kRing - 1);
    cp_async_wait<kRing - 1>();
    __syncwarp();
    if ((slot_live >> (i % kRing)) & 1u) staging[(w0 + n_warps * i) * 32 + lane] = slots[i % kRing][lane];
    __syncwarp();  // the slot is refilled by the next issue
  }
  cp_async_wait<0>();
}

spc_status launch_host_gather(const spc_dims* d, const uint16_t* host_dev, int64_t n_cap, const int32_t* idx,
                              int32_t k, uint16_t* staging, int32_t max_ctas, cudaStream_t stream,
                              const int32_t* src, const uint16_t* prev, int32_t prev_k) {
  const int64_t total_rows = (int64_t)d->B * d->Hkv * k;
  if (total_rows == 0) return SPC_OK;
  // one warp per 32 rows at most, up to two CTAs per SM
  const int64_t need = (total_rows + 32 * kGatherWarps - 1) / (32 * kGatherWarps);
  int64_t grid = std::min<int64_t>(need, (int64_t)spc_host::sm_count() * 2);
  if (max_ctas > 0) grid = std::min<int64_t>(grid, max_ctas);
  host_gather_kernel<<<(unsigned)grid, 32 * kGatherWarps, 0, stream>>>(
      host_dev, n_cap, idx, k, reinterpret_cast<uint4*>(staging), total_rows, prev != nullptr ? src : nullptr, prev,
      prev != nullptr ? prev_k : 0);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    spc_host::set_cuda_error(e);
    return SPC_ERR_CUDA;
  }
  return SPC_OK;
}

}  // namespace spc
