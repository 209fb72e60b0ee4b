// GPU twin of the seeded input generator in synth/__init__.py (same
// definition, bit-identical output): SplitMix64 draws (Steele, Lea & Flood,
// OOPSLA 2014) turned into bf16 standard-normal values by the inverse-CDF
// table of synth/normal_bf16_table.npz.  It holds none of the SpeCache
// method's arithmetic; it only makes the large synthetic K/V tensors quickly.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

constexpr int kBucketBits = 12;  // index on the top 12 of the 63 uniform bits
constexpr int kBuckets = 1 << kBucketBits;

// Number of thresholds <= u in th[lo..hi) (the answer lies in [lo, hi]).
__device__ __forceinline__ int upper_bound(const uint64_t* th, int lo, int hi, uint64_t u) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (th[mid] <= u)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

// Magnitude index = number of thresholds <= u; the bucket table narrows the
// search to the thresholds that share u's top bits.
__device__ __forceinline__ uint16_t normal_bits(uint64_t r, const uint64_t* th, const uint16_t* vals,
                                                const uint16_t* bstart, const uint16_t* bend) {
  const uint64_t u = r & 0x7FFFFFFFFFFFFFFFull;
  const int bkt = (int)(u >> (63 - kBucketBits));
  const int j = upper_bound(th, bstart[bkt], bend[bkt], u);
  return (uint16_t)(vals[j] | ((uint16_t)(r >> 63) << 15));
}

__device__ __forceinline__ uint16_t times8_bf16(uint16_t b) {
  float f = __uint_as_float((uint32_t)b << 16) * 8.0f;  // exact: a power-of-two scaling
  return (uint16_t)(__float_as_uint(f) >> 16);
}

__global__ void synth_kv_kernel(uint64_t key_k, uint64_t key_v, int64_t total, int32_t Hkv, int32_t N,
                                int32_t D, const int32_t* __restrict__ outl, const uint64_t* __restrict__ th_g,
                                const uint16_t* __restrict__ vals_g, int32_t n_th, uint16_t* __restrict__ K,
                                uint16_t* __restrict__ V) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* th = reinterpret_cast<uint64_t*>(smem);
  uint16_t* bstart = reinterpret_cast<uint16_t*>(th + n_th);
  uint16_t* bend = bstart + kBuckets;
  uint16_t* vals = bend + kBuckets;
  for (int i = threadIdx.x; i < n_th; i += blockDim.x) th[i] = th_g[i];
  for (int i = threadIdx.x; i <= n_th; i += blockDim.x) vals[i] = vals_g[i];
  __syncthreads();
  for (int j = threadIdx.x; j < kBuckets; j += blockDim.x) {
    const uint64_t first = (uint64_t)j << (63 - kBucketBits);
    const uint64_t last = first + ((1ull << (63 - kBucketBits)) - 1);
    bstart[j] = (uint16_t)upper_bound(th, 0, n_th, first);
    bend[j] = (uint16_t)upper_bound(th, 0, n_th, last);
  }
  __syncthreads();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t step = (uint64_t)(i + 1) * kGamma;
    if (K != nullptr) {
      uint16_t kb = normal_bits(mix64(key_k + step), th, vals, bstart, bend);
      if (outl != nullptr) {
        const int c = (int)(i % D);
        const int h = (int)((i / ((int64_t)D * N)) % Hkv);
        const int32_t* oc = outl + 4 * h;
        if (c == oc[0] || c == oc[1] || c == oc[2] || c == oc[3]) kb = times8_bf16(kb);
      }
      K[i] = kb;
    }
    if (V != nullptr) V[i] = normal_bits(mix64(key_v + step), th, vals, bstart, bend);
  }
}

}  // namespace

extern "C" {

// K, V: bf16 [B][Hkv][N][D]; element i is draw i of the streams key_k, key_v.
// outliers: device int32 [Hkv][4] (key channels scaled by 8) or NULL.
// K or V may be NULL to skip that tensor.  Returns a cudaError_t.
int32_t spc_synth_kv(uint64_t key_k, uint64_t key_v, int32_t B, int32_t Hkv, int32_t N, int32_t D,
                     const int32_t* outliers, const uint64_t* thresh, const uint16_t* vals, int32_t n_thresh,
                     uint16_t* K, uint16_t* V, cudaStream_t stream) {
  const int64_t total = (int64_t)B * Hkv * N * D;
  if (total == 0) return 0;
  const size_t smem = (size_t)n_thresh * 8 + 2 * (size_t)kBuckets * 2 + ((size_t)n_thresh + 1) * 2;
  if (n_thresh >= 65535) return (int32_t)cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(synth_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int32_t)e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (total + 255) / 256;
  const int grid = (int)(want < (int64_t)sms * 2 ? want : (int64_t)sms * 2);
  synth_kv_kernel<<<grid, 1024, smem, stream>>>(key_k, key_v, total, Hkv, N, D, outliers, thresh, vals, n_thresh, K,
                                                V);
  return (int32_t)cudaGetLastError();
}

}  // extern "C"
