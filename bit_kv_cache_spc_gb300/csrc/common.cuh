// Shared device helpers of libspc (sm_103a).  Nothing here is method
// arithmetic; the kernels in quantize.cu, attention.cu, topk.cu and gather.cu
// carry the SpeCache steps.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spc.h"

namespace spc {

constexpr int kD = 128;       // head dimension handled by this build
constexpr int kGroup = 32;    // tokens per record; tokens (keys) / channels (values) per group at g = 32
constexpr int kMaxRows = 8;   // 2 queries x G query heads per KV head, G <= 4

// Quantised tokens: whole groups of `group` (32 or 64) tokens, leaving at
// least R (and fewer than R + group) tokens in the bf16 residual window.
__host__ __device__ inline int32_t num_quantized(int32_t N, int32_t R, int32_t group) {
  return N > R ? ((N - R) / group) * group : 0;
}

// Bytes of one record of the low-bit copy: a 32-token group at g = 32; a
// 64-token group at g = 64, its two halves' code planes with the group's
// metadata stored once.
__host__ __device__ inline int64_t record_bytes(int32_t bits, int32_t group = 32) {
  return group == 64 ? 2048 * (int64_t)bits + 1024 : 1024 * (int64_t)(bits + 1);
}
// Records per (b, hkv) for a capacity of q_groups_cap 32-token groups.
__host__ __device__ inline int32_t records_cap(int32_t group, int32_t q_groups_cap) {
  return group == 64 ? (q_groups_cap + 1) / 2 : q_groups_cap;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Round binary32 to bf16, nearest-even (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte global->shared copy that bypasses L1 (cp.async.cg).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
// 4-byte global->shared copy (cp.async.ca: the only form for sizes below 16).
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_addr(smem_dst)), "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// D = A(16x16, f16, row) * B(16x8, f16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 values packed as f16x2 (x in the low half), round to nearest.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed binary32 pairs (sm_100+ f32x2 instructions): one issue for two lanes
// of arithmetic, each rounded like the scalar instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_pack(a.x, a.y)), "l"(f2_pack(b.x, b.y)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n"
      : "=l"(r)
      : "l"(f2_pack(a.x, a.y)), "l"(f2_pack(b.x, b.y)), "l"(f2_pack(c.x, c.y)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_pack(a.x, a.y)), "l"(f2_pack(b.x, b.y)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(r) : "l"(f2_pack(a.x, a.y)), "l"(f2_pack(b.x, b.y)));
  return f2_unpack(r);
}

// Packed fp16 addition on the bit patterns of two f16x2 values.
__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation waits here until the previous kernel in the stream has
// completed and its memory is visible (immediately when there is none), then
// lets the next kernel's CTAs be scheduled while this grid still runs.
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
  return r;
}

}  // namespace spc

namespace spc {
// A Pre-fetch job carried by an attention launch: rows idx of the mapped host
// cache host_dev ([B][Hkv][n_cap][2][D] bf16) into staging ([B][Hkv][k][2][D]).
// With src (else null), row j whose src[j] >= 0 is still staged from the
// previous selection and is copied from prev ([B][Hkv][prev_k][2][D], device)
// instead of the host.
struct PrefetchJob {
  const uint16_t* host_dev;
  int64_t n_cap;
  const int32_t* idx;
  int32_t k;
  uint16_t* staging;
  const int32_t* src;
  const uint16_t* prev;
  int32_t prev_k;
};

// ArgTopK fused into a merged attention launch (spc_decode_step).  With src
// (else null), each selected position's index in the launch's own idx (the
// previous selection), or -1.
struct SelectJob {
  int32_t* idx;      // [B][Hkv][k]
  uint32_t* bitmap;  // [B][Hkv][q_groups_cap]
  int32_t k;
  int32_t* src;      // [B][Hkv][k]
};
}  // namespace spc

// Host-side helpers shared by the entry points.
namespace spc_host {

void set_cuda_error(cudaError_t e);
int sm_count();  // SMs of the current device (cached per device)
bool aligned16(const void* p);
int current_device();

// Raises a kernel's dynamic shared-memory limit once per device (the attribute
// is per context); later calls are free, so launches inside a stream capture
// make no runtime configuration calls.  `done` holds one bit per device < 64
// and must be a distinct static of the caller for every kernel.
template <typename Kernel>
cudaError_t ensure_smem_limit(unsigned long long& done, Kernel* fn, int bytes) {
  const int dev = current_device();
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0ull && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0ull) __atomic_fetch_or(&done, bit, __ATOMIC_ACQ_REL);
  return e;
}

}  // namespace spc_host
