// Shared device helpers for the KDA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

namespace kda {

// Device-side status word of the library (one per device, in the library's own image; the
// library is a single translation unit). Kernels on every stream record the first error they
// meet into the same word; kda_sync_status() takes it and clears it in one atomic exchange.
__device__ unsigned int g_status = 0u;

// Slots into which kda_sync_status() moves the status word (one slot per call in flight, so
// that overlapping calls from several host threads do not read each other's result).
constexpr int kStatusSlots = 64;
__device__ unsigned int g_status_taken[kStatusSlots];

__global__ void take_status_kernel(int slot) {
  g_status_taken[slot] = atomicExch(&g_status, 0u);
}

__device__ __forceinline__ void record_status(unsigned int code) {
  atomicCAS(&g_status, 0u, code);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device, once per
// (kernel, device): the attribute persists, so later launches skip the driver call.
inline cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

}  // namespace kda
