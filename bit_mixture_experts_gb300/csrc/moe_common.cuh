// Shared device helpers of libmoe_w4 (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <utility>

#include "moe_w4.h"

namespace moe {

// Device error word: the first kernel-side fault wins (atomicCAS from 0).
// Kernels receive its address; the word itself lives in moe_abi.cu.
__device__ __forceinline__ void set_device_error(int* err, int code) {
  atomicCAS(err, 0, code);
}

// Host: address of the device error word on the current device.
int* device_error_ptr();

// Host: add n to the process-wide count of kernels launched by the library.
void note_launches(int n);

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Host-side argument checks shared by the entry points (moe_abi.cu and the
// no-allocation routing entry point in moe_route.cu), so their limits agree.
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sizes every layer call must satisfy (the GEMM kernels add their own: H and
// F multiples of 128, block_n within the chosen kernel's tile height).
inline int check_shape(int T, int H, int F, int E, int k, int bn) {
  if (T < 1 || T > (1 << 20)) return MOE_ERR_SHAPE;
  if (E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_SHAPE;
  if (H < 64 || H % 64 != 0 || F < 64 || F % 64 != 0) return MOE_ERR_SHAPE;
  if (bn < 1 || bn > 1024) return MOE_ERR_SHAPE;
  return MOE_OK;
}

// Routing-only sizes (no H or F involved).
inline int check_route_shape(int T, int E, int k, int bn) { return check_shape(T, 64, 64, E, k, bn); }

// MOE_ERR_NULL for any null pointer, then MOE_ERR_ALIGN for any pointer not 16-byte aligned.
template <typename... P>
int check_ptrs(P... ps) {
  const void* arr[] = {static_cast<const void*>(ps)...};
  for (const void* p : arr)
    if (!p) return MOE_ERR_NULL;
  for (const void* p : arr)
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  return MOE_OK;
}

// bf16 bits -> float (exact).
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// float -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Two floats -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Block-map entry of tile b.
struct Tile {
  int expert;
  int row0;
  int rows;
};

// Host side: raise a kernel's dynamic shared memory limit (cudaFuncSetAttribute) only when a launch
// needs more than the current device was given before -- the attribute persists, and the driver
// call costs microseconds of host time on every launch that repeats it.
inline cudaError_t ensure_dyn_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> given;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = given[std::make_pair(dev, func)];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) have = bytes;
  return e;
}

// Host side: resident CTAs per SM of a kernel at a block size and dynamic shared memory size,
// computed once per device and configuration.
inline cudaError_t cached_occupancy(const void* func, int threads, size_t smem, int* per_sm) {
  static std::mutex mu;
  static std::map<std::pair<std::pair<int, const void*>, std::pair<int, size_t>>, int> seen;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(std::make_pair(dev, func), std::make_pair(threads, smem));
  auto it = seen.find(key);
  if (it != seen.end()) {
    *per_sm = it->second;
    return cudaSuccess;
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, func, threads, smem);
  if (e == cudaSuccess) seen[key] = *per_sm;
  return e;
}

}  // namespace moe
