// Shared device helpers of libmoe_w4 (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

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

}  // namespace moe
