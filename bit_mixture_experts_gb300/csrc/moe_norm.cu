// Unit-gain RMS norm of each token's activations, the glue between MoE layers
// in the decode chain: out[t] = bf16(x[t] / sqrt(mean_c x[t, c]^2 + eps)).
//
// The pages' model is a stack of blocks ("Perplexity Open Sources Lily",
// Technical Details, Model bullet), whose MoE layers read normalised
// activations; the pages give no detail of the normalisation, so the chain
// uses the plainest one: RMS over the hidden dimension, no learned gain.
//
// One warp per token: 16-byte loads of 8 bf16, the sum of squares in FP32 per
// lane then over the warp (shuffles), the scale 1 / sqrt(mean + eps) with IEEE
// square root and division, each output rounded once to nearest even.
#include "moe_common.cuh"

namespace moe {

__global__ void __launch_bounds__(256) rms_norm_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ out,
                                                       int T, int H, float eps) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int c8 = H / 8;
  for (int t = warp; t < T; t += nwarps) {
    const uint4* row = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    float ss = 0.f;
    for (int c = lane; c < c8; c += 32) {
      const uint4 v = __ldg(row + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = __uint_as_float(u[q] << 16), b = __uint_as_float(u[q] & 0xffff0000u);
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
    uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H);
    for (int c = lane; c < c8; c += 32) {
      const uint4 v = __ldg(row + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o[q] = pack_bf16x2(__uint_as_float(u[q] << 16) * r, __uint_as_float(u[q] & 0xffff0000u) * r);
      dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

cudaError_t launch_rms_norm(const uint16_t* x, uint16_t* out, int T, int H, float eps, int num_sms, cudaStream_t s) {
  int blocks = (T * 32 + 255) / 256;
  if (blocks > 4 * num_sms) blocks = 4 * num_sms;
  if (blocks < 1) blocks = 1;
  rms_norm_kernel<<<blocks, 256, 0, s>>>(x, out, T, H, eps);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
