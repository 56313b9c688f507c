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

namespace moe {

// Norm and router projection of a decode step (T <= 8 tokens) in one launch:
// every CTA computes the RMS norm of the T tokens (the same arithmetic as
// rms_norm_kernel, so the same bits) into shared memory, CTA 0 writes it out
// (the layer's input), and each warp computes the logits of one expert:
// logits[t, e] = sum_c bf16(x[t, c] r_t) * Wr[e, c] in FP32 (each lane a
// strided share of the 16-byte chunks, then the warp's shuffle sum).  The
// router matrix is read once, spread over E/8 CTAs, so a batch-1 step does not
// stream it through a few SMs.
constexpr int NR_WARPS = 8;
constexpr int NR_MAXT = 8;

__global__ void __launch_bounds__(NR_WARPS * 32) norm_router_kernel(const uint16_t* __restrict__ x,
                                                                    const uint16_t* __restrict__ wr,
                                                                    uint16_t* __restrict__ xn,
                                                                    float* __restrict__ logits, int T, int H, int E,
                                                                    float eps) {
  extern __shared__ uint4 nr_smem[];  // the normalised tokens, [T][H] bf16
  __shared__ float s_r[NR_MAXT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c8 = H / 8;
  if (warp < T) {
    const uint4* row = reinterpret_cast<const uint4*>(x + static_cast<size_t>(warp) * H);
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
    if (lane == 0) s_r[warp] = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * c8; i += blockDim.x) {
    const int t = i / c8, c = i - t * c8;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H) + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    const float r = s_r[t];
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = pack_bf16x2(__uint_as_float(u[q] << 16) * r, __uint_as_float(u[q] & 0xffff0000u) * r);
    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
    nr_smem[i] = ov;
    if (blockIdx.x == 0) reinterpret_cast<uint4*>(xn + static_cast<size_t>(t) * H)[c] = ov;
  }
  __syncthreads();
  const int e = blockIdx.x * NR_WARPS + warp;
  if (e >= E) return;
  const uint4* wrow = reinterpret_cast<const uint4*>(wr + static_cast<size_t>(e) * H);
  float acc[NR_MAXT];
#pragma unroll
  for (int t = 0; t < NR_MAXT; ++t) acc[t] = 0.f;
  for (int c = lane; c < c8; c += 32) {
    const uint4 wv = __ldg(wrow + c);
    const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int t = 0; t < NR_MAXT; ++t) {
      if (t >= T) break;
      const uint4 xv = nr_smem[t * c8 + c];
      const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[t] = fmaf(__uint_as_float(xu[q] << 16), __uint_as_float(wu[q] << 16), acc[t]);
        acc[t] = fmaf(__uint_as_float(xu[q] & 0xffff0000u), __uint_as_float(wu[q] & 0xffff0000u), acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NR_MAXT; ++t) {
    if (t >= T) break;
    float v = acc[t];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    if (lane == 0) logits[static_cast<size_t>(t) * E + e] = v;
  }
}

int norm_router_max_tokens() { return NR_MAXT; }

cudaError_t launch_norm_router(const uint16_t* x, const uint16_t* wr, uint16_t* xn, float* logits, int T, int H,
                               int E, float eps, cudaStream_t s) {
  if (T > NR_MAXT || H % 8 != 0) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(T) * H * sizeof(uint16_t);
  if (smem > 48 * 1024) {
    const cudaError_t e0 = ensure_dyn_smem(reinterpret_cast<const void*>(norm_router_kernel), smem);
    if (e0 != cudaSuccess) return e0;
  }
  norm_router_kernel<<<(E + NR_WARPS - 1) / NR_WARPS, NR_WARPS * 32, smem, s>>>(x, wr, xn, logits, T, H, E, eps);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
