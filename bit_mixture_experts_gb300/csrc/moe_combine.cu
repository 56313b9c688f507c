// Weighted gather-combine of the layer: each token's k routed rows of y and
// its shared-expert row, back to token order.
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details, Model
// bullet: every token goes through 8 of the 256 routed experts plus one shared
// expert, so its output is the router-weighted sum of its 8 routed expert
// outputs plus the shared expert's (weight 1; the pages give it no gate).
#include "moe_common.cuh"

namespace moe {

// --------------------------------------------------------------------------
// combine: out[t] = bf16(sum_j topk_w[t, j] y[inv_perm[t k + j]] + y[A + t])
// One thread per 8 channels of a token (16-byte loads of each y row), the
// FP32 sum in the fixed order j = 0 .. k-1, then the shared row.  Rows are
// taken 16 at a time (k + 1 <= 16 in one batch) with all their index and row
// loads issued before the sums, so the latency of the gather is paid once.
// RB rows per batch: k + 1 rounded up to one of the instantiated sizes, so
// the rows of a token normally arrive in one batch without idle registers.
// --------------------------------------------------------------------------
template <int RB>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y,
                                                      const int32_t* __restrict__ inv_perm,
                                                      const float* __restrict__ topk_w, uint16_t* __restrict__ out,
                                                      int T, int H, int k, int* err) {
  const int c8 = H / 8;  // 8-channel chunks per row
  const int A = T * k;
  const size_t n = static_cast<size_t>(T) * c8;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / c8), c = static_cast<int>(i - static_cast<size_t>(t) * c8);
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j0 = 0; j0 <= k; j0 += RB) {
      int r[RB];
      float w[RB];
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        const int j = j0 + b;
        r[b] = -1;
        w[b] = 0.f;
        if (j < k) {
          r[b] = __ldg(inv_perm + static_cast<size_t>(t) * k + j);
          w[b] = __ldg(topk_w + static_cast<size_t>(t) * k + j);
        } else if (j == k) {
          r[b] = A + t;
          w[b] = 1.0f;
        }
      }
      uint4 v[RB];
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        const int j = j0 + b;
        const bool ok = j <= k && r[b] >= 0 && r[b] < A + T && (j == k || r[b] < A);
        if (j <= k && !ok) set_device_error(err, MOE_DEV_BAD_INDEX);
        v[b] = ok ? __ldg(reinterpret_cast<const uint4*>(y + static_cast<size_t>(r[b]) * H) + c)
                  : make_uint4(0u, 0u, 0u, 0u);
        if (!ok) w[b] = 0.f;
      }
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        const uint32_t u[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = fmaf(w[b], __uint_as_float(u[q] << 16), acc[2 * q]);
          acc[2 * q + 1] = fmaf(w[b], __uint_as_float(u[q] & 0xffff0000u), acc[2 * q + 1]);
        }
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H)[c] = o;
  }
}

// Grid of the resident CTAs only (each thread then takes the same number of
// items, give or take one), from the occupancy of the instantiated kernel.
template <int RB>
static cudaError_t launch_combine_rb(const uint16_t* y, const int32_t* inv_perm, const float* topk_w, uint16_t* out,
                                     int T, int H, int k, int num_sms, cudaStream_t s) {
  static int occ = 0;
  if (occ == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, combine_kernel<RB>, 256, 0) != cudaSuccess)
    occ = 0;
  if (occ <= 0) occ = 2;
  const size_t n = static_cast<size_t>(T) * (H / 8);
  size_t blocks = (n + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms) * occ;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  combine_kernel<RB><<<static_cast<unsigned>(blocks), 256, 0, s>>>(y, inv_perm, topk_w, out, T, H, k,
                                                                   device_error_ptr());
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* y, const int32_t* inv_perm, const float* topk_w, uint16_t* out, int T,
                           int H, int k, int num_sms, cudaStream_t s) {
  if (k + 1 <= 3) return launch_combine_rb<3>(y, inv_perm, topk_w, out, T, H, k, num_sms, s);
  if (k + 1 <= 9) return launch_combine_rb<9>(y, inv_perm, topk_w, out, T, H, k, num_sms, s);
  return launch_combine_rb<16>(y, inv_perm, topk_w, out, T, H, k, num_sms, s);
}

}  // namespace moe
