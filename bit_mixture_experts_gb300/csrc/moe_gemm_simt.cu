// CUDA-core grouped expert GEMM over canonical 4-bit weights: the
// correctness-first kernel of the layer, and the one the tensor-core kernel
// is debugged against on the device.
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details, Prefill
// optimizations bullet: groupwise affine 4-bit weights (64 per group) are
// dequantised inside the grouped GEMM and accumulated in FP32.  Here each CTA
// expands a 32-wide K slice of its weight rows into shared memory (bf16
// values held as float), multiplies it with the tile's gathered rows, and never
// writes expanded weights to global memory.
//
// CTA = (block-map tile b, 32 output columns).  Warp w owns tile rows w, w+8,
// ...; lane L owns output column c0 + L.
#include "moe_common.cuh"

namespace moe {

namespace {
constexpr int SIMT_BN = 128;  // max rows per tile
constexpr int KC = 32;        // half a quantisation group per K step
constexpr int LD = KC + 1;    // padded row pitch of the shared tiles
}  // namespace

// Validates block-map entry b and fills the per-row token / weight tables.
// Returns false (and records a device error) for a malformed entry.
__device__ bool load_tile(const int32_t* __restrict__ block_map, int b, int E, int A, int T, int bn_max,
                          const int32_t* __restrict__ perm, const float* __restrict__ topk_w, int k,
                          Tile* tile, int* s_tok, float* s_wt, int* err) {
  Tile t;
  t.expert = block_map[3 * b];
  t.row0 = block_map[3 * b + 1];
  t.rows = block_map[3 * b + 2];
  bool ok = t.expert >= 0 && t.expert <= E && t.rows >= 1 && t.rows <= bn_max && t.row0 >= 0;
  if (ok) {
    if (t.expert < E) ok = t.row0 + t.rows <= A;
    else ok = t.row0 >= A && t.row0 + t.rows <= A + T;
  }
  if (!ok) {
    if (threadIdx.x == 0) set_device_error(err, MOE_DEV_BAD_BLOCK);
    return false;
  }
  for (int i = threadIdx.x; i < t.rows; i += blockDim.x) {
    int r = t.row0 + i;
    if (r < A) {
      int a = perm[r];
      if (a < 0 || a >= A) {
        set_device_error(err, MOE_DEV_BAD_INDEX);
        a = 0;
      }
      s_tok[i] = a / k;
      s_wt[i] = topk_w[a];
    } else {
      s_tok[i] = r - A;
      s_wt[i] = 1.0f;
    }
  }
  *tile = t;
  return true;
}

// MODE 0: gate/up + SwiGLU -> h bf16 [A+T, F].  MODE 1: down -> y bf16 [A+T, H].
template <int MODE>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const uint16_t* __restrict__ act, int T, int H, int F,
                                                        int E, int k, const uint32_t* __restrict__ wq,
                                                        const uint16_t* __restrict__ ws,
                                                        const uint16_t* __restrict__ wb,
                                                        const int32_t* __restrict__ perm,
                                                        const float* __restrict__ topk_w,
                                                        const int32_t* __restrict__ block_map,
                                                        const int32_t* __restrict__ num_blocks, int bn,
                                                        void* __restrict__ out, int* err) {
  constexpr int NR = MODE == 0 ? 64 : 32;  // weight rows per CTA
  __shared__ float s_x[SIMT_BN * LD];
  __shared__ float s_w[NR * LD];
  __shared__ int s_tok[SIMT_BN];
  __shared__ float s_wt[SIMT_BN];
  __shared__ Tile s_tile;

  const int b = blockIdx.x;
  if (b >= *num_blocks) return;
  const int A = T * k;
  {
    Tile t;
    bool ok = load_tile(block_map, b, E, A, T, min(bn, SIMT_BN), perm, topk_w, k, &t, s_tok, s_wt, err);
    if (!ok) return;  // uniform across the CTA: every thread read the same entry
    if (threadIdx.x == 0) s_tile = t;
  }
  __syncthreads();
  const Tile tile = s_tile;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = MODE == 0 ? H : F;
  const int rows_total = MODE == 0 ? 2 * F : H;
  const int c0 = blockIdx.y * 32;  // output column block (feature f or channel c)
  const size_t mat = static_cast<size_t>(tile.expert) * rows_total;

  float acc0[16], acc1[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc0[j] = acc1[j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += KC) {
    // gathered activation rows -> float
    for (int idx = threadIdx.x; idx < tile.rows * (KC / 8); idx += blockDim.x) {
      const int i = idx / (KC / 8), v = idx % (KC / 8);
      const size_t src_row = MODE == 0 ? static_cast<size_t>(s_tok[i]) : static_cast<size_t>(tile.row0 + i);
      const uint4 q = *reinterpret_cast<const uint4*>(act + src_row * K + k0 + v * 8);
      const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        s_x[i * LD + v * 8 + 2 * h] = __uint_as_float(wv[h] << 16);
        s_x[i * LD + v * 8 + 2 * h + 1] = __uint_as_float(wv[h] & 0xffff0000u);
      }
    }
    // weight rows of this K group, expanded to bf16 values: w = bf16(q*s + b)
    for (int idx = threadIdx.x; idx < NR * (KC / 8); idx += blockDim.x) {
      const int rr = idx / (KC / 8), wd = idx % (KC / 8);
      int grow;
      if (MODE == 0) grow = rr < 32 ? c0 + rr : F + c0 + (rr - 32);  // gate rows then up rows
      else grow = c0 + rr;
      const size_t row = mat + grow;
      const uint32_t word = wq[row * (K / 8) + k0 / 8 + wd];
      const float s = bf16_bits_to_float(ws[row * (K / 64) + k0 / 64]);
      const float bb = bf16_bits_to_float(wb[row * (K / 64) + k0 / 64]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float q = static_cast<float>((word >> (4 * i)) & 0xfu);
        s_w[rr * LD + wd * 8 + i] = bf16_bits_to_float(float_to_bf16_bits(fmaf(q, s, bb)));
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < KC; ++kk) {
      const float w0 = s_w[lane * LD + kk];
      const float w1 = MODE == 0 ? s_w[(32 + lane) * LD + kk] : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int i = warp + 8 * j;
        if (i < tile.rows) {
          const float xv = s_x[i * LD + kk];
          acc0[j] = fmaf(xv, w0, acc0[j]);
          if (MODE == 0) acc1[j] = fmaf(xv, w1, acc1[j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int i = warp + 8 * j;
    if (i >= tile.rows) continue;
    if (MODE == 0) {
      uint16_t* h = static_cast<uint16_t*>(out);
      h[static_cast<size_t>(tile.row0 + i) * F + c0 + lane] = float_to_bf16_bits(silu(acc0[j]) * acc1[j]);
    } else {
      uint16_t* y = static_cast<uint16_t*>(out);
      y[static_cast<size_t>(tile.row0 + i) * H + c0 + lane] = float_to_bf16_bits(acc0[j]);
    }
  }
}

cudaError_t launch_gemm_simt(int mode, const uint16_t* act, int T, int H, int F, int E, int k, const uint32_t* wq,
                             const uint16_t* ws, const uint16_t* wb, const int32_t* perm, const float* topk_w,
                             const int32_t* block_map, const int32_t* num_blocks, int bn, int nb_cap, void* out,
                             cudaStream_t s) {
  int* err = device_error_ptr();
  if (mode == MOE_GATE_UP_SWIGLU) {
    dim3 grid(nb_cap, F / 32);
    gemm_simt_kernel<0><<<grid, 256, 0, s>>>(act, T, H, F, E, k, wq, ws, wb, perm, topk_w, block_map, num_blocks,
                                             bn, out, err);
  } else {
    dim3 grid(nb_cap, H / 32);
    gemm_simt_kernel<1><<<grid, 256, 0, s>>>(act, T, H, F, E, k, wq, ws, wb, perm, topk_w, block_map, num_blocks,
                                             bn, out, err);
  }
  note_launches(1);
  return cudaGetLastError();
}

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
