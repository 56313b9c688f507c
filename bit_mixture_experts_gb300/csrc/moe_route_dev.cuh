// Device helpers of the routing step, shared by the routing kernels and the
// fused decode kernel so that both compute the same top-k, weights, scan and
// block map (see moe_route.cu for the step itself).
#pragma once
#include "moe_common.cuh"

namespace moe {
namespace route_dev {

constexpr unsigned FULL = 0xffffffffu;

// Monotone map float -> uint32 (larger float, larger key); -0.0 and +0.0 map to
// the same key so equal logits tie and the lower expert index wins.
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t key) {
  uint32_t u = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(u);
}

// Top-k of one token by one warp.  Lane L holds experts L, L+32, ...; each of
// the k rounds takes every lane's best unchosen expert, reduces the keys with
// redux.sync (max) and then, among the lanes holding that key, the expert
// indices (min): the largest logit wins and, among equal logits, the lowest
// index.  Lane j < k ends with the j-th choice in (*id, *w).
//
// Weights: w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0) in float.  The
// difference l_j - l_0 is carried exactly as hi + lo (two-sum), so the only
// errors are expf's (<= 2 ulp), the float sum of k terms and the division:
// well under 1e-6 relative.
// COHERENT reads the row through L2 only (a row written earlier by other CTAs
// of the same kernel); otherwise through the read-only path.
template <int EPL, bool COHERENT = false>
__device__ __forceinline__ void warp_topk(const float* __restrict__ row, int E, int k, int lane,
                                          int* id_out, float* w_out) {
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    int e = i * 32 + lane;
    key[i] = e < E ? float_key(COHERENT ? __ldcg(row + e) : __ldg(row + e)) : 0u;
  }
  uint32_t chosen = 0;
  int my_id = 0;
  uint32_t my_key = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E && !((chosen >> i) & 1u) && (bi < 0 || key[i] > bk)) {
        bk = key[i];
        bi = i;
      }
    }
    const uint32_t kmax = __reduce_max_sync(FULL, bk);
    const uint32_t cand = (bi >= 0 && bk == kmax) ? static_cast<uint32_t>(bi * 32 + lane) : 0xffffffffu;
    const uint32_t e_win = __reduce_min_sync(FULL, cand);
    if ((e_win & 31u) == static_cast<uint32_t>(lane)) chosen |= 1u << (e_win >> 5);
    if (lane == j) {
      my_id = static_cast<int>(e_win);
      my_key = kmax;
    }
  }
  const float lj = key_float(my_key);
  const float l0 = key_float(__shfl_sync(FULL, my_key, 0));
  // two-sum: lj - l0 == dh + dl exactly
  const float nl0 = -l0;
  const float dh = lj + nl0;
  const float bb = dh - lj;
  const float dl = (lj - (dh - bb)) + (nl0 - bb);
  float z = 0.f;
  if (lane < k) z = expf(dh) * (1.0f + dl);
  float s = z;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) s += __shfl_xor_sync(FULL, s, m);
  *id_out = my_id;
  *w_out = z / s;
}

template <bool COHERENT = false>
__device__ __forceinline__ void warp_topk_any(const float* row, int E, int k, int lane, int* id, float* w) {
  if (E <= 32) warp_topk<1, COHERENT>(row, E, k, lane, id, w);
  else if (E <= 64) warp_topk<2, COHERENT>(row, E, k, lane, id, w);
  else if (E <= 128) warp_topk<4, COHERENT>(row, E, k, lane, id, w);
  else if (E <= 256) warp_topk<8, COHERENT>(row, E, k, lane, id, w);
  else if (E <= 512) warp_topk<16, COHERENT>(row, E, k, lane, id, w);
  else warp_topk<32, COHERENT>(row, E, k, lane, id, w);
}

// Exclusive scan of one uint64 per thread over the whole block (blockDim.x a
// multiple of 32, at most 1024).  `sm` holds 33 uint64.  Returns the exclusive
// prefix; *total receives the block sum.
__device__ __forceinline__ uint64_t block_exclusive_scan(uint64_t v, uint64_t* sm, uint64_t* total) {
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint32_t lo = __shfl_up_sync(FULL, static_cast<uint32_t>(x), d);
    uint32_t hi = __shfl_up_sync(FULL, static_cast<uint32_t>(x >> 32), d);
    if (lane >= d) x += (static_cast<uint64_t>(hi) << 32) | lo;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint64_t w = lane < nw ? sm[lane] : 0;
    uint64_t y = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      uint32_t lo = __shfl_up_sync(FULL, static_cast<uint32_t>(y), d);
      uint32_t hi = __shfl_up_sync(FULL, static_cast<uint32_t>(y >> 32), d);
      if (lane >= d) y += (static_cast<uint64_t>(hi) << 32) | lo;
    }
    if (lane < nw) sm[lane] = y - w;  // exclusive warp base
    if (lane == 31) sm[32] = y;       // block total (lanes >= nw add zero)
  }
  __syncthreads();
  uint64_t res = sm[warp] + x - v;
  *total = sm[32];
  __syncthreads();
  return res;
}

// Write the block-map rows of expert e (count c starting at row off) from
// tile index first.
__device__ __forceinline__ void emit_expert_tiles(int32_t* bm, int first, int e, int off, int c, int bn) {
  for (int i = 0, r = 0; r < c; ++i, r += bn) {
    int32_t* p = bm + 3 * (first + i);
    p[0] = e;
    p[1] = off + r;
    p[2] = min(bn, c - r);
  }
}

}  // namespace route_dev
}  // namespace moe
