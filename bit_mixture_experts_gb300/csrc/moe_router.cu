// Router projection fused with the top-k: logits = x Wr^T (bf16 operands,
// FP32 accumulation on the tensor cores) and, in the same kernel, the k
// largest logits of every token with their renormalised softmax weights.
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details, Model
// bullet: a router chooses 8 of the 256 experts for every token.  The router
// is a projection of the token's activations onto one row per expert; its
// logits feed the top-k of the routing step.
//
// Work: one cluster of E/64 CTAs per block of 128 tokens.  CTA r of the
// cluster computes the logits of experts 64r .. 64r+63 for the block's 128
// tokens with tcgen05 MMAs (M = 128 tokens, N = 64 experts, K = 64 per stage;
// x and Wr tiles staged by TMA in 128-byte swizzled atoms, accumulator in
// TMEM) and writes them to the logits output.  After a cluster barrier every
// logit of the block is visible to the whole cluster, and CTA r takes the
// top-k of its share of the block's tokens (one warp per token, the same
// selection and weight arithmetic as moe_route, reading the logits through
// L2).
//
// Roles (256 threads): warp 0 issues the TMA copies, warp 1 allocates TMEM and
// issues the MMAs, warps 4-7 read the accumulator (one token per thread);
// then all eight warps run the top-k.  Every wait is bounded (MOE_DEV_TIMEOUT).
#include <cuda.h>
#include <string.h>

#include "moe_common.cuh"
#include "moe_ptx.cuh"
#include "moe_route_dev.cuh"
#include "moe_tmap.cuh"

namespace moe {

namespace {

constexpr int RT_M = 128;        // tokens per cluster (the MMA's M)
constexpr int RT_N = 64;         // experts per CTA (the MMA's N)
constexpr int RT_K = 64;         // K per stage: one 128-byte swizzled atom of bf16
constexpr int RT_STAGES = 4;
constexpr int RT_THREADS = 256;
constexpr int RT_A_BYTES = RT_M * 128;   // x tile of one stage
constexpr int RT_B_BYTES = RT_N * 128;   // Wr tile of one stage
constexpr int RT_STAGE_BYTES = RT_A_BYTES + RT_B_BYTES;
constexpr int RT_BAR_FULL = 0, RT_BAR_EMPTY = RT_STAGES, RT_BAR_D = 2 * RT_STAGES, RT_NBAR = 2 * RT_STAGES + 1;
constexpr int RT_SMEM = RT_STAGES * RT_STAGE_BYTES + 256 + 1024;

struct RouterParams {
  float* logits;
  int32_t* ids;
  float* w;
  int* err;
  unsigned long long wait_cycles;
  uint32_t sleep_ns;
  int T, H, E, k;
};

// Bounded wait of a whole warp on phase `parity` of `bar`; false on timeout (recorded).
__device__ __forceinline__ bool rt_wait(uint32_t bar, uint32_t parity, const RouterParams& p) {
  // the first probe does not block: a try_wait without a time hint may wait for a while inside the
  // instruction, past a short limit, without the limit being checked
  if (__all_sync(0xffffffffu, ptx::mbar_test_wait(bar, parity))) return true;
  const long long t0 = clock64();
  for (;;) {
    // a limit shorter than 20 us is polled without sleeping (the sleep is only a hint)
    const bool done = p.sleep_ns >= 20000u ? ptx::mbar_try_wait_sleep(bar, parity, p.sleep_ns)
                                           : ptx::mbar_test_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if (static_cast<unsigned long long>(clock64() - t0) > p.wait_cycles) {
      if ((threadIdx.x & 31) == 0) set_device_error(p.err, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// Wait that ignores the time limit for at least about 10 ms: copies and MMAs
// already issued must not outlive the CTA or its tensor memory.
__device__ __forceinline__ void rt_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait_sleep(bar, parity, 20000u))
    if (clock64() - t0 > 20000000ll) return;
}

}  // namespace

__global__ void __launch_bounds__(RT_THREADS) router_kernel(const RouterParams p,
                                                            const __grid_constant__ CUtensorMap tmap_x,
                                                            const __grid_constant__ CUtensorMap tmap_w) {
  extern __shared__ uint8_t rt_smem_raw[];
  const uint32_t raw = ptx::smem_u32(rt_smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = rt_smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + RT_STAGES * RT_STAGE_BYTES;
  auto bar = [bar0](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + RT_STAGES * RT_STAGE_BYTES + 8 * RT_NBAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const int csize = p.E / RT_N;
  const int t0 = static_cast<int>(ptx::cluster_id_x()) * RT_M;
  const int e0 = rank * RT_N;
  const int NS = p.H / RT_K;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RT_STAGES; ++s) {
      ptx::mbar_init(bar(RT_BAR_FULL + s), 1);
      ptx::mbar_init(bar(RT_BAR_EMPTY + s), 1);
    }
    ptx::mbar_init(bar(RT_BAR_D), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), RT_N);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    // ------------------------------------------------ TMA: x rows t0.. and Wr rows e0.., K slice ks
    int issued = 0;
    for (int ks = 0; ks < NS; ++ks, ++issued) {
      const int s = ks % RT_STAGES, r = ks / RT_STAGES;
      if (r > 0 && !rt_wait(bar(RT_BAR_EMPTY + s), (r - 1) & 1, p)) break;
      const uint32_t dst = sbase + s * RT_STAGE_BYTES;
      ptx::mbar_arrive_expect_tx_elect(bar(RT_BAR_FULL + s), RT_STAGE_BYTES);
      ptx::tma_load_2d_elect(dst, &tmap_x, ks * RT_K, t0, bar(RT_BAR_FULL + s));
      ptx::tma_load_2d_elect(dst + RT_A_BYTES, &tmap_w, ks * RT_K, e0, bar(RT_BAR_FULL + s));
    }
    // every copy issued has landed before the CTA goes on (at once unless a wait gave up)
    if (lane == 0)
      for (int t = issued > RT_STAGES ? issued - RT_STAGES : 0; t < issued; ++t)
        rt_drain(bar(RT_BAR_FULL + t % RT_STAGES), (t / RT_STAGES) & 1);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issue: D[token, expert] += x Wr^T
    const uint32_t idesc = ptx::idesc_bf16_f32(RT_M, RT_N);
    int ks = 0;
    for (; ks < NS; ++ks) {
      const int s = ks % RT_STAGES, r = ks / RT_STAGES;
      if (!rt_wait(bar(RT_BAR_FULL + s), r & 1, p)) break;
      ptx::tc_fence_after();
      const uint32_t a = sbase + s * RT_STAGE_BYTES;
      ptx::mma_group_ss_elect(tmem, ptx::smem_desc_sw128(a), ptx::smem_desc_sw128(a + RT_A_BYTES), idesc,
                              ks != 0 ? 1u : 0u);
      ptx::mma_commit_elect(bar(RT_BAR_EMPTY + s));
    }
    ptx::mma_commit_elect(bar(RT_BAR_D));  // also after an early stop: the epilogue's wait ends
  } else if (warp >= 4) {
    // ------------------------------------------------ accumulator -> logits, one token per thread
    const int q = warp - 4;
    const bool ok = rt_wait(bar(RT_BAR_D), 0, p);
    if (!ok && lane == 0) rt_drain(bar(RT_BAR_D), 0);  // the MMAs in flight end before TMEM is released
    __syncwarp();
    ptx::tc_fence_after();
    uint32_t v[2][32];
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    ptx::tmem_ld_32x32b_x32(taddr, v[0]);
    ptx::tmem_ld_32x32b_x32(taddr + 32, v[1]);
    ptx::tmem_wait_ld();
    const int t = t0 + 32 * q + lane;
    if (ok && t < p.T) {
      float4* dst = reinterpret_cast<float4*>(p.logits + static_cast<size_t>(t) * p.E + e0);
#pragma unroll
      for (int c = 0; c < RT_N / 4; ++c)
        dst[c] = make_float4(__uint_as_float(v[c / 8][(4 * c) % 32]), __uint_as_float(v[c / 8][(4 * c + 1) % 32]),
                             __uint_as_float(v[c / 8][(4 * c + 2) % 32]), __uint_as_float(v[c / 8][(4 * c + 3) % 32]));
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, RT_N);
  }
  // every logit of the block, from every CTA of the cluster, is written and visible
  ptx::cluster_sync();

  // ------------------------------------------------ top-k of this CTA's share of the block's tokens
  const int per = RT_M / csize;
  for (int i = warp; i < per; i += RT_THREADS / 32) {
    const int t = t0 + rank * per + i;
    if (t >= p.T) break;
    int id;
    float w;
    route_dev::warp_topk_any<true>(p.logits + static_cast<size_t>(t) * p.E, p.E, p.k, lane, &id, &w);
    if (lane < p.k) {
      p.ids[static_cast<size_t>(t) * p.k + lane] = id;
      p.w[static_cast<size_t>(t) * p.k + lane] = w;
    }
  }
}

namespace {

// A 2D bf16 tensor [rows, cols] (row-major) as 128-byte swizzled boxes of box_rows x 64.
bool encode_bf16_2d(CUtensorMap* map, const uint16_t* base, int rows, int cols, int box_rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {RT_K, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

unsigned long long wait_limit_ns();

cudaError_t launch_router(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, float* logits,
                          int32_t* ids, float* w, cudaStream_t s) {
  if (H % RT_K != 0 || E % RT_N != 0 || E / RT_N > 8) return cudaErrorInvalidValue;
  RouterParams prm;
  prm.logits = logits;
  prm.ids = ids;
  prm.w = w;
  prm.err = device_error_ptr();
  const unsigned long long ns = wait_limit_ns();
  prm.wait_cycles = ns > (~0ull) / 3 ? ~0ull : ns * 21 / 10;
  prm.sleep_ns = ns < 20000ull ? static_cast<uint32_t>(ns > 0 ? ns : 1) : 20000u;
  prm.T = T;
  prm.H = H;
  prm.E = E;
  prm.k = k;
  CUtensorMap tx, tw;
  memset(&tx, 0, sizeof(tx));
  memset(&tw, 0, sizeof(tw));
  if (!encode_bf16_2d(&tx, x, T, H, RT_M) || !encode_bf16_2d(&tw, w_router, E, H, RT_N))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(router_kernel), RT_SMEM);
  if (e != cudaSuccess) return e;
  const int csize = E / RT_N;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize * ((T + RT_M - 1) / RT_M));
  cfg.blockDim = dim3(RT_THREADS);
  cfg.dynamicSmemBytes = RT_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, router_kernel, prm, tx, tw);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
