// GPU-resident routing for the W4 MoE layer: router top-k with renormalised
// softmax weights, per-expert histogram, exclusive prefix scan, stable scatter
// (a permutation of the assignments grouped by expert) and the tile block map.
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details, Model
// bullet (8 of 256 experts plus one shared expert) and Prefill optimizations
// bullet (routing histogram, prefix scan, scatter and block map stay on the GPU
// in one submission with no CPU synchronisation).  Here that is one CUDA stream
// with no host sync: the block map and its length are produced on the device
// and consumed on the device by the grouped GEMM.
//
// Kernels:
//   route_small_kernel   one CTA does everything (T*k <= 1024; decode)
//   route_topk_kernel    warp-per-token top-k + per-chunk expert counts
//   route_scan_kernel    one CTA: counts, offsets, per-chunk bases, block map
//   route_scatter_kernel per chunk: stable ranks with warp match, no atomics
#include "moe_common.cuh"
#include "moe_route_dev.cuh"

namespace moe {

using namespace route_dev;

// --------------------------------------------------------------------------
// Single-CTA routing for small T*k (decode): everything in one launch.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) route_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int bn, int32_t* __restrict__ topk_ids,
    float* __restrict__ topk_w, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm, int32_t* __restrict__ block_map,
    int32_t* __restrict__ num_blocks) {
  extern __shared__ int smem_i[];
  int* s_cnt = smem_i;                    // [E]
  int* s_wc = smem_i + E;                 // [32][E] per-warp counts
  __shared__ int s_ids[1024];
  __shared__ uint64_t s_scan[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int A = T * k;

  for (int i = threadIdx.x; i < 33 * E; i += blockDim.x) smem_i[i] = 0;
  for (int t = warp; t < T; t += 32) {
    int id;
    float w;
    warp_topk_any(logits + static_cast<size_t>(t) * E, E, k, lane, &id, &w);
    if (lane < k) {
      topk_ids[t * k + lane] = id;
      topk_w[t * k + lane] = w;
      s_ids[t * k + lane] = id;
    }
  }
  __syncthreads();
  // stable ranks: assignment a = threadIdx.x (A <= 1024, one round)
  const int a = threadIdx.x;
  const bool valid = a < A;
  const int e = valid ? s_ids[a] : -1;
  const unsigned mask = __match_any_sync(FULL, e);
  const int rank_w = __popc(mask & ((1u << lane) - 1u));
  if (valid && lane == __ffs(mask) - 1) s_wc[warp * E + e] = __popc(mask);
  __syncthreads();
  // per-expert totals, then offsets and tile starts
  uint64_t mine = 0;
  int cnt = 0;
  if (threadIdx.x < E) {
    for (int w = 0; w < 32; ++w) cnt += s_wc[w * E + threadIdx.x];
    mine = (static_cast<uint64_t>(cnt) << 32) | static_cast<uint32_t>(ceil_div(cnt, bn));
  }
  uint64_t total;
  uint64_t ex = block_exclusive_scan(mine, s_scan, &total);
  const int off = static_cast<int>(ex >> 32), tile0 = static_cast<int>(ex & 0xffffffffu);
  const int ntiles = static_cast<int>(total & 0xffffffffu);
  if (threadIdx.x < E) {
    counts[threadIdx.x] = cnt;
    offsets[threadIdx.x] = off;
    s_cnt[threadIdx.x] = off;
    emit_expert_tiles(block_map, tile0, threadIdx.x, off, cnt, bn);
  }
  if (threadIdx.x == 0) {
    offsets[E] = A;
    num_blocks[0] = ntiles + ceil_div(T, bn);
  }
  for (int i = threadIdx.x, r = threadIdx.x * bn; r < T; i += blockDim.x, r += blockDim.x * bn) {
    int32_t* p = block_map + 3 * (ntiles + i);
    p[0] = E;
    p[1] = A + r;
    p[2] = min(bn, T - r);
  }
  __syncthreads();
  if (valid) {
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_wc[w * E + e];
    int pos = s_cnt[e] + before + rank_w;
    perm[pos] = a;
    inv_perm[a] = pos;
  }
}

// --------------------------------------------------------------------------
// Multi-CTA routing.
// --------------------------------------------------------------------------
// Kernel 1: chunk c = tokens [c*tc, (c+1)*tc); one warp per token; per-chunk
// expert counts go to cc[c][e] (chunk-major).
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                         int k, int tc, int32_t* __restrict__ topk_ids,
                                                         float* __restrict__ topk_w, int32_t* __restrict__ cc) {
  extern __shared__ int s_hist[];  // [E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int t0 = c * tc, t1 = min(T, t0 + tc);
  for (int t = t0 + warp; t < t1; t += 8) {
    int id;
    float w;
    warp_topk_any(logits + static_cast<size_t>(t) * E, E, k, lane, &id, &w);
    if (lane < k) {
      topk_ids[static_cast<size_t>(t) * k + lane] = id;
      topk_w[static_cast<size_t>(t) * k + lane] = w;
      atomicAdd(&s_hist[id], 1);  // integer counts: order-independent
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) cc[static_cast<size_t>(c) * E + i] = s_hist[i];
}

// Kernel 2 (one CTA, 1024 threads): per-expert totals over chunks, exclusive
// scan over experts, the absolute start of every (chunk, expert) run written
// back into cc, and the block map.
__global__ void __launch_bounds__(1024) route_scan_kernel(int T, int E, int k, int bn, int nch,
                                                          int32_t* __restrict__ cc, int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ block_map,
                                                          int32_t* __restrict__ num_blocks) {
  __shared__ int s_part[1024];
  __shared__ int s_off[1024];
  __shared__ uint64_t s_scan[33];
  int er = 1;
  while (er < E) er <<= 1;
  const int parts = 1024 / er;
  const int e = threadIdx.x % er, part = threadIdx.x / er;
  const int cpp = ceil_div(nch, parts);
  const int c0 = min(nch, part * cpp), c1 = min(nch, c0 + cpp);
  int sum = 0;
  if (e < E) {
    int c = c0;
    for (; c + 16 <= c1; c += 16) {  // 16 independent loads in flight
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = cc[static_cast<size_t>(c + i) * E + e];
#pragma unroll
      for (int i = 0; i < 16; ++i) sum += v[i];
    }
    for (; c < c1; ++c) sum += cc[static_cast<size_t>(c) * E + e];
  }
  s_part[threadIdx.x] = sum;
  __syncthreads();
  uint64_t mine = 0;
  int cnt = 0;
  if (threadIdx.x < E) {
    for (int p = 0; p < parts; ++p) {
      int v = s_part[p * er + threadIdx.x];
      s_part[p * er + threadIdx.x] = cnt;
      cnt += v;
    }
    mine = (static_cast<uint64_t>(cnt) << 32) | static_cast<uint32_t>(ceil_div(cnt, bn));
  }
  __syncthreads();
  uint64_t total;
  uint64_t ex = block_exclusive_scan(mine, s_scan, &total);
  const int A = T * k;
  const int ntiles = static_cast<int>(total & 0xffffffffu);
  if (threadIdx.x < E) {
    const int off = static_cast<int>(ex >> 32), tile0 = static_cast<int>(ex & 0xffffffffu);
    counts[threadIdx.x] = cnt;
    offsets[threadIdx.x] = off;
    s_off[threadIdx.x] = off;
    emit_expert_tiles(block_map, tile0, threadIdx.x, off, cnt, bn);
  }
  if (threadIdx.x == 0) {
    offsets[E] = A;
    num_blocks[0] = ntiles + ceil_div(T, bn);
  }
  for (int i = threadIdx.x, r = threadIdx.x * bn; r < T; i += blockDim.x, r += blockDim.x * bn) {
    int32_t* p = block_map + 3 * (ntiles + i);
    p[0] = E;
    p[1] = A + r;
    p[2] = min(bn, T - r);
  }
  __syncthreads();
  if (e < E) {
    int run = s_off[e] + s_part[part * er + e];
    int c = c0;
    for (; c + 16 <= c1; c += 16) {
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = cc[static_cast<size_t>(c + i) * E + e];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        cc[static_cast<size_t>(c + i) * E + e] = run;
        run += v[i];
      }
    }
    for (; c < c1; ++c) {
      int32_t* p = cc + static_cast<size_t>(c) * E + e;
      int v = *p;
      *p = run;
      run += v;
    }
  }
}

// Kernel 3: per chunk, the stable rank of each assignment among the chunk's
// assignments of the same expert, computed without atomics: __match_any_sync
// groups equal experts within a warp, each group's leader publishes its size
// per (warp, expert), and a thread adds the sizes of the earlier warps.
__global__ void __launch_bounds__(256) route_scatter_kernel(const int32_t* __restrict__ topk_ids, int T, int E,
                                                            int k, int tc, const int32_t* __restrict__ cc,
                                                            int32_t* __restrict__ perm,
                                                            int32_t* __restrict__ inv_perm, int* err) {
  extern __shared__ int smem_i[];
  int* s_base = smem_i;      // [E] next free position of each expert
  int* s_wc = smem_i + E;    // [8][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const int A = T * k;
  const int a0 = c * tc * k, a1 = min(A, a0 + tc * k);
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_base[i] = cc[static_cast<size_t>(c) * E + i];
  for (int ab = a0; ab < a1; ab += 256) {
    for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) s_wc[i] = 0;
    __syncthreads();
    const int a = ab + threadIdx.x;
    int e = a < a1 ? topk_ids[a] : -1;
    if (e >= E || e < -1) {
      set_device_error(err, MOE_DEV_BAD_INDEX);
      e = -1;
    }
    const unsigned mask = __match_any_sync(FULL, e);
    const int rank_w = __popc(mask & ((1u << lane) - 1u));
    if (e >= 0 && lane == __ffs(mask) - 1) s_wc[warp * E + e] = __popc(mask);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_wc[w * E + e];
      const int pos = s_base[e] + before + rank_w;
      perm[pos] = a;
      inv_perm[a] = pos;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
      int add = 0;
      for (int w = 0; w < 8; ++w) add += s_wc[w * E + i];
      s_base[i] += add;
    }
    __syncthreads();
  }
}

// --------------------------------------------------------------------------
// host side
// --------------------------------------------------------------------------
int route_chunk_tokens(int T) {
  int tc = 8;
  while (ceil_div(T, tc) > 256) tc <<= 1;
  return tc;
}

bool route_use_small(int T, int k) { return T * k <= 1024; }

size_t route_workspace_bytes(int T, int E, int k) {
  if (route_use_small(T, k)) return 0;
  int tc = route_chunk_tokens(T);
  return static_cast<size_t>(ceil_div(T, tc)) * E * sizeof(int32_t);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int bn, int32_t* ids, float* w,
                         int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* bm,
                         int32_t* nb, void* ws, cudaStream_t s) {
  int* err = device_error_ptr();
  if (route_use_small(T, k)) {
    size_t sm = static_cast<size_t>(33) * E * sizeof(int);
    if (sm > 48 * 1024) {
      cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
    }
    route_small_kernel<<<1, 1024, sm, s>>>(logits, T, E, k, bn, ids, w, counts, offsets, perm, inv_perm, bm, nb);
    note_launches(1);
    return cudaGetLastError();
  }
  const int tc = route_chunk_tokens(T);
  const int nch = ceil_div(T, tc);
  int32_t* cc = static_cast<int32_t*>(ws);
  route_topk_kernel<<<nch, 256, E * sizeof(int), s>>>(logits, T, E, k, tc, ids, w, cc);
  route_scan_kernel<<<1, 1024, 0, s>>>(T, E, k, bn, nch, cc, counts, offsets, bm, nb);
  size_t sm = static_cast<size_t>(9) * E * sizeof(int);
  if (sm > 48 * 1024) {
    cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
  }
  route_scatter_kernel<<<nch, 256, sm, s>>>(ids, T, E, k, tc, cc, perm, inv_perm, err);
  note_launches(3);
  return cudaGetLastError();
}

}  // namespace moe

// --------------------------------------------------------------------------
// moe_route_noalloc: the same routing with its per-chunk counts kept in a
// fixed device array owned by this library, for callers that are not allowed
// to allocate device memory (see include/moe_w4.h).
// --------------------------------------------------------------------------
#include <mutex>

// 256 chunks x 256 experts of int32 counts: every T this library accepts (at
// most 256 chunks) with up to 256 routed experts.  Resident on each device
// that loads the library until the process exits.
static __device__ __align__(256) int32_t moe_route_scratch[256 * 256];

namespace {

constexpr size_t kRouteScratchBytes = sizeof(int32_t) * 256 * 256;

// Device address of moe_route_scratch on the current device, looked up once
// per device (the host-side name is only a stand-in for the device symbol).
void* route_scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, moe_route_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_route_noalloc(const float* logits, int T, int E, int k, int block_n, int32_t* topk_ids,
                                 float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv_perm, int32_t* block_map, int32_t* num_blocks,
                                 moe_stream_t stream) {
  if (T < 1 || T > (1 << 20) || E < 1 || E > 1024 || k < 1 || k > 32 || k > E || block_n < 1 || block_n > 1024)
    return MOE_ERR_SHAPE;
  const void* ptrs[] = {logits, topk_ids, topk_w, counts, offsets, perm, inv_perm, block_map, num_blocks};
  for (const void* q : ptrs)
    if (!q) return MOE_ERR_NULL;
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_ALIGN;
  const size_t need = moe::route_workspace_bytes(T, E, k);
  if (need > kRouteScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = route_scratch_address();
    if (!scratch) return MOE_ERR_CUDA;
  }
  if (!moe::device_error_ptr()) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_route(logits, T, E, k, block_n, topk_ids, topk_w, counts, offsets, perm,
                                          inv_perm, block_map, num_blocks, scratch,
                                          reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

