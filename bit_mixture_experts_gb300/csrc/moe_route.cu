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
//   route_fused_kernel   one CTA per chunk of tokens, one cooperative launch:
//                        top-k and chunk counts | grid barrier | totals, scan,
//                        block map | stable scatter (ranks with warp match)
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
    int32_t* __restrict__ num_blocks, int ids_given) {
  extern __shared__ int smem_i[];
  int* s_cnt = smem_i;                    // [E]
  int* s_wc = smem_i + E;                 // [32][E] per-warp counts
  __shared__ int s_ids[1024];
  __shared__ uint64_t s_scan[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int A = T * k;

  for (int i = threadIdx.x; i < 33 * E; i += blockDim.x) smem_i[i] = 0;
  for (int t = warp; t < T; t += 32) {
    if (ids_given) {  // top-k already chosen (moe_route_x): take the ids
      if (lane < k) s_ids[t * k + lane] = min(max(__ldg(topk_ids + t * k + lane), 0), E - 1);
      continue;
    }
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
// Multi-CTA routing: one cooperative launch of nch CTAs, chunk c = tokens
// [c*tc, (c+1)*tc), 256 threads.
//   1. top-k of the chunk's tokens (one warp per token) and the chunk's
//      per-expert counts cc[c][e] (chunk-major, in the workspace);
//   -  grid barrier (a counter in the workspace; every CTA is resident);
//   2. every CTA sums the counts of all chunks per expert (L2 reads), scans
//      them over the experts (offsets and the first tile of each expert) and
//      takes its own chunk's start in each expert's run; CTA 0 also writes
//      counts, offsets, the block map and its length;
//   3. the stable rank of each of the chunk's assignments among the chunk's
//      assignments of the same expert, without atomics: __match_any_sync
//      groups equal experts within a warp, each group's leader publishes its
//      size per (warp, expert), and a thread adds the sizes of earlier warps.
//   The last CTA to finish returns the counters to zero for the next call.
// --------------------------------------------------------------------------
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(256) route_fused_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                          int tc, int bn, int32_t* topk_ids, float* topk_w,
                                                          int32_t* cc, int* ctr, int32_t* counts, int32_t* offsets,
                                                          int32_t* perm, int32_t* inv_perm, int32_t* block_map,
                                                          int32_t* num_blocks, int cap, int* err,
                                                          unsigned long long wait_cycles, int ids_given) {
  extern __shared__ int smem_i[];
  int* s_hist = smem_i;        // [E] chunk counts, then the chunk's next free row per expert
  int* s_wc = smem_i + E;      // [8][E] per-warp group sizes
  int* s_tot = s_wc + 8 * E;   // [E] totals over all chunks
  __shared__ uint64_t s_scan[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x, nch = gridDim.x;
  const int A = T * k;

  // ---- 1: top-k and the chunk's counts
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int t0 = c * tc, t1 = min(T, t0 + tc);
  for (int t = t0 + warp; t < t1; t += 8) {
    int id;
    float w;
    if (ids_given) {  // top-k already chosen (moe_route_x): take the ids
      id = lane < k ? __ldg(topk_ids + static_cast<size_t>(t) * k + lane) : 0;
      if (id < 0 || id >= E) {
        set_device_error(err, MOE_DEV_BAD_INDEX);
        id = 0;
      }
      if (lane < k) atomicAdd(&s_hist[id], 1);
      continue;
    }
    warp_topk_any(logits + static_cast<size_t>(t) * E, E, k, lane, &id, &w);
    if (lane < k) {
      topk_ids[static_cast<size_t>(t) * k + lane] = id;
      topk_w[static_cast<size_t>(t) * k + lane] = w;
      atomicAdd(&s_hist[id], 1);  // integer counts: order-independent
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) cc[static_cast<size_t>(c) * E + i] = s_hist[i];

  // ---- grid barrier: every chunk's counts are written
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int before_me = atomicAdd(ctr, 1);
    if (before_me < 0 || before_me >= nch) set_device_error(err, MOE_DEV_BAD_WORKSPACE);  // counter not zero at the start
    const long long w0 = clock64();
    while (ld_acquire_gpu(ctr) < nch) {
      if (static_cast<unsigned long long>(clock64() - w0) > wait_cycles) {
        set_device_error(err, MOE_DEV_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
  }
  __syncthreads();

  // ---- 2: totals, this chunk's start per expert, offsets and the block map
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int tot = 0, before = 0;
    int cq = 0;
    for (; cq + 64 <= nch; cq += 64) {  // 64 independent loads in flight
      int v[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = __ldcg(cc + static_cast<size_t>(cq + i) * E + e);
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        tot += v[i];
        before += cq + i < c ? v[i] : 0;
      }
    }
    for (; cq < nch; ++cq) {
      const int v = __ldcg(cc + static_cast<size_t>(cq) * E + e);
      tot += v;
      before += cq < c ? v : 0;
    }
    s_tot[e] = tot;
    s_hist[e] = before;
  }
  // Counts that cannot come from this call (a workspace that was not zero
  // when the call began breaks the barrier and the per-chunk counts): every
  // total must be >= 0 and they must add up to T*k with the tiles fitting in
  // the block map; otherwise nothing below is written and the error is recorded.
  bool bad = false;
  for (int e = threadIdx.x; e < E; e += blockDim.x) bad |= s_tot[e] < 0 || s_hist[e] < 0 || s_hist[e] > s_tot[e];
  bad = __syncthreads_or(bad);
  {
    const int per = ceil_div(E, static_cast<int>(blockDim.x));
    const int e0 = min(E, static_cast<int>(threadIdx.x) * per), e1 = min(E, e0 + per);
    uint64_t loc = 0;
    for (int e = e0; e < e1; ++e)
      loc += (static_cast<uint64_t>(s_tot[e]) << 32) | static_cast<uint32_t>(ceil_div(s_tot[e], bn));
    uint64_t total;
    uint64_t run = block_exclusive_scan(loc, s_scan, &total);
    const int ntiles = static_cast<int>(total & 0xffffffffu);
    bad = bad || static_cast<int>(total >> 32) != A || ntiles + ceil_div(T, bn) > cap;
    if (bad && threadIdx.x == 0) set_device_error(err, MOE_DEV_BAD_WORKSPACE);
    for (int e = e0; e < e1 && !bad; ++e) {
      const int cnt = s_tot[e];
      const int off = static_cast<int>(run >> 32), tile0 = static_cast<int>(run & 0xffffffffu);
      s_hist[e] += off;
      if (c == 0) {
        counts[e] = cnt;
        offsets[e] = off;
        emit_expert_tiles(block_map, tile0, e, off, cnt, bn);
      }
      run += (static_cast<uint64_t>(cnt) << 32) | static_cast<uint32_t>(ceil_div(cnt, bn));
    }
    if (c == 0 && !bad) {
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
    }
  }
  __syncthreads();

  // ---- 3: stable scatter of the chunk's assignments (bad is the same in every thread of the CTA)
  const int a0 = c * tc * k, a1 = bad ? a0 : min(A, a0 + tc * k);
  for (int ab = a0; ab < a1; ab += 256) {
    for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) s_wc[i] = 0;
    __syncthreads();
    const int a = ab + threadIdx.x;
    int e = a < a1 ? __ldcg(topk_ids + a) : -1;
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
      const int pos = s_hist[e] + before + rank_w;
      if (pos >= 0 && pos < A) {
        perm[pos] = a;
        inv_perm[a] = pos;
      } else {
        set_device_error(err, MOE_DEV_BAD_INDEX);
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
      int add = 0;
      for (int w = 0; w < 8; ++w) add += s_wc[w * E + i];
      s_hist[i] += add;
    }
    __syncthreads();
  }

  // ---- the last CTA returns the counters to zero
  if (threadIdx.x == 0 && atomicAdd(ctr + 1, 1) == nch - 1) {
    ctr[0] = 0;
    ctr[1] = 0;
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

// Multi-CTA path: per-chunk counts [nch][E] at the start of the workspace; 4 ints
// of counters (zero between calls) in its last 16 bytes, wherever the counts of
// a call with another T ended, so that a larger earlier call cannot leave counts
// where a smaller later one keeps its counters.
size_t route_workspace_bytes(int T, int E, int k) {
  if (route_use_small(T, k)) return 0;
  int tc = route_chunk_tokens(T);
  return static_cast<size_t>(ceil_div(T, tc)) * E * sizeof(int32_t) + 4 * sizeof(int32_t);
}

unsigned long long wait_limit_ns();

cudaError_t launch_route(const float* logits, int T, int E, int k, int bn, int32_t* ids, float* w,
                         int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* bm,
                         int32_t* nb, void* ws, size_t ws_bytes, cudaStream_t s, int ids_given) {
  int* err = device_error_ptr();
  if (route_use_small(T, k)) {
    size_t sm = static_cast<size_t>(33) * E * sizeof(int);
    if (sm > 48 * 1024) {
      const cudaError_t e0 = ensure_dyn_smem(reinterpret_cast<const void*>(route_small_kernel), sm);
      if (e0 != cudaSuccess) return e0;
    }
    route_small_kernel<<<1, 1024, sm, s>>>(logits, T, E, k, bn, ids, w, counts, offsets, perm, inv_perm, bm, nb,
                                           ids_given);
    note_launches(1);
    return cudaGetLastError();
  }
  const int tc = route_chunk_tokens(T);
  const int nch = ceil_div(T, tc);
  int32_t* cc = static_cast<int32_t*>(ws);
  int* ctr = reinterpret_cast<int*>(static_cast<char*>(ws) + ((ws_bytes - 16) & ~static_cast<size_t>(3)));
  const size_t sm = static_cast<size_t>(10) * E * sizeof(int);
  if (sm > 48 * 1024) {
    cudaError_t e0 = ensure_dyn_smem(reinterpret_cast<const void*>(route_fused_kernel), sm);
    if (e0 != cudaSuccess) return e0;
  }
  const unsigned long long ns = wait_limit_ns();
  const unsigned long long wait_cycles = ns > (~0ull) / 3 ? ~0ull : ns * 21 / 10;
  // cooperative launch: the grid barrier needs every chunk's CTA resident (nch <= 256)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nch);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int cap = moe_block_map_capacity(T, E, k, bn);
  cudaError_t e = cudaLaunchKernelEx(&cfg, route_fused_kernel, logits, T, E, k, tc, bn, ids, w, cc, ctr, counts,
                                     offsets, perm, inv_perm, bm, nb, cap, err, wait_cycles, ids_given);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
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
static __device__ __align__(256) int32_t moe_route_scratch[256 * 256 + 4];

namespace {

constexpr size_t kRouteScratchBytes = sizeof(int32_t) * (256 * 256 + 4);

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

}  // namespace

extern "C" int moe_route_noalloc(const float* logits, int T, int E, int k, int block_n, int32_t* topk_ids,
                                 float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv_perm, int32_t* block_map, int32_t* num_blocks,
                                 moe_stream_t stream) {
  int rc = moe::check_route_shape(T, E, k, block_n);
  if (rc) return rc;
  rc = moe::check_ptrs(logits, topk_ids, topk_w, counts, offsets, perm, inv_perm, block_map, num_blocks);
  if (rc) return rc;
  const size_t need = moe::route_workspace_bytes(T, E, k);
  if (need > kRouteScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = route_scratch_address();
    if (!scratch) return MOE_ERR_CUDA;
    // The grid barrier's counters (the array's last 16 bytes) are cleared before every multi-CTA
    // call, in stream order: a call that overlapped another one on the GPU, or one whose barrier
    // gave up, cannot leave them counted for the calls after it.
    if (cudaMemsetAsync(static_cast<char*>(scratch) + kRouteScratchBytes - 16, 0, 16,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (!moe::device_error_ptr()) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_route(logits, T, E, k, block_n, topk_ids, topk_w, counts, offsets, perm,
                                          inv_perm, block_map, num_blocks, scratch, kRouteScratchBytes,
                                          reinterpret_cast<cudaStream_t>(stream), 0);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

