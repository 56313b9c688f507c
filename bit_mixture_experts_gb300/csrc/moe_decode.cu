// Fused decode forward: the whole layer for at most DEC_MAXT tokens in one
// persistent launch -- routing, gate/up GEMV + SwiGLU, down GEMV and the
// weighted gather-combine.
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details: the
// decode step is a small batch through 8 routed experts plus the shared
// expert, every weight byte is read once per step, and the routing stays on
// the GPU with no host synchronisation.  At batch 1 the four kernels of the
// general path (route, gate/up, down, combine) each last only a few
// microseconds, so their launch and dependency latencies dominate; here they
// become phases of one kernel whose CTAs are all resident (cooperative
// launch) and hand work to each other through counters in global memory.
//
// Phases, in every CTA (256 threads, GV_CTAS_PER_SM per SM):
//   R  routing, recomputed by every CTA in shared memory from the logits with
//      the same device code as moe_route (top-k and weights, counts, offsets,
//      stable permutation, block map); CTA 0 also writes moe_route's outputs.
//   G  gate/up work items (tile, 16 features), exactly as the GEMV kernel
//      (the first down item's weights are already streaming during the last).
//   -  grid barrier: every h value is written.
//   D  down work items (tile, 32 channels); h is read through L2 only.
//   -  grid barrier: every y value is written.
//   C  the gather-combine, one warp per (token, 32 channels):
//      out = bf16(sum_j topk_w[t, j] * y[row(t, j)] + y[shared row]), FP32 in
//      the same fixed order as moe_combine.
//   The last CTA to finish resets the barrier counters for the next call.
// The grid barriers are counters in global memory (one fence and one atomic
// per CTA); they rely on every CTA being resident, which the cooperative
// launch guarantees.  Each wait is bounded nonetheless; on expiry it records
// MOE_DEV_TIMEOUT and goes on.  (A first version signalled per work item --
// a counter per tile for h, per token and 32 channels for y -- and spent
// most of its time in the fences those signals need.)
#include "moe_common.cuh"
#include "moe_gemv_dev.cuh"
#include "moe_ptx.cuh"
#include "moe_route_dev.cuh"

namespace moe {

using namespace gemv_dev;

namespace {

constexpr int DEC_MAXT = 8;                         // tokens per call
constexpr int DEC_MAXA = DEC_MAXT * 32;             // assignments (k <= 32)
constexpr int DEC_MAXTILES = DEC_MAXA + DEC_MAXT;   // routed tiles (>= 1 row each) + shared tiles

struct DecParams {
  const uint16_t* x;
  const float* logits;
  const uint8_t* w13;
  const uint8_t* w2;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* block_map;
  int32_t* num_blocks;
  uint16_t* h;
  uint16_t* y;
  uint16_t* out;
  int* ws;  // grid barrier counters: [0] h written, [1] y written, [2] CTAs done
  int* err;
  unsigned long long wait_cycles;
  int T, H, F, E, k, bn;
  int G;  // K groups per thread (max over the two matrices)
};

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Small-batch routing (at most 64 assignments, T <= bn so that every expert's
// rows form one tile), by warps 0 and 1, thread a = assignment a: its
// permuted row is its rank among the keys (expert, assignment) -- by expert,
// then in assignment order, as moe_route's stable scatter -- and a tile
// starts wherever the expert changes along the sorted rows (found by warp 0);
// the shared expert's T rows follow as one tile.  s_ok receives the number
// of routed tiles.
__device__ __noinline__ void route_small_batch(const int* s_ids, int* s_inv, int* s_tok, int* s_sorted,
                                               int (*s_tile)[3], int* s_ok, int A, int T, int E, int k) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int a = 32 * warp + lane;
  if (a < A) {
    const int e = s_ids[a];
    const int key = e * 64 + a;
    int r = 0;
    for (int a2 = 0; a2 < A; ++a2) r += s_ids[a2] * 64 + a2 < key;
    s_inv[a] = r;
    s_tok[r] = a / k;
    s_sorted[r] = e;
  }
  ptx::named_bar_sync(1, 64);
  if (warp != 0) return;
  // a run of one expert starts at sorted row r when r == 0 or the expert changes there
  unsigned long long starts = 0;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int r = lane + 32 * q;
    const bool st = r < A && (r == 0 || s_sorted[r] != s_sorted[r - 1]);
    starts |= static_cast<unsigned long long>(__ballot_sync(0xffffffffu, st)) << (32 * q);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int r = lane + 32 * q;
    if ((starts >> r) & 1ull) {
      const int ti = __popcll(starts & ((1ull << r) - 1ull));
      const unsigned long long later = r == 63 ? 0ull : starts & ~((2ull << r) - 1ull);
      s_tile[ti][0] = s_sorted[r];
      s_tile[ti][1] = r;
      s_tile[ti][2] = (later ? __ffsll(static_cast<long long>(later)) - 1 : A) - r;
    }
  }
  if (lane == 0) {
    const int n = __popcll(starts);
    *s_ok = n;
    s_tile[n][0] = E;
    s_tile[n][1] = A;
    s_tile[n][2] = T;
  }
  if (lane < T) s_tok[A + lane] = lane;
}

// General routing in shared memory, by the whole CTA: per-expert counts,
// their exclusive scan (offsets and first tiles), the stable permutation and
// the block map, as moe_route computes them.  s_ok receives the number of
// routed tiles.
__device__ __noinline__ void route_general(const int* s_ids, int* s_inv, int* s_tok, int (*s_tile)[3], int* s_cnt,
                                           int* s_off, int* s_tile0, uint64_t* s_scan, int* s_ok, int A, int T,
                                           int E, int k, int bn) {
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += GV_THREADS) s_cnt[e] = 0;
  __syncthreads();
  for (int a = tid; a < A; a += GV_THREADS) atomicAdd(&s_cnt[s_ids[a]], 1);  // integer counts
  __syncthreads();
  {
    // offsets and first tile of every expert: exclusive scan of (count, tiles) in expert order
    const int per = ceil_div(E, GV_THREADS);
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    uint64_t loc = 0;
    for (int e = e0; e < e1; ++e) {
      const int c = s_cnt[e];
      loc += (static_cast<uint64_t>(c) << 32) | static_cast<uint32_t>(ceil_div(c, bn));
    }
    uint64_t total;
    uint64_t run = route_dev::block_exclusive_scan(loc, s_scan, &total);
    for (int e = e0; e < e1; ++e) {
      const int c = s_cnt[e];
      s_off[e] = static_cast<int>(run >> 32);
      s_tile0[e] = static_cast<int>(run & 0xffffffffu);
      run += (static_cast<uint64_t>(c) << 32) | static_cast<uint32_t>(ceil_div(c, bn));
    }
    if (tid == 0) *s_ok = static_cast<int>(total & 0xffffffffu);  // routed tiles
  }
  __syncthreads();
  const int ntr = *s_ok;
  // stable permutation: by expert, then by assignment index
  for (int a = tid; a < A; a += GV_THREADS) {
    const int e = s_ids[a];
    int r = 0;
    for (int a2 = 0; a2 < a; ++a2) r += s_ids[a2] == e;
    const int row = s_off[e] + r;
    s_inv[a] = row;
    s_tok[row] = a / k;
  }
  for (int t = tid; t < T; t += GV_THREADS) s_tok[A + t] = t;
  for (int e = tid; e < E; e += GV_THREADS) {
    const int c = s_cnt[e];
    for (int i = 0, r = 0; r < c; ++i, r += bn) {
      s_tile[s_tile0[e] + i][0] = e;
      s_tile[s_tile0[e] + i][1] = s_off[e] + r;
      s_tile[s_tile0[e] + i][2] = min(bn, c - r);
    }
  }
  for (int i = tid, r = tid * bn; r < T; i += GV_THREADS, r += GV_THREADS * bn) {
    s_tile[ntr + i][0] = E;
    s_tile[ntr + i][1] = A + r;
    s_tile[ntr + i][2] = min(bn, T - r);
  }
  __syncthreads();
}

}  // namespace

__global__ void __launch_bounds__(GV_THREADS, GV_CTAS_PER_SM) decode_kernel(const DecParams p) {
  __shared__ int s_ids[DEC_MAXA];
  __shared__ float s_w[DEC_MAXA];
  __shared__ int s_inv[DEC_MAXA];                // assignment -> permuted row
  __shared__ int s_tok[DEC_MAXA + DEC_MAXT];     // permuted row -> token
  __shared__ int s_tile[DEC_MAXTILES][3];        // (expert, first row, rows)
  __shared__ uint64_t s_scan[33];
  __shared__ int s_sorted[64];                   // small-batch path: expert of each permuted row
  __shared__ int s_ok;
  extern __shared__ uint4 dec_smem[];
  const int T = p.T, E = p.E, k = p.k, bn = p.bn, H = p.H, F = p.F;
  const int A = T * k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // dynamic shared memory: weight slots of two items, (scale, bias) slots, partial sums, per-expert tables
  const int G = p.G;
  const int slot_q = 2 * G * GV_THREADS, slot_sb = G * GV_THREADS;
  uint4* swq0 = dec_smem;
  uint32_t* swsb0 = reinterpret_cast<uint32_t*>(dec_smem + 2 * slot_q);
  float* spart0 = reinterpret_cast<float*>(swsb0 + 2 * slot_sb);
  int* s_cnt = reinterpret_cast<int*>(spart0 + 2 * GV_WARPS * GV_MAXN * 32);  // [E]
  int* s_off = s_cnt + E;                                                     // [E]
  int* s_tile0 = s_off + E;                                                   // [E]
  int* ws_bar = p.ws;  // [0] h written, [1] y written, [2] CTAs done

  // ---------------------------------------------------------------- R: routing
  if (warp < T) {
    int id;
    float w;
    route_dev::warp_topk_any(p.logits + static_cast<size_t>(warp) * E, E, k, lane, &id, &w);
    if (lane < k) {
      s_ids[warp * k + lane] = id;
      s_w[warp * k + lane] = w;
    }
  }
  // Small batches (at most 64 assignments, every expert's rows in one tile):
  // two warps rank the assignments and read the tiles off the sorted rows,
  // with no pass over all E experts (the same result as the general path).
  if (A <= 64 && T <= bn) {
    __syncthreads();  // s_ids
    if (warp < 2) route_small_batch(s_ids, s_inv, s_tok, s_sorted, s_tile, &s_ok, A, T, E, k);
    if (blockIdx.x == 0) {  // counts and offsets of every expert, for moe_route's outputs
      for (int e = tid; e < E; e += GV_THREADS) {
        int c = 0, o = 0;
        for (int a = 0; a < A; ++a) {
          c += s_ids[a] == e;
          o += s_ids[a] < e;
        }
        s_cnt[e] = c;
        s_off[e] = o;
      }
    }
    __syncthreads();
  } else {
    route_general(s_ids, s_inv, s_tok, s_tile, s_cnt, s_off, s_tile0, s_scan, &s_ok, A, T, E, k, bn);
  }
  const int ntr = s_ok;
  const int nt = ntr + ceil_div(T, bn);
  if (blockIdx.x == 0) {
    // the outputs of moe_route for the same logits
    for (int a = tid; a < A; a += GV_THREADS) {
      p.topk_ids[a] = s_ids[a];
      p.topk_w[a] = s_w[a];
      p.inv_perm[a] = s_inv[a];
      p.perm[s_inv[a]] = a;
    }
    for (int e = tid; e < E; e += GV_THREADS) {
      p.counts[e] = s_cnt[e];
      p.offsets[e] = s_off[e];
    }
    for (int i = tid; i < nt; i += GV_THREADS) {
      p.block_map[3 * i] = s_tile[i][0];
      p.block_map[3 * i + 1] = s_tile[i][1];
      p.block_map[3 * i + 2] = s_tile[i][2];
    }
    if (tid == 0) {
      p.offsets[E] = A;
      p.num_blocks[0] = nt;
    }
  }

  // ---------------------------------------------------------------- G, D: work items
  const int IPT0 = F / 16, IPT1 = H / 32;
  const int MT0 = (2 * F) / TC_M, MT1 = H / TC_M;
  const int KT0 = H / KG, KT1 = F / KG;
  const int nG = nt * IPT0, nD = nt * IPT1;
  // this CTA's items: its gate/up items, then its down items
  const int myG = blockIdx.x < nG ? ceil_div(nG - blockIdx.x, gridDim.x) : 0;
  const int myD = blockIdx.x < nD ? ceil_div(nD - blockIdx.x, gridDim.x) : 0;

  // copies of item q of this CTA (this thread's weight row) into slot buffer b; one commit group
  auto issue = [&](int q, int b) {
    if (q < myG + myD) {
      const bool down = q >= myG;
      const int u = blockIdx.x + (down ? q - myG : q) * gridDim.x;
      const int ipt = down ? IPT1 : IPT0;
      const int tile = u / ipt, j = u - tile * ipt;
      int mt, L;
      if (down) item_row<1>(j, lane, &mt, &L);
      else item_row<0>(j, lane, &mt, &L);
      const int KT = down ? KT1 : KT0;
      const uint8_t* wrow = (down ? p.w2 : p.w13) +
                            (static_cast<size_t>(s_tile[tile][0]) * (down ? MT1 : MT0) + mt) * KT *
                                static_cast<size_t>(W_BLOCK);
      uint4* qd = swq0 + b * slot_q + tid;
      uint32_t* sd = swsb0 + b * slot_sb + tid;
#pragma unroll 1
      for (int i = 0; i < G; ++i) {
        const int kg = warp + GV_WARPS * i;
        if (kg >= KT) break;
        const uint8_t* blk = wrow + static_cast<size_t>(kg) * W_BLOCK;
        ptx::cp_async_16(ptx::smem_u32(qd + (2 * i) * GV_THREADS), blk + L * 16);
        ptx::cp_async_16(ptx::smem_u32(qd + (2 * i + 1) * GV_THREADS), blk + 2048 + L * 16);
        ptx::cp_async_4(ptx::smem_u32(sd + i * GV_THREADS), blk + W_PACKED + L * 4);
      }
    }
    ptx::cp_async_commit();
  };

  // every CTA has passed the barrier once all have arrived; bounded, records a timeout
  auto grid_barrier = [&](int* bar) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();  // this CTA's h / y values before its arrival
      const int before_me = atomicAdd(bar, 1);
      if (before_me < 0 || before_me >= static_cast<int>(gridDim.x))
        set_device_error(p.err, MOE_DEV_BAD_WORKSPACE);  // the workspace was not zero at the start
      const long long t0 = clock64();
      while (ld_acquire(bar) < static_cast<int>(gridDim.x)) {
        if (static_cast<unsigned long long>(clock64() - t0) > p.wait_cycles) {
          set_device_error(p.err, MOE_DEV_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    __syncthreads();
  };

  issue(0, 0);
  for (int q = 0; q < myG + myD; ++q) {
    const int buf = q & 1;
    if (q == myG) grid_barrier(ws_bar);  // all of h is written before any down item reads it
    issue(q + 1, buf ^ 1);  // the next item's weights stream during this one
    const bool down = q >= myG;
    const int u = blockIdx.x + (down ? q - myG : q) * gridDim.x;
    const int ipt = down ? IPT1 : IPT0;
    const int tile = u / ipt, j = u - tile * ipt;
    const int row0 = s_tile[tile][1], nrow = s_tile[tile][2];
    // activation row of this lane's token column (gate/up: x of the row's token; down: the row of h);
    // columns past the tile read the tile's first row
    const int r = row0 + ((lane >> 2) < nrow ? (lane >> 2) : 0);
    const uint32_t xo = down ? static_cast<uint32_t>(r) * static_cast<uint32_t>(F)
                             : static_cast<uint32_t>(s_tok[r]) * static_cast<uint32_t>(H);
    float d[2][4] = {};
    ptx::cp_async_wait<1>();  // this thread's copies of item q have landed
    __syncwarp();             // ... and those of the warp's other lanes, whose rows this lane reads
    const uint4* sw = swq0 + buf * slot_q + 32 * warp;
    const uint32_t* ssbw = swsb0 + buf * slot_sb + 32 * warp;
    if (down) item_mma<true>(sw, ssbw, p.h, xo, warp, lane, KT1, G, d);
    else item_mma<false>(sw, ssbw, p.x, xo, warp, lane, KT0, G, d);

    // reduce the warps' partial sums (fixed order) and write the item's outputs
    float* spart = spart0 + buf * (GV_WARPS * GV_MAXN * 32);
    store_partials(spart, d, warp, lane, nrow);
    __syncthreads();
    if (!down) {
      if (tid < nrow * 16) {
        const int n = tid >> 4, fi = tid & 15;
        float gs = 0.f, us = 0.f;
        for (int w = 0; w < GV_WARPS; ++w) {
          gs += spart[(w * GV_MAXN + n) * 32 + fi];
          us += spart[(w * GV_MAXN + n) * 32 + 16 + fi];
        }
        p.h[static_cast<size_t>(row0 + n) * F + 16 * j + fi] = float_to_bf16_bits(silu(gs) * us);
      }
    } else if (warp < nrow) {
      float yv = 0.f;
      for (int w = 0; w < GV_WARPS; ++w) yv += spart[(w * GV_MAXN + warp) * 32 + lane];
      p.y[static_cast<size_t>(row0 + warp) * H + 32 * j + lane] = float_to_bf16_bits(yv);
    }
  }
  if (myD == 0) grid_barrier(ws_bar);  // CTAs without down items still take part in the first barrier
  ptx::cp_async_wait_all();
  grid_barrier(ws_bar + 1);  // all of y is written

  // ---------------------------------------------------------------- C: combine, one warp per (token, 32 channels)
  for (int c = blockIdx.x * GV_WARPS + warp; c < T * IPT1; c += gridDim.x * GV_WARPS) {
    const int t = c / IPT1, jb = c - t * IPT1;
    // rows loaded eight at a time before they are summed (one L2 round trip per batch)
    const uint16_t ys = __ldcg(p.y + static_cast<size_t>(A + t) * H + 32 * jb + lane);
    float o = 0.f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint16_t yb[8];
#pragma unroll
      for (int b = 0; b < 8; ++b)
        yb[b] = j0 + b < k ? __ldcg(p.y + static_cast<size_t>(s_inv[t * k + j0 + b]) * H + 32 * jb + lane) : 0;
#pragma unroll
      for (int b = 0; b < 8; ++b)
        if (j0 + b < k) o = fmaf(s_w[t * k + j0 + b], bf16_bits_to_float(yb[b]), o);
    }
    o = fmaf(1.0f, bf16_bits_to_float(ys), o);
    p.out[static_cast<size_t>(t) * H + 32 * jb + lane] = float_to_bf16_bits(o);
  }

  // ---------------------------------------------------------------- the last CTA resets the counters
  __syncthreads();
  if (tid == 0) {
    if (atomicAdd(ws_bar + 2, 1) == static_cast<int>(gridDim.x) - 1) {
      ws_bar[0] = 0;
      ws_bar[1] = 0;
      ws_bar[2] = 0;
    }
  }
}

int decode_max_tokens() { return DEC_MAXT; }

size_t decode_workspace_bytes(int, int) { return 4 * sizeof(int); }

static size_t decode_smem_bytes(int G, int E) {
  return 2 * static_cast<size_t>(G) * GV_THREADS * (2 * 16 + 4) +
         2 * static_cast<size_t>(GV_WARPS) * GV_MAXN * 32 * sizeof(float) + 3 * static_cast<size_t>(E) * sizeof(int);
}

cudaError_t launch_decode(const uint16_t* x, const float* logits, const void* w13, const void* w2, int T, int H, int F,
                          int E, int k, int bn, int32_t* topk_ids, float* topk_w, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* inv_perm, int32_t* block_map, int32_t* num_blocks, uint16_t* h,
                          uint16_t* y, uint16_t* out, void* ws, unsigned long long wait_ns, int num_sms,
                          cudaStream_t s) {
  if (T > DEC_MAXT || k > 32 || bn > GV_MAXN) return cudaErrorInvalidValue;
  DecParams prm;
  prm.x = x;
  prm.logits = logits;
  prm.w13 = static_cast<const uint8_t*>(w13);
  prm.w2 = static_cast<const uint8_t*>(w2);
  prm.topk_ids = topk_ids;
  prm.topk_w = topk_w;
  prm.counts = counts;
  prm.offsets = offsets;
  prm.perm = perm;
  prm.inv_perm = inv_perm;
  prm.block_map = block_map;
  prm.num_blocks = num_blocks;
  prm.h = h;
  prm.y = y;
  prm.out = out;
  prm.ws = static_cast<int*>(ws);
  prm.err = device_error_ptr();
  prm.wait_cycles = wait_ns > (~0ull) / 3 ? ~0ull : wait_ns * 21 / 10;
  prm.T = T;
  prm.H = H;
  prm.F = F;
  prm.E = E;
  prm.k = k;
  prm.bn = bn;
  const int g0 = (H / KG + GV_WARPS - 1) / GV_WARPS, g1 = (F / KG + GV_WARPS - 1) / GV_WARPS;
  prm.G = g0 > g1 ? g0 : g1;
  if (prm.G > GV_GB) return cudaErrorInvalidValue;
  const size_t smem = decode_smem_bytes(prm.G, E);
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(decode_kernel), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cached_occupancy(reinterpret_cast<const void*>(decode_kernel), GV_THREADS, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidValue;
  if (per_sm > GV_CTAS_PER_SM) per_sm = GV_CTAS_PER_SM;
  // cooperative launch: every CTA resident at once, which the counters between them rely on
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms * per_sm);
  cfg.blockDim = dim3(GV_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_kernel, prm);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
