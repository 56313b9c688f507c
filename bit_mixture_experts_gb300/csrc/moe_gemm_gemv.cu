// Grouped GEMV over groupwise-affine 4-bit weights, for decode-sized tiles (at
// most GV_MAXN token rows per block-map tile).
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details: at batch
// 1 every routed expert's weights are read once per token, so the layer is a
// stream of the 8 + 1 selected experts' packed weights and the work per weight
// is a handful of operations.  What matters is keeping that stream in flight
// on every SM, spending few instructions per weight and keeping the chain of
// dependent steps per work item short.
//
// Weights use the repacked layout of the tensor-core kernel (per matrix, per
// 128-row M-tile, per 64-wide K group: [2 halves][128 rows][16 B] nibbles +
// [128 rows](scale, bias)), so one copy of the weights serves both kernels and
// a warp's 32 rows of one half are 512 contiguous bytes.
//
// Work item (persistent grid, GV_CTAS_PER_SM CTAs of 256 threads per SM; 32
// weight rows per item so that a batch-1 layer still gives every CTA work):
//   gate/up: (tile, 16 features): rows 0-15 are the gate rows and rows 16-31
//            the up rows of those features (M-tiles 2j, 2j+1 of the repacked
//            pair layout); warp w takes K groups w, w+8, ...
//   down:    (tile, 32 output channels); warp w takes K groups w, w+8, ...
// Thread r of a warp copies row r's groups (36 bytes each) into its own
// shared-memory slots with cp.async one item ahead (two slot buffers), so the
// next item's weights stream while this one is computed; it waits for its own
// copies and a warp barrier makes the warp's rows visible to all its lanes
// (no CTA barrier guards the weight stream).  The products run on the tensor
// cores with mma.sync m16n8k16 (bf16 operands, FP32 accumulation): the item's
// 32 rows are two 16-row A blocks and the tile's token rows (at most 8) the
// columns of B, read straight from global memory through L1.  Each lane
// expands only the weight pairs of its own A fragments, exactly as the
// tensor-core kernel expands them (w = bf16(q * scale + bias), one
// fma.rn.bf16x2 per pair), so every weight is expanded once per item whatever
// the tile's row count; a first version multiplied on the FMA pipe with
// bf16 x bf16 -> FP32 FMAs and spent more instructions converting their
// operands than on the dequantisation (decode of 8 tokens: 76 -> 62 µs per
// step with the MMAs).  The warps' partial sums are added in shared memory in
// a fixed order (one barrier per item; the partial-sum buffer alternates
// between items).
#include "moe_common.cuh"
#include "moe_ptx.cuh"
#include "moe_gemv_dev.cuh"

namespace moe {

using namespace gemv_dev;

namespace {

struct GvParams {
  const uint16_t* act;
  const uint8_t* w;
  const int32_t* perm;
  const float* topk_w;
  const int32_t* block_map;
  const int32_t* num_blocks;
  void* out;
  int* err;
  int T, H, F, E, k, bn, cap;
  int G;  // K groups per thread: ceil(K / 64 / 8)
};

__device__ __forceinline__ bool gv_tile(const GvParams& p, int b, Tile* t) {
  t->expert = __ldg(p.block_map + 3 * b);
  t->row0 = __ldg(p.block_map + 3 * b + 1);
  t->rows = __ldg(p.block_map + 3 * b + 2);
  const int A = p.T * p.k;
  bool ok = t->expert >= 0 && t->expert <= p.E && t->rows >= 1 && t->rows <= p.bn && t->rows <= GV_MAXN &&
            t->row0 >= 0;
  if (ok) ok = t->expert < p.E ? (t->row0 + t->rows <= A) : (t->row0 >= A && t->row0 + t->rows <= A + p.T);
  return ok;
}

}  // namespace

// MODE 0: h[r, f] = bf16(silu(g) * u) for the tile's rows r.  MODE 1: y[r, c] = bf16(h[r] . Wd[c]).
template <int MODE>
__global__ void __launch_bounds__(GV_THREADS, GV_CTAS_PER_SM) gemv_kernel(const GvParams p) {
  extern __shared__ uint4 gv_smem[];
  const int K = MODE == 0 ? p.H : p.F;
  const int KT = K / KG;
  const int G = p.G;
  const int MT = MODE == 0 ? (2 * p.F) / TC_M : p.H / TC_M;
  const int IPT = MODE == 0 ? p.F / 16 : p.H / 32;  // work items per tile
  const int A = p.T * p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // shared memory: per buffer b: weight slots [2 G][threads] x 16 B and (scale, bias)
  // slots [G][threads] x 4 B; then partial sums [2][warps][GV_MAXN][32] floats
  const int slot_q = 2 * G * GV_THREADS, slot_sb = G * GV_THREADS;
  uint4* swq0 = gv_smem;
  uint32_t* swsb0 = reinterpret_cast<uint32_t*>(gv_smem + 2 * slot_q);
  float* spart0 = reinterpret_cast<float*>(swsb0 + 2 * slot_sb);

  int nb = __ldg(p.num_blocks);
  if (nb < 0 || nb > p.cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
    nb = nb < 0 ? 0 : p.cap;
  }
  const int items = nb * IPT;

  // copies of item u's row of this thread into buffer b (one commit group, possibly empty)
  auto issue = [&](int u, int b) {
    if (u < items) {
      const int tb = u / IPT, j = u - tb * IPT;
      Tile t;
      if (gv_tile(p, tb, &t)) {
        int mt, L;
        item_row<MODE>(j, lane, &mt, &L);
        const uint8_t* wrow = p.w + (static_cast<size_t>(t.expert) * MT + mt) * KT * static_cast<size_t>(W_BLOCK);
        uint4* q = swq0 + b * slot_q + threadIdx.x;
        uint32_t* sb = swsb0 + b * slot_sb + threadIdx.x;
#pragma unroll 1
        for (int i = 0; i < G; ++i) {
          const int kg = warp + GV_WARPS * i;
          if (kg >= KT) break;
          const uint8_t* blk = wrow + static_cast<size_t>(kg) * W_BLOCK;
          ptx::cp_async_16(ptx::smem_u32(q + (2 * i) * GV_THREADS), blk + L * 16);
          ptx::cp_async_16(ptx::smem_u32(q + (2 * i + 1) * GV_THREADS), blk + 2048 + L * 16);
          ptx::cp_async_4(ptx::smem_u32(sb + i * GV_THREADS), blk + W_PACKED + L * 4);
        }
      }
    }
    ptx::cp_async_commit();
  };

  issue(blockIdx.x, 0);
  int it = 0;
  for (int u = blockIdx.x; u < items; u += gridDim.x, ++it) {
    const int buf = it & 1;
    issue(u + gridDim.x, buf ^ 1);  // next item's weights stream during this one
    const int tb = u / IPT, j = u - tb * IPT;
    Tile t;
    if (!gv_tile(p, tb, &t)) {
      if (threadIdx.x == 0) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
      continue;
    }
    // gate/up: token of tile row n in lane n (the down GEMM reads the h rows in place)
    const int nrow = t.rows;
    int tok_l = -1;
    if (MODE == 0 && lane < nrow) {
      const int r = t.row0 + lane;
      if (r < A) {
        const int a = __ldg(p.perm + r);
        if (a >= 0 && a < A) tok_l = a / p.k;
        else if (warp == 0) set_device_error(p.err, MOE_DEV_BAD_INDEX);
      } else {
        tok_l = r - A;
      }
    }
    // element offset of the activations of this lane's token column (lane / 4) in act (below 2^32:
    // T x H and (A+T) x F are checked on the host); columns past the tile read a valid row
    const int col = lane >> 2;
    const int tk = __shfl_sync(0xffffffffu, tok_l, col);
    // MODE 0: token row of x (a bad index reads token 0); MODE 1: row of h
    const uint32_t xo = MODE == 0 ? static_cast<uint32_t>(tk < 0 ? 0 : tk) * static_cast<uint32_t>(K)
                                  : static_cast<uint32_t>(t.row0 + (col < nrow ? col : 0)) * static_cast<uint32_t>(K);
    float d[2][4] = {};
    ptx::cp_async_wait<1>();  // this thread's copies of item u have landed
    __syncwarp();             // ... and those of the warp's other lanes, whose rows this lane reads
    item_mma<false>(swq0 + buf * slot_q + 32 * warp, swsb0 + buf * slot_sb + 32 * warp, p.act, xo, warp, lane, KT,
                    G, d);

    // reduce the warps' partial sums (fixed order) and finish the item
    float* spart = spart0 + buf * (GV_WARPS * GV_MAXN * 32);
    store_partials(spart, d, warp, lane, nrow);
    __syncthreads();
    if (MODE == 0) {
      if (threadIdx.x < nrow * 16) {
        const int n = threadIdx.x >> 4, fi = threadIdx.x & 15;
        float gs = 0.f, us = 0.f;
        for (int w = 0; w < GV_WARPS; ++w) {
          gs += spart[(w * GV_MAXN + n) * 32 + fi];
          us += spart[(w * GV_MAXN + n) * 32 + 16 + fi];
        }
        uint16_t* h = static_cast<uint16_t*>(p.out);
        h[static_cast<size_t>(t.row0 + n) * p.F + 16 * j + fi] = float_to_bf16_bits(silu(gs) * us);
      }
    } else {
      // warp n finishes tile row n: y[row0 + n, 32 j + lane]
      if (warp < nrow) {
        float y = 0.f;
        for (int w = 0; w < GV_WARPS; ++w) y += spart[(w * GV_MAXN + warp) * 32 + lane];
        static_cast<uint16_t*>(p.out)[static_cast<size_t>(t.row0 + warp) * p.H + 32 * j + lane] =
            float_to_bf16_bits(y);
      }
    }
  }
  ptx::cp_async_wait_all();  // no copy may still be landing when the CTA exits
}

int gemv_max_rows() { return GV_MAXN; }

static int gemv_groups(int K) { return (K / KG + GV_WARPS - 1) / GV_WARPS; }

size_t gemv_smem_bytes(int mode, int H, int F) {
  const int G = gemv_groups(mode == MOE_GATE_UP_SWIGLU ? H : F);
  return 2 * static_cast<size_t>(G) * GV_THREADS * (2 * 16 + 4) + 2 * static_cast<size_t>(GV_WARPS) * GV_MAXN * 32 * 4;
}

cudaError_t launch_gemm_gemv(int mode, const uint16_t* act, int T, int H, int F, int E, int k, const void* w,
                             const int32_t* perm, const float* topk_w, const int32_t* block_map,
                             const int32_t* num_blocks, int bn, int cap, void* out, int num_sms, cudaStream_t s) {
  if (bn > GV_MAXN) return cudaErrorInvalidValue;
  // activation offsets are 32-bit
  if (static_cast<unsigned long long>(T) * H >= (1ull << 32) ||
      static_cast<unsigned long long>(T) * (k + 1) * F >= (1ull << 32))
    return cudaErrorInvalidValue;
  GvParams prm;
  prm.act = act;
  prm.w = static_cast<const uint8_t*>(w);
  prm.perm = perm;
  prm.topk_w = topk_w;
  prm.block_map = block_map;
  prm.num_blocks = num_blocks;
  prm.out = out;
  prm.err = device_error_ptr();
  prm.T = T;
  prm.H = H;
  prm.F = F;
  prm.E = E;
  prm.k = k;
  prm.bn = bn;
  prm.cap = cap;
  prm.G = gemv_groups(mode == MOE_GATE_UP_SWIGLU ? H : F);
  if (prm.G > GV_GB) return cudaErrorInvalidValue;
  const size_t smem = gemv_smem_bytes(mode, H, F);
  static int max_smem = 0;
  if (!max_smem) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  }
  if (smem > static_cast<size_t>(max_smem)) return cudaErrorInvalidValue;
  const int grid = num_sms * GV_CTAS_PER_SM;
  if (mode == MOE_GATE_UP_SWIGLU) {
    const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(gemv_kernel<0>), smem);
    if (e != cudaSuccess) return e;
    gemv_kernel<0><<<grid, GV_THREADS, smem, s>>>(prm);
  } else {
    const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(gemv_kernel<1>), smem);
    if (e != cudaSuccess) return e;
    gemv_kernel<1><<<grid, GV_THREADS, smem, s>>>(prm);
  }
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
