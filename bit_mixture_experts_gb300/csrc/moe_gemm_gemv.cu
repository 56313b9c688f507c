// CUDA-core grouped GEMV over groupwise-affine 4-bit weights, for decode-sized
// tiles (at most GV_MAXN token rows per block-map tile).
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details: at batch
// 1 every routed expert's weights are read once per token, so the layer is a
// stream of the 8 + 1 selected experts' packed weights and the work per weight
// is a handful of ALU operations.  There is nothing for the tensor cores to do
// here; what matters is keeping enough of that stream in flight on every SM.
//
// Weights use the repacked layout of the tensor-core kernel (per matrix, per
// 128-row M-tile, per 64-wide K group: [2 halves][128 rows][16 B] nibbles +
// [128 rows](scale, bias)), so one copy of the weights serves both kernels and
// a warp's 32 rows of one half are 512 contiguous bytes.
//
// Work item (persistent grid, GV_CTAS_PER_SM CTAs of 256 threads per SM):
//   gate/up: (tile, 32 features): the 32 gate and 32 up rows of those
//            features (M-tiles 2j, 2j+1 of the repacked pair layout) against
//            all H; warp w takes K groups w, w+8, ...; lane = feature.
//   down:    (tile, 128 output channels = one M-tile) against all F; warp w
//            takes lane quarter w % 4 and K groups w / 4, w / 4 + 2, ...
// Each thread first issues the loads of all its weight words (up to GV_GB
// groups) into registers, then stages the tile's activation rows in shared
// memory, then expands each word to bf16 pairs exactly as the tensor-core
// kernel does (w = bf16(q * scale + bias), one fma.rn.bf16x2 per pair) and
// accumulates w * x in FP32 with mixed-precision FMAs.  Partial sums of the
// warps are added in shared memory in a fixed order.
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int GV_THREADS = 256;
constexpr int GV_WARPS = GV_THREADS / 32;
constexpr int GV_MAXN = 8;  // token rows per tile
constexpr int GV_GB = 4;    // K groups a thread holds in registers at once
constexpr int GV_CTAS_PER_SM = 2;
constexpr int KG = 64;
constexpr int TC_M = 128;
constexpr int W_PACKED = TC_M * 32;
constexpr int W_BLOCK = W_PACKED + TC_M * 4;

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
};

// bf16 pair of weights (element 2j in the low half, 2j+1 in the high half) of
// a repacked word: 128 + q exactly, minus 128, times scale plus bias, rounded once.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t word, int j, uint32_t s2, uint32_t b2) {
  constexpr uint32_t MAGIC = 0x43004300u;
  uint32_t x = ((word >> (4 * j)) & 0x000f000fu) | MAGIC, r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(MAGIC));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(r), "r"(s2), "r"(b2));
  return r;
}

// acc += w.lo * x.lo + w.hi * x.hi (bf16 operands, FP32 accumulation, products exact)
__device__ __forceinline__ void dot_pair(float& acc, uint32_t w2, uint32_t x2) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\tmov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\tfma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
      : "+f"(acc)
      : "r"(w2), "r"(x2));
}

// One repacked row of one K group: 8 words (K elements 8w .. 8w+7) + (scale, bias).
struct RowGroup {
  uint4 lo, hi;
  uint32_t sb;
};

__device__ __forceinline__ RowGroup load_row_group(const uint8_t* blk, int L) {
  RowGroup g;
  g.lo = __ldg(reinterpret_cast<const uint4*>(blk + L * 16));
  g.hi = __ldg(reinterpret_cast<const uint4*>(blk + 2048 + L * 16));
  g.sb = __ldg(reinterpret_cast<const uint32_t*>(blk + W_PACKED + L * 4));
  return g;
}

__device__ __forceinline__ uint32_t word_of(const RowGroup& g, int w) {
  const uint4& v = w < 4 ? g.lo : g.hi;
  switch (w & 3) {
    case 0: return v.x;
    case 1: return v.y;
    case 2: return v.z;
    default: return v.w;
  }
}

// acc[n] += sum over the group's 64 K of w * x[n], n < rows (x: bf16 rows in smem, pitch K)
template <int NM>
__device__ __forceinline__ void group_dot(const RowGroup (&g)[NM], const uint16_t* sx, int K, int k0, int rows,
                                          float (&acc)[NM][GV_MAXN]) {
  uint32_t s2[NM], b2[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    s2[m] = (g[m].sb & 0xffffu) * 0x10001u;
    b2[m] = (g[m].sb >> 16) * 0x10001u;
  }
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t wp[NM][4];
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const uint32_t word = word_of(g[m], w);
#pragma unroll
      for (int j = 0; j < 4; ++j) wp[m][j] = dequant_pair(word, j, s2[m], b2[m]);
    }
#pragma unroll
    for (int n = 0; n < GV_MAXN; ++n) {
      if (n < rows) {
        const uint4 xv = *reinterpret_cast<const uint4*>(sx + n * K + k0 + 8 * w);
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          dot_pair(acc[m][n], wp[m][0], xv.x);
          dot_pair(acc[m][n], wp[m][1], xv.y);
          dot_pair(acc[m][n], wp[m][2], xv.z);
          dot_pair(acc[m][n], wp[m][3], xv.w);
        }
      }
    }
  }
}

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

// MODE 0: h[r, f] = bf16(silu(g) * u) for the tile's rows r.  MODE 1: acc[token] += w * y.
template <int MODE>
__global__ void __launch_bounds__(GV_THREADS, GV_CTAS_PER_SM) gemv_kernel(const GvParams p) {
  extern __shared__ uint4 gv_smem[];
  __shared__ int s_tok[GV_MAXN];
  __shared__ float s_wt[GV_MAXN];
  constexpr int NM = MODE == 0 ? 2 : 1;  // matrices per thread: gate and up, or down
  const int K = MODE == 0 ? p.H : p.F;
  const int KT = K / KG;
  const int MT = MODE == 0 ? (2 * p.F) / TC_M : p.H / TC_M;
  const int IPT = MODE == 0 ? p.F / 32 : MT;  // work items per tile
  const int A = p.T * p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint16_t* sx = reinterpret_cast<uint16_t*>(gv_smem);  // [GV_MAXN][K] bf16
  float* spart = reinterpret_cast<float*>(sx + GV_MAXN * K);
  // MODE 0: spart[warp][m][n][lane]; MODE 1: spart[khalf][n][128 rows]

  int nb = __ldg(p.num_blocks);
  if (nb < 0 || nb > p.cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
    nb = nb < 0 ? 0 : p.cap;
  }
  const int items = nb * IPT;
  // K groups of this thread: MODE 0: warp, warp + 8, ...; MODE 1: khalf, khalf + 2, ...
  const int kstep = MODE == 0 ? GV_WARPS : 2;
  const int kfirst = MODE == 0 ? warp : (warp >> 2);
  const int L = MODE == 0 ? 0 : 32 * (warp & 3) + lane;  // MODE 1: row within the M-tile

  for (int u = blockIdx.x; u < items; u += gridDim.x) {
    const int b = u / IPT, j = u - b * IPT;
    Tile t;
    if (!gv_tile(p, b, &t)) {
      if (threadIdx.x == 0) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
      continue;
    }
    // weight rows of this item
    const uint8_t* wbase[NM];
    int Lw;
    if (MODE == 0) {
      const int f = 32 * j + lane, pair = f / TC_M;
      Lw = f % TC_M;
      wbase[0] = p.w + (static_cast<size_t>(t.expert) * MT + 2 * pair) * KT * static_cast<size_t>(W_BLOCK);
      if (NM > 1) wbase[NM - 1] = wbase[0] + static_cast<size_t>(KT) * W_BLOCK;
    } else {
      Lw = L;
      wbase[0] = p.w + (static_cast<size_t>(t.expert) * MT + j) * KT * static_cast<size_t>(W_BLOCK);
    }
    float acc[NM][GV_MAXN];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int n = 0; n < GV_MAXN; ++n) acc[m][n] = 0.f;

    __syncthreads();  // the previous item is done with sx / spart / s_tok
    for (int kb = 0; kb < KT; kb += kstep * GV_GB) {
      // 1. this thread's weight words for up to GV_GB groups, all loads in flight at once
      RowGroup g[GV_GB][NM];
#pragma unroll
      for (int i = 0; i < GV_GB; ++i) {
        const int kg = kb + kfirst + kstep * i;
        if (kg < KT) {
#pragma unroll
          for (int m = 0; m < NM; ++m) g[i][m] = load_row_group(wbase[m] + static_cast<size_t>(kg) * W_BLOCK, Lw);
        }
      }
      // 2. (first batch) the tile's activation rows -> smem, while those loads are in flight
      if (kb == 0) {
        if (threadIdx.x < t.rows) {
          const int i = threadIdx.x, r = t.row0 + i;
          int tok = -1;
          float wt = 0.f;
          if (r < A) {
            const int a = __ldg(p.perm + r);
            if (a >= 0 && a < A) {
              tok = a / p.k;
              wt = __ldg(p.topk_w + a);
            } else {
              set_device_error(p.err, MOE_DEV_BAD_INDEX);
            }
          } else {
            tok = r - A;
            wt = 1.0f;
          }
          s_tok[i] = tok;
          s_wt[i] = wt;
        }
        __syncthreads();
        const int cpr = K / 8;  // 16-byte chunks per row
        for (int idx = threadIdx.x; idx < t.rows * cpr; idx += GV_THREADS) {
          const int i = idx / cpr, c = idx - i * cpr;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (MODE == 0) {
            const int tok = s_tok[i];
            if (tok >= 0) v = __ldg(reinterpret_cast<const uint4*>(p.act + static_cast<size_t>(tok) * K) + c);
          } else {
            v = __ldg(reinterpret_cast<const uint4*>(p.act + static_cast<size_t>(t.row0 + i) * K) + c);
          }
          reinterpret_cast<uint4*>(sx + i * K)[c] = v;
        }
        __syncthreads();
      }
      // 3. expand and accumulate
#pragma unroll
      for (int i = 0; i < GV_GB; ++i) {
        const int kg = kb + kfirst + kstep * i;
        if (kg < KT) group_dot<NM>(g[i], sx, K, kg * KG, t.rows, acc);
      }
    }

    // reduce the warps' partial sums (fixed order) and finish the item
    if (MODE == 0) {
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int n = 0; n < GV_MAXN; ++n)
          if (n < t.rows) spart[((warp * NM + m) * GV_MAXN + n) * 32 + lane] = acc[m][n];
      __syncthreads();
      if (threadIdx.x < t.rows * 32) {
        const int n = threadIdx.x >> 5;
        float gs = 0.f, us = 0.f;
        for (int w = 0; w < GV_WARPS; ++w) {
          gs += spart[((w * NM + 0) * GV_MAXN + n) * 32 + lane];
          us += spart[((w * NM + NM - 1) * GV_MAXN + n) * 32 + lane];
        }
        uint16_t* h = static_cast<uint16_t*>(p.out);
        h[static_cast<size_t>(t.row0 + n) * p.F + 32 * j + lane] = float_to_bf16_bits(silu(gs) * us);
      }
    } else {
      const int kh = warp >> 2;
#pragma unroll
      for (int n = 0; n < GV_MAXN; ++n)
        if (n < t.rows) spart[(kh * GV_MAXN + n) * TC_M + L] = acc[0][n];
      __syncthreads();
      float* out = static_cast<float*>(p.out);
      for (int idx = threadIdx.x; idx < t.rows * TC_M; idx += GV_THREADS) {
        const int n = idx / TC_M, row = idx - n * TC_M;
        const int tok = s_tok[n];
        if (tok >= 0) {
          const float y = spart[n * TC_M + row] + spart[(GV_MAXN + n) * TC_M + row];
          atomicAdd(out + static_cast<size_t>(tok) * p.H + TC_M * j + row, s_wt[n] * y);
        }
      }
    }
  }
}

int gemv_max_rows() { return GV_MAXN; }

size_t gemv_smem_bytes(int mode, int H, int F) {
  const int K = mode == MOE_GATE_UP_SWIGLU ? H : F;
  const size_t part = mode == MOE_GATE_UP_SWIGLU ? static_cast<size_t>(GV_WARPS) * 2 * GV_MAXN * 32 * 4
                                                 : static_cast<size_t>(2) * GV_MAXN * TC_M * 4;
  return static_cast<size_t>(GV_MAXN) * K * 2 + part;
}

cudaError_t launch_gemm_gemv(int mode, const uint16_t* act, int T, int H, int F, int E, int k, const void* w,
                             const int32_t* perm, const float* topk_w, const int32_t* block_map,
                             const int32_t* num_blocks, int bn, int cap, void* out, int num_sms, cudaStream_t s) {
  if (bn > GV_MAXN) return cudaErrorInvalidValue;
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
  const size_t smem = gemv_smem_bytes(mode, H, F);
  int dev = 0, max_smem = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (smem > static_cast<size_t>(max_smem)) return cudaErrorInvalidValue;
  const int grid = num_sms * GV_CTAS_PER_SM;
  if (mode == MOE_GATE_UP_SWIGLU) {
    cudaFuncSetAttribute(gemv_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    gemv_kernel<0><<<grid, GV_THREADS, smem, s>>>(prm);
  } else {
    cudaFuncSetAttribute(gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    gemv_kernel<1><<<grid, GV_THREADS, smem, s>>>(prm);
  }
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
