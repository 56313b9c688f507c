// Device helpers of the decode GEMV over repacked 4-bit weights, shared by
// the GEMV kernel and the fused decode kernel (see moe_gemm_gemv.cu).
#pragma once
#include "moe_common.cuh"

namespace moe {
namespace gemv_dev {

constexpr int GV_THREADS = 256;
constexpr int GV_WARPS = GV_THREADS / 32;
constexpr int GV_MAXN = 8;  // token rows per tile
constexpr int GV_GB = 8;    // K groups per thread at most (K <= 64 * 8 * 8 = 4096)
constexpr int GV_CTAS_PER_SM = 2;
constexpr int KG = 64;
constexpr int TC_M = 128;
constexpr int W_PACKED = TC_M * 32;
constexpr int W_BLOCK = W_PACKED + TC_M * 4;

// Weight pair j = sh / 4 of a repacked word as bf16x2 (element 2j in the low
// half, 2j + 1 in the high half): 128 + q exactly, minus 128, times scale plus
// bias, rounded once.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t word, int sh, uint32_t s2, uint32_t b2) {
  constexpr uint32_t MAGIC = 0x43004300u;
  uint32_t x = ((word >> sh) & 0x000f000fu) | MAGIC, r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(MAGIC));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(r), "r"(s2), "r"(b2));
  return r;
}

// d += A (16 x 16, bf16, row-major fragments a0..a3) * B (16 x 8, bf16, b0, b1), FP32 accumulation.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One work item's share of warp `warp`: its K groups kg = warp + GV_WARPS * i
// (i < G, kg < KT) of the item's 32 weight rows against the tile's token rows,
// on the tensor cores (mma.sync m16n8k16, bf16 operands, FP32 accumulation).
// Rows 0-15 and 16-31 of the item are the two 16-row A blocks; the tile's
// token rows are the 8 columns of B (columns past the tile's rows read a valid
// row and are ignored).  The weights come from the slots of the warp's 32
// threads (thread 32 warp + r holds row r's group: words at sw[(2 i) *
// GV_THREADS + r] and sw[(2 i + 1) * GV_THREADS + r], (scale, bias) at
// ssbw[i * GV_THREADS + r]).  Lane (g, t) = (lane / 4, lane % 4) expands pair
// t of every word of rows g, g + 8, 16 + g, 24 + g: for k-step m (16 K values)
// its A registers are pair t of words 2m and 2m + 1 of two rows, which is the
// fragment layout of K = 16m + 2t and 16m + 8 + 2t, and its B registers are
// the activations of the same K for token column g, read from `act` at
// element offset xo (+ 64 kg): no element is expanded twice and no
// conversion of a product operand to FP32 is needed.  d[mb][0..3] receive
// rows 16 mb + g (d0, d1) and 16 mb + g + 8 (d2, d3), columns 2t and 2t + 1.
template <bool COHERENT>
__device__ __forceinline__ void item_mma(const uint4* sw, const uint32_t* ssbw, const uint16_t* act, uint32_t xo,
                                         int warp, int lane, int KT, int G, float (&d)[2][4]) {
  const int g = lane >> 2, sh = 4 * (lane & 3);
#pragma unroll 1
  for (int i = 0; i < G; ++i) {
    const int kg = warp + GV_WARPS * i;
    if (kg >= KT) break;
    // B: the activation pairs K = 8w + 2t (w = 0..7) of the group, token column g
    const uint32_t* xp = reinterpret_cast<const uint32_t*>(act + xo + kg * KG) + (lane & 3);
    uint32_t b[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) b[w] = COHERENT ? __ldcg(xp + 4 * w) : __ldg(xp + 4 * w);
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
      const int r0 = 16 * mb + g, r1 = r0 + 8;
      const uint4 lo0 = sw[(2 * i) * GV_THREADS + r0], hi0 = sw[(2 * i + 1) * GV_THREADS + r0];
      const uint4 lo1 = sw[(2 * i) * GV_THREADS + r1], hi1 = sw[(2 * i + 1) * GV_THREADS + r1];
      const uint32_t sb0 = ssbw[i * GV_THREADS + r0], sb1 = ssbw[i * GV_THREADS + r1];
      const uint32_t s20 = (sb0 & 0xffffu) * 0x10001u, b20 = (sb0 >> 16) * 0x10001u;
      const uint32_t s21 = (sb1 & 0xffffu) * 0x10001u, b21 = (sb1 >> 16) * 0x10001u;
      const uint32_t w0[8] = {lo0.x, lo0.y, lo0.z, lo0.w, hi0.x, hi0.y, hi0.z, hi0.w};
      const uint32_t w1[8] = {lo1.x, lo1.y, lo1.z, lo1.w, hi1.x, hi1.y, hi1.z, hi1.w};
#pragma unroll
      for (int m = 0; m < 4; ++m)
        mma_16816(d[mb], dequant_pair(w0[2 * m], sh, s20, b20), dequant_pair(w1[2 * m], sh, s21, b21),
                  dequant_pair(w0[2 * m + 1], sh, s20, b20), dequant_pair(w1[2 * m + 1], sh, s21, b21), b[2 * m],
                  b[2 * m + 1]);
    }
  }
}

// The warp's partial sums of one item into spart[(warp * GV_MAXN + n) * 32 + row] for the
// tile's token rows n < nrow (the layout the items' reductions read).
__device__ __forceinline__ void store_partials(float* spart, const float (&d)[2][4], int warp, int lane, int nrow) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mb = 0; mb < 2; ++mb)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = 2 * t + (e & 1), row = 16 * mb + g + 8 * (e >> 1);
      if (n < nrow) spart[(warp * GV_MAXN + n) * 32 + row] = d[mb][e];
    }
}

// Weight row of item j of a tile for this lane: (M-tile, row within it).
template <int MODE>
__device__ __forceinline__ void item_row(int j, int lane, int* mt, int* L) {
  if (MODE == 0) {
    const int f = 16 * j + (lane & 15);
    *mt = 2 * (f / TC_M) + (lane >> 4);  // gate M-tile, or the up M-tile after it
    *L = f % TC_M;
  } else {
    const int c = 32 * j + lane;
    *mt = c / TC_M;
    *L = c % TC_M;
  }
}

}  // namespace gemv_dev
}  // namespace moe
