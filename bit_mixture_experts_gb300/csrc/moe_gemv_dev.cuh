// Device helpers of the CUDA-core GEMV over repacked 4-bit weights, shared by
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

// Partial sums per token row: four independent chains (one per pair slot of a
// word), so the FMAs of a row do not form one long dependent chain; they are
// added in a fixed order at the end (acc_total).
constexpr int GV_NACC = 4;

__device__ __forceinline__ float acc_total(const float (&a)[GV_NACC]) { return (a[0] + a[1]) + (a[2] + a[3]); }

// acc[n] += sum over one K group of w * x[n] for token rows n = N0 .. N0+NT-1:
// the row's packed words (lo: K 0..31, hi: K 32..63 of the group), its
// (scale, bias) and the group's activations of each row at xg + xoff[n]
// (bf16, global; read through L1, or through L2 only when COHERENT, for
// activations written earlier by the same kernel).
template <int N0, int NT, bool COHERENT = false>
__device__ __forceinline__ void group_dot(uint4 lo, uint4 hi, uint32_t sb, const uint16_t* xg,
                                          const uint32_t (&xoff)[GV_MAXN], float (&acc)[GV_MAXN][GV_NACC]) {
  const uint32_t s2 = (sb & 0xffffu) * 0x10001u;
  const uint32_t b2 = (sb >> 16) * 0x10001u;
  const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t wp[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) wp[j] = dequant_pair(words[w], j, s2, b2);
#pragma unroll
    for (int n = N0; n < N0 + NT; ++n) {
      const uint4* xp = reinterpret_cast<const uint4*>(xg + xoff[n]) + w;
      const uint4 x = COHERENT ? __ldcg(xp) : __ldg(xp);
      dot_pair(acc[n][0], wp[0], x.x);
      dot_pair(acc[n][1], wp[1], x.y);
      dot_pair(acc[n][2], wp[2], x.z);
      dot_pair(acc[n][3], wp[3], x.w);
    }
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
