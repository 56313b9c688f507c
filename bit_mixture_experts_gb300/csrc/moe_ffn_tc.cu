// Fused expert FFN per token tile: the gate/up projection with SwiGLU and the
// down projection of one block-map tile in one pass of the tensor-core
// pipeline, the intermediate h kept in shared memory between the two.
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details, Prefill
// optimizations bullet: the 4-bit weights are expanded inside the grouped
// GEMM and never stored expanded; the itinai.com post on the same engine says
// the same of the bf16 copy.  Here h follows that rule too: it never leaves the
// SM that computes it.
//
// Work unit: one block-map tile (an expert and at most 64 token rows).  Its
// sub-units, in order:
//   G_j (j < F/128): gate/up of features 128j .. 128j+127 over K = H, stages of
//        K = 128 with two M-tiles (the gate rows and the up rows); the
//        epilogue writes h = bf16(silu(g) u) into the tile's h buffer in shared
//        memory, as 128B-swizzled K-major atoms of 64 features -- the layout
//        from which the MMA reads its B operand;
//   D_m (m < H/128): down rows 128m .. 128m+127 over K = F, stages of K = 256
//        with one M-tile, B = the h buffer; the epilogue writes y = bf16(acc)
//        rows to global memory, as the down GEMM does.
// Both kinds of stage carry four repacked 128 x 64 blocks (18 KB) and fill 128
// TMEM columns with dequantised weights, so one weight ring, one A ring and
// one dequantisation serve both.  The roles are those of the one-CTA grouped
// GEMM (moe_gemm_tc.cu).  h is handed over by two barriers: HREADY (the four
// epilogue warps, after the last G_j; the MMA warp waits before D_0) and HFREE
// (committed by the MMA warp after the tile's last down MMAs; the epilogue
// waits before it writes the next tile's h).
//
// The MMAs into each accumulator run in the same order as in the two separate
// GEMMs, and the epilogues compute the same expressions, so h and y (and the
// layer's output after moe_combine) are bit for bit those of the separate
// path.  The h buffer takes (F/64) x 64 rows x 128 bytes of shared memory (64
// KB at F = 512), hence the limit of 64 rows per tile.
#include <cuda.h>
#include <string.h>

#include "moe_common.cuh"
#include "moe_ptx.cuh"
#include "moe_tc_dev.cuh"

namespace moe {

using namespace tc_dev;

namespace {

constexpr int FF_THREADS = 512;
constexpr int FF_BLOCKS = 4;                    // repacked 128 x 64 blocks per stage
constexpr int FF_WSTAGE = FF_BLOCKS * W_BLOCK;  // 18,432 bytes of packed weights per stage
constexpr int FF_ACOLS = FF_BLOCKS * 32;        // TMEM columns of one dequantised stage
constexpr int FF_NWMAX = 12;                    // weight ring slots (an even run-time depth)
constexpr int FF_NA = 2;                        // A ring slots: one per dequant warpgroup
constexpr int FF_NBMAX = 8;                     // activation ring slots
constexpr int FF_GATHER_T = 64;                 // threads gathering activation rows
constexpr int FF_TMEM_COLS = 512;
constexpr int FF_EPI_ROWS = 32;
constexpr int FF_STAGE_BYTES = 2 * FF_EPI_ROWS * TC_M * 2;  // epilogue staging: two chunks of 32 rows
constexpr int FF_EPI_BAR = 1;                   // named barrier of the four epilogue warps
constexpr int FF_MAX_ROWS = 64;

constexpr int FB_WFULL = 0;
constexpr int FB_WEMPTY = FB_WFULL + FF_NWMAX;
constexpr int FB_AFULL = FB_WEMPTY + FF_NWMAX;
constexpr int FB_AEMPTY = FB_AFULL + FF_NA;
constexpr int FB_BFULL = FB_AEMPTY + FF_NA;
constexpr int FB_BEMPTY = FB_BFULL + FF_NBMAX;
constexpr int FB_DFULL = FB_BEMPTY + FF_NBMAX;
constexpr int FB_DEMPTY = FB_DFULL + 2;
constexpr int FB_HREADY = FB_DEMPTY + 2;
constexpr int FB_HFREE = FB_HREADY + 1;
constexpr int FB_FIN = FB_HFREE + 1;
constexpr int FB_N = FB_FIN + 1;
constexpr int FF_BAR_BYTES = (FB_N * 8 + 15) & ~15;
constexpr int FF_MISC = 16;  // abort flag, TMEM base

struct FfParams {
  const uint16_t* x;
  const uint8_t* w13;
  const uint8_t* w2;
  const int32_t* perm;
  const int32_t* block_map;
  const int32_t* num_blocks;
  uint16_t* y;
  int* err;
  unsigned long long wait_cycles;
  uint32_t sleep_ns;
  int T, H, F, E, k, bn, cap;
  int boxr;  // rows per activation stage and per h atom (block_n rounded up to 16, <= 64)
  int nb;    // activation ring depth
  int nw;    // weight ring depth (even)
  int sb;    // bytes of one activation stage: two atoms of boxr rows x 128 bytes
};

// Block-map entry b, or false for a malformed one (every role decides alike).
__device__ __forceinline__ bool ff_tile(const FfParams& p, int b, Tile* t) {
  t->expert = __ldg(p.block_map + 3 * b);
  t->row0 = __ldg(p.block_map + 3 * b + 1);
  t->rows = __ldg(p.block_map + 3 * b + 2);
  const int A = p.T * p.k;
  bool ok = t->expert >= 0 && t->expert <= p.E && t->rows >= 1 && t->rows <= p.bn && t->row0 >= 0;
  if (ok) ok = t->expert < p.E ? (t->row0 + t->rows <= A) : (t->row0 >= A && t->row0 + t->rows <= A + p.T);
  return ok;
}

}  // namespace

__global__ void __launch_bounds__(FF_THREADS, 1) ffn_tc_kernel(const FfParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int NB = p.nb, SB = p.sb, NW = p.nw, BOXR = p.boxr;
  const uint32_t atom = static_cast<uint32_t>(BOXR) * 128u;
  const int NG = p.F / TC_M, NDN = p.H / TC_M;          // gate/up and down sub-units of a tile
  const int NSG = p.H / (2 * KG), NSD = p.F / (4 * KG);  // stages of each
  const int KT0 = p.H / KG, KT1 = p.F / KG, MT0 = (2 * p.F) / TC_M, MT1 = p.H / TC_M;
  const uint32_t off_h = static_cast<uint32_t>(NB * SB);                      // h buffer: F / 64 atoms
  const uint32_t off_w = off_h + static_cast<uint32_t>(p.F / KG) * atom;      // weight ring
  const uint32_t off_bar = off_w + static_cast<uint32_t>(NW * FF_WSTAGE);
  const uint32_t bar0 = sbase + off_bar;
  auto bar = [bar0](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + off_bar + FF_BAR_BYTES);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + off_bar + FF_BAR_BYTES + 4);
  uint16_t* s_stage = reinterpret_cast<uint16_t*>(smem + off_bar + FF_BAR_BYTES + FF_MISC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int A = p.T * p.k;
  const int DM = BOXR;                                  // accumulator columns of one M-tile
  const uint32_t A0 = static_cast<uint32_t>(4 * DM);  // two buffers of two M-tiles, then the A ring
  const int SU = NG + NDN;
  int nb = __ldg(p.num_blocks);
  if (nb < 0 || nb > p.cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
    nb = nb < 0 ? 0 : p.cap;
  }

  if (threadIdx.x == 0) {
    *s_abort = 0;
    for (int s = 0; s < FF_NWMAX; ++s) {
      ptx::mbar_init(bar(FB_WFULL + s), 1);
      ptx::mbar_init(bar(FB_WEMPTY + s), 4);
    }
    for (int s = 0; s < FF_NA; ++s) {
      ptx::mbar_init(bar(FB_AFULL + s), 4);
      ptx::mbar_init(bar(FB_AEMPTY + s), 1);
    }
    for (int s = 0; s < FF_NBMAX; ++s) {
      ptx::mbar_init(bar(FB_BFULL + s), FF_GATHER_T);
      ptx::mbar_init(bar(FB_BEMPTY + s), 1);
    }
    for (int d = 0; d < 2; ++d) {
      ptx::mbar_init(bar(FB_DFULL + d), 1);
      ptx::mbar_init(bar(FB_DEMPTY + d), 4);
    }
    ptx::mbar_init(bar(FB_HREADY), 4);
    ptx::mbar_init(bar(FB_HFREE), 1);
    ptx::mbar_init(bar(FB_FIN), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), FF_TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const unsigned long long lim = p.wait_cycles;
  int prod_w = 0;  // weight stages issued, for the drain after a timeout

  if (warp == 0) {
    // ------------------------------------------------ weight producer: W13 blocks, then W2 blocks, per tile
    int& it = prod_w;
    for (int b = blockIdx.x; b < nb; b += gridDim.x) {
      Tile t;
      if (!ff_tile(p, b, &t)) continue;
      for (int j = 0; j < SU; ++j) {
        const bool gu = j < NG;
        const int ns = gu ? NSG : NSD;
        for (int ks = 0; ks < ns; ++ks, ++it) {
          const int s = it % NW, r = it / NW;
          if (r > 0 && !wait_warp(bar(FB_WEMPTY + s), (r - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) goto wprod_done;
          const uint32_t dst = sbase + off_w + static_cast<uint32_t>(s * FF_WSTAGE);
          ptx::mbar_arrive_expect_tx_elect(bar(FB_WFULL + s), static_cast<uint32_t>(FF_WSTAGE));
          if (gu) {
            // the gate M-tile (2j) and the up M-tile (2j + 1) of features 128j.., K groups 2ks, 2ks + 1
            for (int m = 0; m < 2; ++m) {
              const uint8_t* src =
                  p.w13 + ((static_cast<size_t>(t.expert) * MT0 + 2 * j + m) * KT0 + 2 * ks) * W_BLOCK;
              ptx::bulk_g2s_elect(dst + m * 2 * W_BLOCK, src, 2 * W_BLOCK, bar(FB_WFULL + s));
            }
          } else {
            // down M-tile j - NG, K groups 4ks .. 4ks + 3 (contiguous)
            const uint8_t* src =
                p.w2 + ((static_cast<size_t>(t.expert) * MT1 + (j - NG)) * KT1 + 4 * ks) * W_BLOCK;
            ptx::bulk_g2s_elect(dst, src, FF_WSTAGE, bar(FB_WFULL + s));
          }
        }
      }
    }
  wprod_done:;
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    int ui = 0, tc = 0;
    int sa = 0, pa = 0, sbi = 0, pb = 0;
    for (int b = blockIdx.x; b < nb; b += gridDim.x) {
      Tile t;
      if (!ff_tile(p, b, &t)) continue;
      const uint32_t idesc = ptx::idesc_bf16_f32(TC_M, round16(t.rows));
      for (int j = 0; j < SU; ++j) {
        const bool gu = j < NG;
        const int ns = gu ? NSG : NSD;
        const int d = ui & 1, rd = ui >> 1;
        if (rd > 0 && !wait_warp(bar(FB_DEMPTY + d), (rd - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
        // the tile's h is complete before its first down MMA
        if (j == NG && !wait_warp(bar(FB_HREADY), tc & 1, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
        ptx::tc_fence_after();
        const uint32_t d0 = tmem + static_cast<uint32_t>(d * 2 * DM), d1 = d0 + DM;
        for (int ks = 0; ks < ns; ++ks) {
          if (!wait_warp(bar(FB_AFULL + sa), pa, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
          if (gu) {
            if (!wait_warp(bar(FB_BFULL + sbi), pb, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
            ptx::fence_proxy_async_smem();  // cp.async-written rows, read by the tensor core
          }
          ptx::tc_fence_after();
          const uint32_t a0 = tmem + A0 + static_cast<uint32_t>(sa * FF_ACOLS);
          const uint32_t acc0 = ks != 0;
          if (gu) {
            const uint32_t b0 = sbase + static_cast<uint32_t>(sbi * SB);
#pragma unroll
            for (int g = 0; g < 2; ++g)
              ptx::mma_group_ts_elect<true>(d0, d1, a0 + g * 32, a0 + 64 + g * 32, ptx::smem_desc_sw128(b0 + g * atom),
                                            idesc, g == 0 ? acc0 : 1u);
          } else {
            const uint32_t hb = sbase + off_h + static_cast<uint32_t>(4 * ks) * atom;
#pragma unroll
            for (int g = 0; g < 4; ++g)
              ptx::mma_group_ts_elect<false>(d0, d0, a0 + g * 32, a0 + g * 32, ptx::smem_desc_sw128(hb + g * atom),
                                             idesc, g == 0 ? acc0 : 1u);
          }
          ptx::mma_commit_elect(bar(FB_AEMPTY + sa));
          if (++sa == FF_NA) {
            sa = 0;
            pa ^= 1;
          }
          if (gu) {
            ptx::mma_commit_elect(bar(FB_BEMPTY + sbi));
            if (++sbi == NB) {
              sbi = 0;
              pb ^= 1;
            }
          }
        }
        ptx::mma_commit_elect(bar(FB_DFULL + d));
        ++ui;
      }
      ptx::mma_commit_elect(bar(FB_HFREE));  // the tile's down MMAs have read h once they complete
      ++tc;
    }
  mma_done:
    ptx::mma_commit_elect(bar(FB_FIN));
    if (lane == 0) wait_drain(bar(FB_FIN), 0, lim);
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------ activation gather (gate/up stages): token rows of x
    const int gt = threadIdx.x - 64;  // 0..63
    const int chunk = gt & 7, row_a = gt >> 3;
    int it = 0;
    bool aborted = false;
    for (int b = blockIdx.x; b < nb && !aborted; b += gridDim.x) {
      Tile t;
      if (!ff_tile(p, b, &t)) continue;
      int tok[FF_MAX_ROWS / 8];
#pragma unroll
      for (int jj = 0; jj < FF_MAX_ROWS / 8; ++jj) {
        const int i = row_a + 8 * jj;
        const int r = t.row0 + i;
        tok[jj] = (i < t.rows && r < A) ? __ldg(p.perm + r) : 0;
      }
      bool bad = false;
#pragma unroll
      for (int jj = 0; jj < FF_MAX_ROWS / 8; ++jj) {
        const int i = row_a + 8 * jj;
        const int r = t.row0 + i;
        int tk = -1;
        if (i < t.rows) {
          if (r >= A) tk = r - A;  // shared-expert rows follow the routed ones, in token order
          else if (tok[jj] >= 0 && tok[jj] < A) tk = tok[jj] / p.k;
          else bad = true;
        }
        tok[jj] = tk;
      }
      if (bad) set_device_error(p.err, MOE_DEV_BAD_INDEX);
      for (int j = 0; j < NG && !aborted; ++j) {
        for (int ks = 0; ks < NSG; ++ks, ++it) {
          const int s = it % NB, r = it / NB;
          if (r > 0 && !wait_warp(bar(FB_BEMPTY + s), (r - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) {
            aborted = true;
            break;
          }
          const uint32_t dst0 = sbase + static_cast<uint32_t>(s * SB);
#pragma unroll
          for (int jj = 0; jj < FF_MAX_ROWS / 8; ++jj) {
            const int i = row_a + 8 * jj;
            if (tok[jj] >= 0) {
              const uint16_t* src = p.x + static_cast<size_t>(tok[jj]) * p.H + ks * 2 * KG + chunk * 8;
              const uint32_t dst = dst0 + (i >> 3) * 1024 + (i & 7) * 128 + ((chunk ^ (i & 7)) << 4);
#pragma unroll
              for (int g = 0; g < 2; ++g) ptx::cp_async_16(dst + g * atom, src + g * KG);
            }
          }
          ptx::cp_async_mbar_arrive(bar(FB_BFULL + s));
        }
      }
    }
    ptx::cp_async_wait_all();
  } else if (warp < 12) {
    // ------------------------------------------------ dequant: warpgroup wg expands the stages it with
    // it % 2 == wg; every stage is four blocks, block b going to TMEM columns 32b .. 32b + 31 of the
    // A slot (gate/up: the gate M-tile's two K groups, then the up M-tile's; down: four K groups)
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int L = 32 * q + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16) + A0;
    int it = 0;
    for (int b = blockIdx.x; b < nb; b += gridDim.x) {
      Tile t;
      if (!ff_tile(p, b, &t)) continue;
      for (int j = 0; j < SU; ++j) {
        const int ns = j < NG ? NSG : NSD;
        for (int ks = 0; ks < ns; ++ks, ++it) {
          if ((it & 1) != wg) continue;
          const int sa = it % FF_NA, sw = it % NW;
          if (!wait_warp(bar(FB_WFULL + sw), (it / NW) & 1, s_abort, p.err, lim, p.sleep_ns)) goto dequant_done;
          const uint8_t* ws = smem + off_w + sw * FF_WSTAGE;
          uint4 pk[FF_BLOCKS][2];
          uint32_t sbw[FF_BLOCKS];
#pragma unroll
          for (int bb = 0; bb < FF_BLOCKS; ++bb) {
            const uint8_t* blk = ws + bb * W_BLOCK;
            pk[bb][0] = *reinterpret_cast<const uint4*>(blk + L * 16);
            pk[bb][1] = *reinterpret_cast<const uint4*>(blk + 2048 + L * 16);
            sbw[bb] = *reinterpret_cast<const uint32_t*>(blk + W_PACKED + L * 4);
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(FB_WEMPTY + sw));  // this warp's rows are in registers
          uint32_t v0[2][32];
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) expand_group(pk[bb][0], pk[bb][1], sbw[bb], v0[bb]);
          if (it >= FF_NA &&
              !wait_warp(bar(FB_AEMPTY + sa), ((it / FF_NA) - 1) & 1, s_abort, p.err, lim, p.sleep_ns))
            goto dequant_done;
          const uint32_t ta = trow + static_cast<uint32_t>(sa * FF_ACOLS);
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) ptx::tmem_st_32x32b_x32(ta + bb * 32, v0[bb]);
#pragma unroll
          for (int bb = 2; bb < FF_BLOCKS; ++bb) {
            uint32_t v[32];
            expand_group(pk[bb][0], pk[bb][1], sbw[bb], v);
            ptx::tmem_st_32x32b_x32(ta + bb * 32, v);
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(FB_AFULL + sa));
        }
      }
    }
  dequant_done:;
  } else {
    // ------------------------------------------------ epilogue: h into the h buffer, y to global memory
    const int q = warp & 3;
    const int e = threadIdx.x - 12 * 32;  // 0..127
    const int cc = e & 15, rr = e >> 4;    // 16-byte column chunk, first row of this thread's copies
    int sbuf = 0;
    int ui = 0, tc = 0;
    for (int b = blockIdx.x; b < nb; b += gridDim.x) {
      Tile t;
      if (!ff_tile(p, b, &t)) {
        if (threadIdx.x == 12 * 32) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
        continue;
      }
      const int N = round16(t.rows);
      for (int j = 0; j < SU; ++j) {
        const bool gu = j < NG;
        const int d = ui & 1;
        bool ok = wait_warp(bar(FB_DFULL + d), (ui >> 1) & 1, s_abort, p.err, lim, p.sleep_ns);
        if (!ptx::named_bar_and(FF_EPI_BAR, 128, ok)) goto epi_done;
        // the previous tile's down MMAs are done with the h buffer before this tile's h is written
        if (j == 0 && tc > 0) {
          ok = wait_warp(bar(FB_HFREE), (tc - 1) & 1, s_abort, p.err, lim, p.sleep_ns);
          if (!ptx::named_bar_and(FF_EPI_BAR, 128, ok)) goto epi_done;
        }
        ptx::tc_fence_after();
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(d * 2 * DM);
        for (int c0 = 0; c0 < N; c0 += FF_EPI_ROWS, sbuf ^= 1) {
          uint16_t* st = s_stage + sbuf * (FF_EPI_ROWS * TC_M);
          if (gu) {
            uint32_t g[32], uu[32];
            ptx::tmem_ld_32x32b_x32(tq + c0, g);
            ptx::tmem_ld_32x32b_x32(tq + DM + c0, uu);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              st[jj * TC_M + 32 * q + lane] =
                  float_to_bf16_bits(silu_fast(__uint_as_float(g[jj])) * __uint_as_float(uu[jj]));
          } else {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tq + c0, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) st[jj * TC_M + 32 * q + lane] = float_to_bf16_bits(__uint_as_float(v[jj]));
          }
          ptx::named_bar_sync(FF_EPI_BAR, 128);
          const uint4* src = reinterpret_cast<const uint4*>(st) + cc;
#pragma unroll
          for (int r = rr; r < FF_EPI_ROWS; r += 8) {
            const int row = c0 + r;
            if (row >= t.rows) continue;
            if (gu) {
              // features 128j + 8cc .. + 7 of tile row `row`: h atom 2j + cc / 8, 16-byte chunk cc % 8,
              // 128-byte swizzle of the row within its group of eight
              const int a = 2 * j + (cc >> 3), c8 = cc & 7;
              uint8_t* hd = smem + off_h + static_cast<uint32_t>(a) * atom + (row >> 3) * 1024 + (row & 7) * 128 +
                            ((c8 ^ (row & 7)) << 4);
              *reinterpret_cast<uint4*>(hd) = src[r * 16];
            } else {
              uint16_t* yd = p.y + static_cast<size_t>(t.row0 + row) * p.H + TC_M * (j - NG) + 8 * cc;
              *reinterpret_cast<uint4*>(yd) = src[r * 16];
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(FB_DEMPTY + d));  // the accumulator is free
        if (gu && j == NG - 1) {
          ptx::fence_proxy_async_smem();  // this thread's h stores, before the tensor core reads them
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(FB_HREADY));
        }
        ++ui;
      }
      ++tc;
    }
  epi_done:;
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*s_abort && warp == 0 && lane == 0) {
    // after a timeout some weight copies may never have been consumed: let them land first
    for (int t = prod_w - NW < 0 ? 0 : prod_w - NW; t < prod_w; ++t)
      wait_drain(bar(FB_WFULL + t % NW), (t / NW) & 1, lim);
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, FF_TMEM_COLS);
  }
}

namespace {

int ffn_max_dyn_smem() {
  static int v = 0;
  if (!v) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (v <= 0) v = 232448;
  }
  return v;
}

}  // namespace

unsigned long long wait_limit_ns();

// Needs bn <= 64, H % 128 == 0 and F % 256 == 0 (checked by the caller too).
cudaError_t launch_ffn_tc(const uint16_t* x, int T, int H, int F, int E, int k, const void* w13, const void* w2,
                          const int32_t* perm, const int32_t* block_map, const int32_t* num_blocks, int bn, int cap,
                          uint16_t* y, int num_sms, cudaStream_t s) {
  const int boxr = (bn + 15) & ~15;
  if (boxr > FF_MAX_ROWS || H % TC_M != 0 || F % (4 * KG) != 0) return cudaErrorInvalidValue;
  FfParams prm;
  prm.x = x;
  prm.w13 = static_cast<const uint8_t*>(w13);
  prm.w2 = static_cast<const uint8_t*>(w2);
  prm.perm = perm;
  prm.block_map = block_map;
  prm.num_blocks = num_blocks;
  prm.y = y;
  prm.err = device_error_ptr();
  const unsigned long long ns = wait_limit_ns();
  prm.wait_cycles = ns > (~0ull) / 3 ? ~0ull : ns * 21 / 10;
  prm.sleep_ns = ns < 20000ull ? static_cast<uint32_t>(ns > 0 ? ns : 1) : 20000u;
  prm.T = T;
  prm.H = H;
  prm.F = F;
  prm.E = E;
  prm.k = k;
  prm.bn = bn;
  prm.cap = cap;
  prm.boxr = boxr;
  prm.sb = 2 * boxr * 128;
  const int hbytes = (F / KG) * boxr * 128;
  const int fixed = FF_BAR_BYTES + FF_MISC + FF_STAGE_BYTES;
  const int total = ffn_max_dyn_smem() - 1024 - fixed - hbytes;
  int nbs = 0, nws = 0;
  for (int want = 3; want >= 2 && nws < 4; --want) {
    nbs = want;
    nws = (total - nbs * prm.sb) / FF_WSTAGE;
  }
  if (nws < 4 || nbs < 2) return cudaErrorInvalidValue;
  if (nws > FF_NWMAX) nws = FF_NWMAX;
  nws &= ~1;  // each dequant warpgroup keeps its own slots (stage it: slot it % NW, warpgroup it % 2)
  nbs = (total - nws * FF_WSTAGE) / prm.sb;
  if (nbs > FF_NBMAX) nbs = FF_NBMAX;
  prm.nb = nbs;
  prm.nw = nws;
  // TMEM: two accumulator buffers of two M-tiles (4 boxr <= 256 columns), then two A slots of 128
  if (4 * boxr + FF_NA * FF_ACOLS > FF_TMEM_COLS) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(nbs) * prm.sb + hbytes + static_cast<size_t>(nws) * FF_WSTAGE + fixed + 1024;
  const cudaError_t ea = ensure_dyn_smem(reinterpret_cast<const void*>(ffn_tc_kernel), smem);
  if (ea != cudaSuccess) return ea;
  ffn_tc_kernel<<<num_sms, FF_THREADS, smem, s>>>(prm);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
