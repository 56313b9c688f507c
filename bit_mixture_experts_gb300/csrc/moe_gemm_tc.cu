// Tensor-core grouped expert GEMM over groupwise-affine 4-bit weights for
// sm_103a (tcgen05 + TMEM), with the dequantisation fused into the GEMM.
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details,
// Prefill optimizations bullet: 4-bit weights in groups of 64 are expanded
// inside the grouped GEMM and accumulated in FP32; the itinai.com post on the
// same engine (paragraph 2) adds that the expanded bf16 weights never exist as
// a full copy in memory.  The pages' Metal kernel expands them in threadgroup
// memory with 32-row tiles and four simdgroups; on GB300 the expanded tile goes
// to tensor memory instead, where the MMA reads it directly, so shared-memory
// bandwidth is left to the activations:
//
//   D[m, n] = sum_k W[m, k] * X[n, k]      (swap-AB: weight rows on M, tokens on N)
//
//   M = 128 weight rows of one expert (one "M-tile"), N = the tile's token
//   rows rounded up to 16 (<= 128), K = 16 per MMA; a pipeline stage covers
//   two quant groups (K = 128), four in the one-M-tile down GEMM.
//
// Roles (512 threads, one CTA per SM, persistent over work units = (block-map
// tile, group of MG M-tiles), taken round-robin).
// Warps 0-2 run their loops converged with warp-uniform operands and let
// elect.sync pick the lane that issues each copy, MMA or commit:
//   warp 0      streams the packed weights into a shared-memory ring with
//               cp.async.bulk: one copy per M-tile and stage (the stage's
//               quant groups of an M-tile are contiguous), completion counted
//               in bytes on the slot's mbarrier
//   warp 1      allocates TMEM; issues tcgen05.mma (A from TMEM, B from smem)
//   warps 2-3   load the tile's activation rows into 128B-swizzled smem:
//               gate/up gathers the token rows of x with cp.async (16 bytes
//               per copy, completion counted on the stage's mbarrier);
//               down: warp 2 loads tiles of contiguous h rows with TMA
//   warps 4-11  two dequant warpgroups (alternate stages): nibbles -> bf16
//               w = bf16(q*scale + bias) with one fma.rn.bf16x2 per pair,
//               written to TMEM with tcgen05.st
//   warps 12-15 epilogue: tcgen05.ld of the FP32 accumulators, then
//               gate/up: the unit's two M-tiles are the gate and the up rows
//                        of the same 128 features, so each thread holds g and
//                        u of its feature: h = bf16(silu(g) * u) -> h[row, f]
//               down:    y = bf16(acc) -> y[row, channel]
//               staged 32 rows at a time in shared memory and written as
//               whole 256-byte row segments
//
// Every mbarrier wait is bounded by a time limit; on expiry the kernel records
// MOE_DEV_TIMEOUT in the device error word, every role leaves its loop, copies
// in flight are drained, TMEM is freed and the kernel returns.
#include <cuda.h>
#include <string.h>

#include "moe_common.cuh"
#include "moe_ptx.cuh"
#include "moe_tc_dev.cuh"
#include "moe_tmap.cuh"

namespace moe {

using namespace tc_dev;

namespace {

constexpr int NWMAX = 12;              // packed-weight ring slots (run-time depth, at least 4)
constexpr int NAMAX = 4;               // dequantised-weight ring (TMEM), run-time depth 2 to 4
constexpr int NBMAX = 12;              // activation ring (smem), run-time depth 2 to NBMAX
constexpr int TMEM_COLS = 512;        // accumulators first, then the A ring
constexpr int NTHREADS = 512;
constexpr int GATHER_T = 64;           // threads gathering activation rows (gate/up)

// barrier indices
constexpr int BAR_WFULL = 0;
constexpr int BAR_WEMPTY = BAR_WFULL + NWMAX;
constexpr int BAR_AFULL = BAR_WEMPTY + NWMAX;
constexpr int BAR_AEMPTY = BAR_AFULL + NAMAX;
constexpr int BAR_BFULL = BAR_AEMPTY + NAMAX;
constexpr int BAR_BEMPTY = BAR_BFULL + NBMAX;
constexpr int BAR_DFULL = BAR_BEMPTY + NBMAX;
constexpr int BAR_DEMPTY = BAR_DFULL + 2;
constexpr int BAR_FIN = BAR_DEMPTY + 2;
constexpr int NBAR = BAR_FIN + 1;

// smem layout (offsets from a 1024-byte aligned base): B ring | W ring | barriers | misc
constexpr int BAR_BYTES = (NBAR * 8 + 15) & ~15;
constexpr int MISC_BYTES = 16;  // abort flag, TMEM base
constexpr int EPI_ROWS = 32;     // output rows per epilogue chunk (one tcgen05.ld x32)
constexpr int STAGE_BYTES = 2 * EPI_ROWS * TC_M * 2;  // epilogue staging: two chunks of 32 rows x 128 bf16
constexpr int COMB_MAX = 2 * TC_M;      // (token, channel block) pairs one down unit can complete
constexpr int COMB_BYTES = 16 + 4 * COMB_MAX;  // their count and list (down GEMM with the combine)
constexpr int EPI_BAR = 1;       // named barrier of the four epilogue warps

// Pre-expanded weights (the unfused comparison path, moe_expand_w4): per
// (matrix, M-tile, K group) one block of 128 rows x 64 bf16; the 16-byte
// chunk i of row L sits at chunk position i ^ (L & 7), so that the 32 rows a
// warp reads at once fall in different banks.
constexpr int RAW_BLOCK = TC_M * KG * 2;

// Sizes that depend on MG, the M-tiles per work unit (they share each
// activation stage), GPS, the quant groups per pipeline stage, and RAW (the
// weights arrive already expanded to bf16).  The ring depths are chosen at
// launch from the shared memory available.
template <int MG, int GPS, bool RAW = false>
struct UnitCfg {
  static constexpr int WB = RAW ? RAW_BLOCK : W_BLOCK;       // bytes of one (M-tile, K group) block
  static constexpr int W_STAGE = MG * GPS * WB;              // weights of one stage
  static constexpr int A_COLS = MG * GPS * 32;               // TMEM columns of one dequantised stage
  static_assert((GPS * WB) % 16 == 0, "bulk copies move multiples of 16 bytes");
};


struct TcParams {
  const uint16_t* act;
  const uint8_t* w;
  const int32_t* perm;
  const float* topk_w;
  const int32_t* block_map;
  const int32_t* num_blocks;
  void* out;
  // down GEMM with the combine (null otherwise): the token order output, the routing's inverse
  // permutation, and one counter per (token, 128-channel block), zero when the call begins
  uint16_t* cmb_out;
  const int32_t* inv_perm;
  int* cmb_cnt;
  int* err;
  unsigned long long wait_cycles;
  uint32_t sleep_ns;  // suspend hint of the waits: min(20 us, the wait limit)
  int T, H, F, E, k, bn, cap;
  int boxr;     // activation rows per stage buffer (block_n rounded up to 16, <= 128)
  int nb;       // activation ring depth
  int nw;       // packed-weight ring depth
  int sb;       // bytes of one activation stage: one atom of boxr rows x 128 bytes per quant group
  int nd;       // accumulator buffers
  int dm;       // TMEM columns of one M-tile's accumulator (= boxr)
  int na;       // A ring depth
  int a0;       // first TMEM column of the A ring
};

// Unit u = (block-map tile u / MGT, M-group u % MGT).  False for a malformed
// entry (the same decision in every role, so all roles skip it together).
__device__ __forceinline__ bool unit_tile(const TcParams& p, int u, int MGT, Tile* t, int* grp) {
  const int b = u / MGT;
  *grp = u - b * MGT;
  t->expert = __ldg(p.block_map + 3 * b);
  t->row0 = __ldg(p.block_map + 3 * b + 1);
  t->rows = __ldg(p.block_map + 3 * b + 2);
  const int A = p.T * p.k;
  bool ok = t->expert >= 0 && t->expert <= p.E && t->rows >= 1 && t->rows <= p.bn && t->row0 >= 0;
  if (ok) ok = t->expert < p.E ? (t->row0 + t->rows <= A) : (t->row0 >= A && t->row0 + t->rows <= A + p.T);
  return ok;
}

}  // namespace

// Work unit: one block-map tile (<= 128 token rows) x MG M-tiles (MG x 128
// weight rows) of one expert.  Each pipeline stage covers GPS quant groups
// (K = 64 GPS): the M-tiles' packed blocks, their dequantised bf16 in TMEM and
// one activation stage read by every M-tile's MMAs.  Gate/up always takes
// MG = 2 (the gate and the up M-tile of the same features); the down GEMM takes
// MG = 1 for tiles of more than 64 rows, so that two accumulator buffers still
// fit in TMEM and the epilogue of one unit overlaps the next unit's mainloop,
// and then GPS = 4 so that a stage still carries 16 MMAs.
//
// Rings (full/empty mbarriers; stage index = running stage count `it` modulo
// the ring depth):
//   W  packed 4-bit blocks, smem, bulk copies by warp 0 -> dequant warps
//      (freed as soon as a warp has its rows in registers)
//   A  dequantised bf16 weights, TMEM, dequant warps -> MMA (warp 1)
//   B  activation rows, 128B-swizzled K-major atoms of 64 K, smem,
//      gate/up: cp.async gather of token rows (warps 2-3),
//      down: TMA tiles of contiguous h rows (warp 2)  -> MMA
//   D  FP32 accumulators, TMEM, MMA -> epilogue (1 or 2 buffers)
template <int MODE, int MG, int GPS, bool RAW = false>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tmap_act) {
  static_assert(MODE == 1 || MG == 2, "gate/up pairs the gate and the up M-tile in one unit");
  static_assert(MG == 1 || MG == 2, "one or two M-tiles per unit");
  static_assert(GPS == 2 || (GPS == 4 && MODE == 1 && MG == 1), "2-group stages, or 4 for the one-M-tile down GEMM");
  constexpr int W_STAGE = UnitCfg<MG, GPS, RAW>::W_STAGE;
  constexpr int A_COLS = UnitCfg<MG, GPS, RAW>::A_COLS;
  constexpr int WB = UnitCfg<MG, GPS, RAW>::WB;
  const int NW = p.nw;
  const int W_RING_BYTES = NW * W_STAGE;
  constexpr int KS = KG * GPS;               // K per stage
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int NB = p.nb, SB = p.sb, ND = p.nd, BOXR = p.boxr, NA = p.na;
  const uint32_t atom_bytes = static_cast<uint32_t>(BOXR) * 128u;
  const uint32_t off_w = static_cast<uint32_t>(NB * SB);
  const uint32_t bar0 = sbase + off_w + W_RING_BYTES;
  auto bar = [bar0](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + off_w + W_RING_BYTES + BAR_BYTES);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + off_w + W_RING_BYTES + BAR_BYTES + 4);
  uint16_t* s_stage = reinterpret_cast<uint16_t*>(smem + off_w + W_RING_BYTES + BAR_BYTES + MISC_BYTES);
  int* s_ncomb = reinterpret_cast<int*>(smem + off_w + W_RING_BYTES + BAR_BYTES + MISC_BYTES + STAGE_BYTES);
  int* s_comb = s_ncomb + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = MODE == 0 ? p.H : p.F;
  const int KT = K / KG;                     // quant groups along K
  const int NS = K / KS;                     // stages per unit
  const int MT = MODE == 0 ? (2 * p.F) / TC_M : p.H / TC_M;
  const int MGT = (MT + MG - 1) / MG;        // M-groups per tile
  const int A = p.T * p.k;
  const int DM = p.dm;                       // columns per M-tile accumulator
  const int DBUF = MG * DM;                  // columns per accumulator buffer
  const uint32_t A0 = static_cast<uint32_t>(p.a0);
  int nb = __ldg(p.num_blocks);
  if (nb < 0 || nb > p.cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
    nb = nb < 0 ? 0 : p.cap;
  }
  const int units = nb * MGT;

  if (threadIdx.x == 0) {
    *s_abort = 0;
    for (int s = 0; s < NWMAX; ++s) {
      ptx::mbar_init(bar(BAR_WFULL + s), 1);
      ptx::mbar_init(bar(BAR_WEMPTY + s), 4);
    }
    for (int s = 0; s < NAMAX; ++s) {
      ptx::mbar_init(bar(BAR_AFULL + s), 4);
      ptx::mbar_init(bar(BAR_AEMPTY + s), 1);
    }
    for (int s = 0; s < NBMAX; ++s) {
      ptx::mbar_init(bar(BAR_BFULL + s), MODE == 0 ? GATHER_T : 1);
      ptx::mbar_init(bar(BAR_BEMPTY + s), 1);
    }
    for (int d = 0; d < 2; ++d) {
      ptx::mbar_init(bar(BAR_DFULL + d), 1);
      ptx::mbar_init(bar(BAR_DEMPTY + d), 4);
    }
    ptx::mbar_init(bar(BAR_FIN), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const unsigned long long lim = p.wait_cycles;
  int prod_b = 0;  // activation TMA stages issued (down), for the drain after a timeout
  int prod_w = 0;  // weight stages issued, for the drain after a timeout

  if (warp == 0) {
    // ------------------------------------------------ weight producer: bulk copies into the W ring
    int& it = prod_w;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      Tile t;
      int grp;
      if (!unit_tile(p, u, MGT, &t, &grp)) continue;
      const int nm = min(MG, MT - grp * MG);
      const uint8_t* g0 = p.w + (static_cast<size_t>(t.expert) * MT + grp * MG) * KT * static_cast<size_t>(WB);
      for (int ks = 0; ks < NS; ++ks, ++it) {
        const int s = it % NW, r = it / NW;
        if (r > 0 && !wait_warp(bar(BAR_WEMPTY + s), (r - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) goto wprod_done;
        const uint32_t dst = sbase + off_w + s * W_STAGE;
        ptx::mbar_arrive_expect_tx_elect(bar(BAR_WFULL + s), static_cast<uint32_t>(nm * GPS * WB));
        for (int m = 0; m < nm; ++m)
          ptx::bulk_g2s_elect(dst + m * GPS * WB, g0 + (static_cast<size_t>(m) * KT + ks * GPS) * WB, GPS * WB,
                              bar(BAR_WFULL + s));
      }
    }
  wprod_done:;
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp, one lane issues)
    // The issue sequence is kept branch-free and fully unrolled with warp-uniform
    // operands: a data-dependent branch or a run-time trip count around the
    // elect.sync'ed MMAs multiplies their issue cost.
    int ui = 0;
    int sa = 0, pa = 0, sb = 0, pb = 0;  // ring slots and phases
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      Tile t;
      int grp;
      if (!unit_tile(p, u, MGT, &t, &grp)) continue;
      const bool two = MG == 2 && grp * MG + 1 < MT;
      const uint32_t idesc = ptx::idesc_bf16_f32(TC_M, round16(t.rows));
      const int d = ui % ND, rd = ui / ND;
      if (rd > 0 && !wait_warp(bar(BAR_DEMPTY + d), (rd - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
      ptx::tc_fence_after();
      const uint32_t d0 = tmem + d * DBUF, d1 = d0 + DM;
      for (int ks = 0; ks < NS; ++ks) {
        if (!wait_warp(bar(BAR_AFULL + sa), pa, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
        if (!wait_warp(bar(BAR_BFULL + sb), pb, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
        if (MODE == 0) ptx::fence_proxy_async_smem();  // cp.async-written rows, read by the tensor core
        ptx::tc_fence_after();
        const uint32_t a0 = tmem + A0 + sa * A_COLS;
        const uint32_t b0 = sbase + sb * SB;
        const uint32_t acc0 = ks != 0;
        // A columns of the stage: M-tile m, quant group g at m * GPS * 32 + g * 32;
        // group g's activations are B atom g (K = 64, four K16 steps)
        if (two) {
#pragma unroll
          for (int g = 0; g < GPS; ++g)
            ptx::mma_group_ts_elect<true>(d0, d1, a0 + g * 32, a0 + GPS * 32 + g * 32,
                                          ptx::smem_desc_sw128(b0 + g * atom_bytes), idesc, g == 0 ? acc0 : 1u);
        } else {
#pragma unroll
          for (int g = 0; g < GPS; ++g)
            ptx::mma_group_ts_elect<false>(d0, d0, a0 + g * 32, a0 + g * 32, ptx::smem_desc_sw128(b0 + g * atom_bytes),
                                           idesc, g == 0 ? acc0 : 1u);
        }
        ptx::mma_commit_elect(bar(BAR_AEMPTY + sa));
        ptx::mma_commit_elect(bar(BAR_BEMPTY + sb));
        if (++sa == NA) {
          sa = 0;
          pa ^= 1;
        }
        if (++sb == NB) {
          sb = 0;
          pb ^= 1;
        }
      }
      ptx::mma_commit_elect(bar(BAR_DFULL + d));
      ++ui;
    }
  mma_done:
    ptx::mma_commit_elect(bar(BAR_FIN));
    if (lane == 0) wait_drain(bar(BAR_FIN), 0, lim);
    __syncwarp();
  } else if (warp < 4) {
    if (MODE == 1) {
      // ------------------------------------------------ activation producer: TMA tiles of h rows
      if (warp == 2) {
        int& it = prod_b;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
          Tile t;
          int grp;
          if (!unit_tile(p, u, MGT, &t, &grp)) continue;
          for (int ks = 0; ks < NS; ++ks, ++it) {
            const int s = it % NB, r = it / NB;
            if (r > 0 && !wait_warp(bar(BAR_BEMPTY + s), (r - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) goto bprod_done;
            const uint32_t dst = sbase + s * SB;
            ptx::mbar_arrive_expect_tx_elect(bar(BAR_BFULL + s), static_cast<uint32_t>(SB));
            for (int a = 0; a < GPS; ++a)
              ptx::tma_load_2d_elect(dst + a * atom_bytes, &tmap_act, ks * KS + a * KG, t.row0, bar(BAR_BFULL + s));
          }
        }
      bprod_done:;
      }
    } else {
      // ------------------------------------------------ activation gather: token rows of x by cp.async
      const int gt = threadIdx.x - 64;  // 0..63
      const int chunk = gt & 7, row_a = gt >> 3;
      int it = 0;
      bool aborted = false;
      for (int u = blockIdx.x; u < units && !aborted; u += gridDim.x) {
        Tile t;
        int grp;
        if (!unit_tile(p, u, MGT, &t, &grp)) continue;
        // token row of tile rows row_a + 8j: all permutation entries are loaded
        // first (independent loads, one round trip), then checked
        int tok[128 / 8];
#pragma unroll
        for (int j = 0; j < 128 / 8; ++j) {
          const int i = row_a + 8 * j;
          const int r = t.row0 + i;
          tok[j] = (i < t.rows && r < A) ? __ldg(p.perm + r) : 0;
        }
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 128 / 8; ++j) {
          const int i = row_a + 8 * j;
          const int r = t.row0 + i;
          int tk = -1;
          if (i < t.rows) {
            if (r >= A) tk = r - A;  // shared-expert rows follow the routed ones, in token order
            else if (tok[j] >= 0 && tok[j] < A) tk = tok[j] / p.k;
            else bad = true;
          }
          tok[j] = tk;
        }
        if (bad) set_device_error(p.err, MOE_DEV_BAD_INDEX);
        for (int ks = 0; ks < NS; ++ks, ++it) {
          const int s = it % NB, r = it / NB;
          if (r > 0 && !wait_warp(bar(BAR_BEMPTY + s), (r - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) {
            aborted = true;
            break;
          }
          const uint32_t dst0 = sbase + s * SB;
#pragma unroll
          for (int j = 0; j < 128 / 8; ++j) {
            const int i = row_a + 8 * j;
            if (tok[j] >= 0) {
              const uint16_t* src = p.act + static_cast<size_t>(tok[j]) * K + ks * KS + chunk * 8;
              const uint32_t dst = dst0 + (i >> 3) * 1024 + (i & 7) * 128 + ((chunk ^ (i & 7)) << 4);
#pragma unroll
              for (int g = 0; g < GPS; ++g) ptx::cp_async_16(dst + g * atom_bytes, src + g * KG);
            }
          }
          // the barrier counts one arrival per gather thread, made by the hardware
          // once this thread's copies of the stage have landed
          ptx::cp_async_mbar_arrive(bar(BAR_BFULL + s));
        }
      }
      ptx::cp_async_wait_all();
    }
  } else if (warp < 12) {
    // ------------------------------------------------ dequant: warpgroup wg expands the stages it with
    // it % 2 == wg (every M-tile of the stage), so one warpgroup computes while
    // the other waits.  Each thread owns one weight row of each M-tile (= its
    // TMEM lane).  It loads its rows of the stage from the W ring into
    // registers, frees the slot, expands the first M-tile's groups and only
    // then waits for the A slot, so that part of the arithmetic overlaps the
    // MMAs still reading the slot.
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int L = 32 * q + lane;  // weight row within each M-tile = TMEM lane
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16) + A0;
    int it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      Tile t;
      int grp;
      if (!unit_tile(p, u, MGT, &t, &grp)) continue;
      const int nm = min(MG, MT - grp * MG);
      for (int ks = 0; ks < NS; ++ks, ++it) {
        if ((it & 1) != wg) continue;
        const int sa = it % NA, sw = it % NW;
        if (!wait_warp(bar(BAR_WFULL + sw), (it / NW) & 1, s_abort, p.err, lim, p.sleep_ns)) goto dequant_done;
        const uint8_t* ws = smem + off_w + sw * W_STAGE;
        if (RAW) {
          // weights already expanded: this thread's row of every block goes to TMEM as it is
          if (it >= NA && !wait_warp(bar(BAR_AEMPTY + sa), ((it / NA) - 1) & 1, s_abort, p.err, lim, p.sleep_ns))
            goto dequant_done;
          const uint32_t ta = trow + sa * A_COLS;
#pragma unroll
          for (int m = 0; m < MG; ++m) {
            if (m >= nm) break;
#pragma unroll
            for (int g = 0; g < GPS; ++g) {
              const uint4* row = reinterpret_cast<const uint4*>(ws + (m * GPS + g) * WB + L * 128);
              uint32_t v[32];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint4 c = row[i ^ (L & 7)];
                v[4 * i] = c.x;
                v[4 * i + 1] = c.y;
                v[4 * i + 2] = c.z;
                v[4 * i + 3] = c.w;
              }
              ptx::tmem_st_32x32b_x32(ta + m * GPS * 32 + g * 32, v);
            }
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(BAR_WEMPTY + sw));  // the rows are in registers (and stored)
        } else {
        uint4 pk[MG][GPS][2];
        uint32_t sbw[MG][GPS];
#pragma unroll
        for (int m = 0; m < MG; ++m)
#pragma unroll
          for (int g = 0; g < GPS; ++g) {
            const uint8_t* blk = ws + (m * GPS + g) * WB;
            if (m < nm) {
              pk[m][g][0] = *reinterpret_cast<const uint4*>(blk + L * 16);
              pk[m][g][1] = *reinterpret_cast<const uint4*>(blk + 2048 + L * 16);
              sbw[m][g] = *reinterpret_cast<const uint32_t*>(blk + W_PACKED + L * 4);
            }
          }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(BAR_WEMPTY + sw));  // this warp's rows are in registers
        constexpr int PRE = GPS < 2 ? GPS : 2;  // groups expanded before the A slot is free
        uint32_t v0[PRE][32];
#pragma unroll
        for (int g = 0; g < PRE; ++g) expand_group(pk[0][g][0], pk[0][g][1], sbw[0][g], v0[g]);
        if (it >= NA && !wait_warp(bar(BAR_AEMPTY + sa), ((it / NA) - 1) & 1, s_abort, p.err, lim, p.sleep_ns))
          goto dequant_done;
        const uint32_t ta = trow + sa * A_COLS;
#pragma unroll
        for (int g = 0; g < PRE; ++g) ptx::tmem_st_32x32b_x32(ta + g * 32, v0[g]);
#pragma unroll
        for (int m = 0; m < MG; ++m) {
          if (m >= nm) break;
#pragma unroll
          for (int g = m == 0 ? PRE : 0; g < GPS; ++g) {
            uint32_t v[32];
            expand_group(pk[m][g][0], pk[m][g][1], sbw[m][g], v);
            ptx::tmem_st_32x32b_x32(ta + m * GPS * 32 + g * 32, v);
          }
        }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(BAR_AFULL + sa));
      }
    }
  dequant_done:;
  } else {
    // ------------------------------------------------ epilogue
    // Chunks of 32 output rows: each thread converts its lane's 32 values
    // (one feature or channel, 32 rows) into a shared-memory tile of 32 rows
    // x 128 columns; after a barrier of the four warps the tile goes out as
    // whole 256-byte row segments, 16 bytes per thread (two staging buffers,
    // so one barrier per chunk).  The four warps agree on every accumulator
    // wait (AND-reduction barrier), so none is left waiting at a barrier.
    const int q = warp & 3;
    const int e = threadIdx.x - 12 * 32;  // 0..127
    const int cc = e & 15, rr = e >> 4;    // 16-byte column chunk, first row of this thread's copies
    int sbuf = 0;
    int ui = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      Tile t;
      int grp;
      if (!unit_tile(p, u, MGT, &t, &grp)) {
        if (threadIdx.x == 12 * 32) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
        continue;
      }
      const int nm = min(MG, MT - grp * MG);
      const int d = ui % ND;
      const bool ok = wait_warp(bar(BAR_DFULL + d), (ui / ND) & 1, s_abort, p.err, lim, p.sleep_ns);
      if (!ptx::named_bar_and(EPI_BAR, 128, ok)) break;
      ptx::tc_fence_after();
      const int N = round16(t.rows);
      const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16) + d * DBUF;  // this warp's lanes
      for (int m = 0; m < (MODE == 0 ? 1 : nm); ++m) {
        // gate/up: M-tile 0 = gate rows, M-tile 1 = up rows of features 128 grp + (0..127);
        // down: lane = output channel 128 (grp MG + m) + (32 q + lane) of M-tile m
        const int col0 = TC_M * (grp * MG + m) / (MODE == 0 ? MG : 1);
        const int ld = MODE == 0 ? p.F : p.H;
        uint16_t* dst = static_cast<uint16_t*>(p.out) + static_cast<size_t>(t.row0) * ld + col0 + 8 * cc;
        for (int c0 = 0; c0 < N; c0 += EPI_ROWS, sbuf ^= 1) {
          uint16_t* st = s_stage + sbuf * (EPI_ROWS * TC_M);
          if (MODE == 0) {
            uint32_t g[32], uu[32];
            ptx::tmem_ld_32x32b_x32(tq + c0, g);
            ptx::tmem_ld_32x32b_x32(tq + DM + c0, uu);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              st[j * TC_M + 32 * q + lane] =
                  float_to_bf16_bits(silu_fast(__uint_as_float(g[j])) * __uint_as_float(uu[j]));
          } else {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tq + m * DM + c0, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j * TC_M + 32 * q + lane] = float_to_bf16_bits(__uint_as_float(v[j]));
          }
          ptx::named_bar_sync(EPI_BAR, 128);
          const uint4* src = reinterpret_cast<const uint4*>(st) + cc;
#pragma unroll
          for (int r = rr; r < EPI_ROWS; r += 8)
            if (c0 + r < t.rows) *reinterpret_cast<uint4*>(dst + static_cast<size_t>(c0 + r) * ld) = src[r * 16];
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(BAR_DEMPTY + d));  // the accumulator is free for the next unit
      if (MODE == 1 && p.cmb_out) {
        // The combine, fused: every (token, 128-channel block) counts its written y rows; the thread
        // whose row completes the k + 1 of a pair lists it, and the four warps combine the listed
        // pairs -- out = bf16(sum_j topk_w[t, j] y[row(t, j)] + y[shared row]), FP32 in moe_combine's
        // order -- while the MMAs of the next unit already run.  No thread waits for another CTA.
        const int NCB = p.H / TC_M;
        if (e == 0) *s_ncomb = 0;
        ptx::named_bar_sync(EPI_BAR, 128);
        __threadfence();  // the unit's y stores (all four warps', by the barrier) before this thread's counts
        for (int i = e; i < t.rows * nm; i += 128) {
          const int r = i % t.rows, m = i / t.rows;
          const int row = t.row0 + r;
          int tok = row - A;
          if (row < A) {
            const int a = __ldg(p.perm + row);
            tok = (a >= 0 && a < A) ? a / p.k : -1;
          }
          if (tok < 0) {
            set_device_error(p.err, MOE_DEV_BAD_INDEX);
            continue;
          }
          int* c = p.cmb_cnt + static_cast<size_t>(tok) * NCB + grp * MG + m;
          const int before = atomicAdd(c, 1);
          if (before == p.k) {
            __threadfence();  // the other CTAs' rows of this pair, before they are read
            *c = 0;           // left zero for the next call
            s_comb[atomicAdd(s_ncomb, 1)] = tok * NCB + grp * MG + m;
          } else if (before < 0 || before > p.k) {
            set_device_error(p.err, MOE_DEV_BAD_WORKSPACE);
          }
        }
        ptx::named_bar_sync(EPI_BAR, 128);
        const int ncomb = *s_ncomb;
        const uint16_t* yb = static_cast<const uint16_t*>(p.out);
        // half a warp per pair, eight channels per lane; a warp sums two pairs at a time, all of their
        // row loads issued before the sums
        const int half = lane >> 4, ch = 8 * (lane & 15);
        for (int i0 = 2 * q; i0 < ncomb; i0 += 8) {
          const int it2 = i0 + half;
          const bool live = it2 < ncomb;
          const int v = live ? s_comb[it2] : 0, tok = v / NCB, cb = v - tok * NCB;
          const size_t c0 = static_cast<size_t>(cb) * TC_M + ch;
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int j0 = 0; j0 <= p.k; j0 += 9) {
            uint4 yv[9];
            float wv[9];
#pragma unroll
            for (int b = 0; b < 9; ++b) {
              const int j = j0 + b;
              int row = -1;
              float w = 0.f;
              if (live && j < p.k) {
                row = __ldg(p.inv_perm + static_cast<size_t>(tok) * p.k + j);
                w = __ldg(p.topk_w + static_cast<size_t>(tok) * p.k + j);
              } else if (live && j == p.k) {
                row = A + tok;
                w = 1.0f;
              }
              const bool okr = live && j <= p.k && row >= 0 && row < A + p.T && (j == p.k || row < A);
              if (live && j <= p.k && !okr) set_device_error(p.err, MOE_DEV_BAD_INDEX);
              yv[b] = okr ? __ldcg(reinterpret_cast<const uint4*>(yb + static_cast<size_t>(row) * p.H + c0))
                          : make_uint4(0u, 0u, 0u, 0u);
              wv[b] = okr ? w : 0.f;
            }
#pragma unroll
            for (int b = 0; b < 9; ++b) {
              const uint32_t u4[4] = {yv[b].x, yv[b].y, yv[b].z, yv[b].w};
#pragma unroll
              for (int h2 = 0; h2 < 4; ++h2) {
                acc[2 * h2] = fmaf(wv[b], __uint_as_float(u4[h2] << 16), acc[2 * h2]);
                acc[2 * h2 + 1] = fmaf(wv[b], __uint_as_float(u4[h2] & 0xffff0000u), acc[2 * h2 + 1]);
              }
            }
          }
          if (live)
            *reinterpret_cast<uint4*>(p.cmb_out + static_cast<size_t>(tok) * p.H + c0) =
                make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                           pack_bf16x2(acc[6], acc[7]));
        }
      }
      ++ui;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*s_abort && MODE == 1 && warp == 2 && lane == 0) {
    // after a timeout some tile loads may never have been consumed: let them land before the CTA exits
    for (int t = prod_b - NB < 0 ? 0 : prod_b - NB; t < prod_b; ++t)
      wait_drain(bar(BAR_BFULL + t % NB), (t / NB) & 1, lim);
  }
  if (*s_abort && warp == 0 && lane == 0) {
    // the same for the weight copies
    for (int t = prod_w - NW < 0 ? 0 : prod_w - NW; t < prod_w; ++t)
      wait_drain(bar(BAR_WFULL + t % NW), (t / NW) & 1, lim);
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// --------------------------------------------------------------------------
// weight repack: canonical -> per (matrix, M-tile, K group) blocks of
// [2 halves][128 rows][4 words] packed nibbles + [128 rows] (scale, bias).
// Within a word the nibbles are reordered so that (word >> 4j) & 0x000f000f
// yields K elements 2j (low half) and 2j+1 (high half) of that word's eight.
// Gate/up M-tiles come in pairs (gate_up = 1): M-tile 2j holds the gate rows
// and M-tile 2j+1 the up rows of features 128j .. 128j+127 (needs F % 128 == 0);
// or interleaved (gate_up = 2, for the CTA-pair kernel): M-tile j holds the
// gate rows of features 64j .. 64j+63 in rows 0-63 and their up rows in rows
// 64-127.
// --------------------------------------------------------------------------
__global__ void repack_kernel(const uint32_t* __restrict__ packed, const uint16_t* __restrict__ scale,
                              const uint16_t* __restrict__ bias, int n_mat, int rows, int K, int gate_up,
                              uint8_t* __restrict__ out) {
  const int MT = rows / TC_M, KT = K / KG;
  const size_t total = static_cast<size_t>(n_mat) * MT * KT * TC_M;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int L = static_cast<int>(idx % TC_M);
    size_t rest = idx / TC_M;
    const int kg = static_cast<int>(rest % KT);
    rest /= KT;
    const int mt = static_cast<int>(rest % MT);
    const int mat = static_cast<int>(rest / MT);
    int row;
    if (gate_up == 2) {
      // interleaved: rows 0-63 of M-tile mt are the gate rows, rows 64-127 the up rows of
      // features 64 mt .. 64 mt + 63
      row = (L < TC_M / 2 ? 0 : rows / 2) + (TC_M / 2) * mt + (L & (TC_M / 2 - 1));
    } else if (gate_up) {
      row = (mt & 1) * (rows / 2) + TC_M * (mt >> 1) + L;
    } else {
      row = TC_M * mt + L;
    }
    const size_t crow = static_cast<size_t>(mat) * rows + row;
    uint8_t* blk = out + ((static_cast<size_t>(mat) * MT + mt) * KT + kg) * W_BLOCK;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint32_t in = packed[crow * (K / 8) + kg * 8 + w];
      uint32_t o = 0;
#pragma unroll
      for (int slot = 0; slot < 8; ++slot) {
        const int src = slot < 4 ? 2 * slot : 2 * (slot - 4) + 1;
        o |= ((in >> (4 * src)) & 0xfu) << (4 * slot);
      }
      *reinterpret_cast<uint32_t*>(blk + (w >> 2) * 2048 + L * 16 + (w & 3) * 4) = o;
    }
    const uint32_t sb = static_cast<uint32_t>(scale[crow * (K / 64) + kg]) |
                        (static_cast<uint32_t>(bias[crow * (K / 64) + kg]) << 16);
    *reinterpret_cast<uint32_t*>(blk + W_PACKED + L * 4) = sb;
  }
}

// --------------------------------------------------------------------------
// expansion of repacked 4-bit weights into a bf16 copy in the same tile order
// (the unfused path: what the fused kernels never write), blocks of 128 rows
// x 64 bf16 with row L's 16-byte chunk i at position i ^ (L & 7).
// --------------------------------------------------------------------------
__global__ void expand_kernel(const uint8_t* __restrict__ w4, size_t blocks, uint8_t* __restrict__ out) {
  const size_t total = blocks * TC_M;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int L = static_cast<int>(idx % TC_M);
    const size_t b = idx / TC_M;
    const uint8_t* blk = w4 + b * W_BLOCK;
    const uint4 p0 = *reinterpret_cast<const uint4*>(blk + L * 16);
    const uint4 p1 = *reinterpret_cast<const uint4*>(blk + 2048 + L * 16);
    const uint32_t sb = *reinterpret_cast<const uint32_t*>(blk + W_PACKED + L * 4);
    uint32_t v[32];
    expand_group(p0, p1, sb, v);
    uint4* row = reinterpret_cast<uint4*>(out + b * RAW_BLOCK + L * 128);
#pragma unroll
    for (int i = 0; i < 8; ++i) row[i ^ (L & 7)] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

size_t expanded_bytes(int n_mat, int rows, int K) {
  return static_cast<size_t>(n_mat) * (rows / TC_M) * (K / KG) * RAW_BLOCK;
}

cudaError_t launch_expand(const void* w4, int n_mat, int rows, int K, void* out, cudaStream_t s) {
  const size_t blocks = static_cast<size_t>(n_mat) * (rows / TC_M) * (K / KG);
  size_t grid = (blocks * TC_M + 255) / 256;
  if (grid > 65535) grid = 65535;
  expand_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(static_cast<const uint8_t*>(w4), blocks,
                                                            static_cast<uint8_t*>(out));
  note_launches(1);
  return cudaGetLastError();
}

size_t repacked_bytes(int n_mat, int rows, int K) {
  return static_cast<size_t>(n_mat) * (rows / TC_M) * (K / KG) * W_BLOCK;
}

cudaError_t launch_repack(const uint32_t* packed, const uint16_t* scale, const uint16_t* bias, int n_mat, int rows,
                          int K, int gate_up, void* out, cudaStream_t s) {
  const size_t total = static_cast<size_t>(n_mat) * (rows / TC_M) * (K / KG) * TC_M;
  size_t blocks = (total + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  repack_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(packed, scale, bias, n_mat, rows, K, gate_up,
                                                              static_cast<uint8_t*>(out));
  note_launches(1);
  return cudaGetLastError();
}

static unsigned long long g_wait_ns = 1000000000ull;

void set_wait_limit_ns(unsigned long long ns) { g_wait_ns = ns; }

unsigned long long wait_limit_ns() { return g_wait_ns; }

namespace {

int max_dyn_smem() {
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

cudaError_t launch_gemm_tc(int mode, const uint16_t* act, int T, int H, int F, int E, int k, const void* w,
                           const int32_t* perm, const float* topk_w, const int32_t* block_map,
                           const int32_t* num_blocks, int bn, int cap, void* out, int num_sms, cudaStream_t s,
                           bool raw, uint16_t* cmb_out, const int32_t* inv_perm, int* cmb_cnt) {
  TcParams prm;
  prm.cmb_out = cmb_out;
  prm.inv_perm = inv_perm;
  prm.cmb_cnt = cmb_cnt;
  prm.act = act;
  prm.w = static_cast<const uint8_t*>(w);
  prm.perm = perm;
  prm.topk_w = topk_w;
  prm.block_map = block_map;
  prm.num_blocks = num_blocks;
  prm.out = out;
  prm.err = device_error_ptr();
  // the limit is applied in SM cycles; 2.1 cycles per ns bounds the fastest SM clock
  prm.wait_cycles = g_wait_ns > (~0ull) / 3 ? ~0ull : g_wait_ns * 21 / 10;
  prm.sleep_ns = g_wait_ns < 20000ull ? static_cast<uint32_t>(g_wait_ns > 0 ? g_wait_ns : 1) : 20000u;
  prm.T = T;
  prm.H = H;
  prm.F = F;
  prm.E = E;
  prm.k = k;
  prm.bn = bn;
  prm.cap = cap;
  const int boxr = (bn + 15) & ~15;
  if (boxr > 128) return cudaErrorInvalidValue;
  prm.boxr = boxr;
  // M-tiles per unit: gate/up pairs gate and up; the down GEMM keeps two accumulator buffers
  const int MG = (mode == MOE_GATE_UP_SWIGLU || boxr <= 64) ? 2 : 1;
  // quant groups per stage: the one-M-tile down GEMM takes 4 (16 MMAs per stage, as the two-M-tile units)
  // (two for pre-expanded weights, whose four-group stages would not fit twice beside the activations)
  const int GPS = (MG == 1 && F % (4 * KG) == 0 && !raw) ? 4 : 2;
  prm.sb = GPS * boxr * 128;
  const int w_stage = (raw ? RAW_BLOCK : W_BLOCK) * MG * GPS;
  const int a_cols = MG == 2 ? UnitCfg<2, 2>::A_COLS : GPS == 4 ? UnitCfg<1, 4>::A_COLS : UnitCfg<1, 2>::A_COLS;
  const int fixed = BAR_BYTES + MISC_BYTES + STAGE_BYTES + COMB_BYTES;
  const int total = max_dyn_smem() - 1024 - fixed;
  // shared memory: three activation stages when that leaves four weight slots (else two), the
  // weight ring up to NWMAX slots, then more activation stages with what is left
  const int min_w = raw ? 2 : 4;  // pre-expanded stages are 3.6 times larger
  int nbs = 0, nws = 0;
  for (int want = 3; want >= 2 && nws < min_w; --want) {
    nbs = want;
    nws = (total - nbs * prm.sb) / w_stage;
  }
  if (nws < min_w || nbs < 2) return cudaErrorInvalidValue;
  if (nws > NWMAX) nws = NWMAX;
  // an even depth: stage it goes to slot it % NW and to dequant warpgroup it % 2, so every slot
  // keeps one warpgroup.  With an odd depth consecutive fills of a slot alternate between the
  // warpgroups, and one could wait for a slot's next fill while the other's fill before it is
  // still landing -- a parity wait cannot tell those two phases apart.
  nws &= ~1;
  nbs = (total - nws * w_stage) / prm.sb;
  if (nbs > NBMAX) nbs = NBMAX;
  prm.nb = nbs;
  prm.nw = nws;
  prm.dm = boxr;
  // TMEM: accumulators (nd buffers x MG M-tiles x boxr columns), then the A ring
  // a second accumulator buffer (the epilogue of one unit overlaps the next
  // unit's mainloop) when at least two A slots remain
  prm.nd = 2 * (MG * boxr) + 2 * a_cols <= TMEM_COLS ? 2 : 1;
  prm.a0 = prm.nd * MG * boxr;
  prm.na = (TMEM_COLS - prm.a0) / a_cols;
  if (prm.na > NAMAX) prm.na = NAMAX;
  const int smem = nbs * prm.sb + nws * w_stage + fixed + 1024;

  // activation tensor map (down only): tiles of boxr contiguous rows of h [A+T, F]
  CUtensorMap tmap;
  memset(&tmap, 0, sizeof(tmap));
  if (mode == MOE_DOWN) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const int A = T * k;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(F), static_cast<cuuint64_t>(A + T)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(F) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(boxr)};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(act), gdim, gstride, box,
                     estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  void (*kern)(const TcParams, const CUtensorMap) =
      raw ? (mode == MOE_GATE_UP_SWIGLU ? gemm_tc_kernel<0, 2, 2, true>
             : MG == 2                  ? gemm_tc_kernel<1, 2, 2, true>
             : GPS == 4                 ? gemm_tc_kernel<1, 1, 4, true>
                                        : gemm_tc_kernel<1, 1, 2, true>)
          : (mode == MOE_GATE_UP_SWIGLU ? gemm_tc_kernel<0, 2, 2>
             : MG == 2                  ? gemm_tc_kernel<1, 2, 2>
             : GPS == 4                 ? gemm_tc_kernel<1, 1, 4>
                                        : gemm_tc_kernel<1, 1, 2>);
  const cudaError_t ea = ensure_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<size_t>(smem));
  if (ea != cudaSuccess) return ea;
  kern<<<num_sms, NTHREADS, smem, s>>>(prm, tmap);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
