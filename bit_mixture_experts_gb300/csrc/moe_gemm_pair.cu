// Tensor-core grouped expert GEMM on CTA pairs (tcgen05 .cta_group::2) over
// groupwise-affine 4-bit weights, with the dequantisation fused into the GEMM.
//
// "Perplexity Open Sources Lily" (aitrending.vip), Technical Details,
// Prefill optimizations bullet: 4-bit weights in groups of 64 are expanded
// inside the grouped GEMM and accumulated in FP32; the itinai.com post on the
// same engine (paragraph 2) adds that the expanded bf16 weights never exist as
// a full copy in memory.
//
// The two CTAs of a cluster run on two SMs and compute one work unit
// together: 256 weight rows (an M-tile of 128 rows on each SM) times the
// tile's token rows (N = rows rounded up to 32, at most 256; each CTA holds
// N/2 of them):
//
//   D[m, n] = sum_k W[m, k] * X[n, k]      (swap-AB: weight rows on M, tokens on N)
//
// Each SM expands only its own 128 weight rows into its tensor memory (A),
// holds only half of the tile's activation rows in its shared memory (B rows
// 0 .. N/2-1 in the even CTA, N/2 .. N-1 in the odd one) and only its own 128
// accumulator rows (D, N columns).  The even CTA issues the M = 256 MMAs for
// both; completions are multicast to the barriers of both CTAs.  Per SM this
// halves the activation bytes per MMA (an SM with one M-tile of its own would
// otherwise need twice the shared-memory fill bandwidth) and keeps the
// accumulator at N columns, so that two accumulator buffers fit beside the A
// ring for tiles of up to 192 rows.
//
// Gate/up M-tiles are interleaved (the repacked layout with gate_up = 2): rows
// 0-63 of M-tile m are the gate rows and rows 64-127 the up rows of features
// 64m .. 64m+63, so each SM has g and u of its 64 features and SwiGLU needs no
// data from the other SM.
//
// Roles (512 threads per CTA, one CTA per SM):
//   warp 0      streams this SM's packed weights into its W ring (cp.async.bulk)
//   warp 1      allocates the pair's TMEM (one warp in each CTA); in the even
//               CTA it issues the pair MMAs, in the odd CTA it forwards the
//               completion of each activation stage to the even CTA's barrier
//   warps 2-3   load this CTA's half of the tile's activation rows (gate/up:
//               cp.async gather of token rows of x; down: TMA tiles of h rows)
//   warps 4-11  two dequant warpgroups (alternate stages): nibbles -> bf16 in
//               TMEM; arrive on the even CTA's A barrier
//   warps 12-15 epilogue of this SM's 128 accumulator rows (gate/up:
//               h = bf16(silu(g) u) through a shared-memory exchange between
//               the g and u warps; down: y = bf16(acc)); arrive on the even
//               CTA's accumulator barrier when the buffer is drained
//
// Every wait is bounded; on expiry the kernel records MOE_DEV_TIMEOUT, every
// role leaves its loop, copies and MMAs in flight are drained, and both CTAs
// meet at a final cluster barrier before the pair's TMEM is released.
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
constexpr int HALF_MAX = 128;          // activation rows per CTA (tiles of at most 256 rows)
constexpr int TMEM_COLS = 512;
constexpr int NTHREADS = 512;
constexpr int GATHER_T = 64;           // threads loading activation rows (gate/up)
constexpr int GU_F = TC_M / 2;         // gate/up: features per M-tile

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

constexpr int BAR_BYTES = (NBAR * 8 + 15) & ~15;
constexpr int MISC_BYTES = 16;   // abort flag, TMEM base
constexpr int EPI_ROWS = 32;     // accumulator columns (token rows) per epilogue chunk
constexpr int EPI_BAR = 1;       // named barrier of the four epilogue warps
constexpr int STAGE_BUF_DOWN = EPI_ROWS * TC_M * 2;                     // 32 rows x 128 channels bf16
constexpr int STAGE_BUF_GU = EPI_ROWS * GU_F * 4 + EPI_ROWS * GU_F * 2;  // u fp32, then h bf16
template <int MODE>
constexpr int stage_bytes() { return 2 * (MODE == 0 ? STAGE_BUF_GU : STAGE_BUF_DOWN); }

struct PairParams {
  const uint16_t* act;
  const uint8_t* w;
  const int32_t* perm;
  const int32_t* block_map;
  const int32_t* num_blocks;
  void* out;
  int* err;
  unsigned long long wait_cycles;
  uint32_t sleep_ns;  // suspend hint of the waits: min(20 us, the wait limit)
  int T, H, F, E, k, bn, cap;
  int half;     // activation rows per CTA and stage buffer (tile height rounded up to 32, halved)
  int nb, nw;   // activation and packed-weight ring depths
  int sb;       // bytes of one activation stage in one CTA
  int nd;       // accumulator buffers
  int dm;       // TMEM columns of one accumulator buffer (= 2 half)
  int na;       // A ring depth
  int a0;       // first TMEM column of the A ring
};

// The bounded waits (wait_warp, wait_drain) are moe_tc_dev.cuh's: a phase completed by arrivals
// from the other CTA of the pair is waited for the same way.

// Unit u = (block-map tile u / MGT, M-tile pair u % MGT).  False for a
// malformed entry (the same decision in every role of both CTAs).
__device__ __forceinline__ bool unit_tile(const PairParams& p, int u, int MGT, Tile* t, int* grp) {
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

// MMA width of a tile: its rows rounded up to 32 (16 per CTA of the pair).
__device__ __forceinline__ int round32(int n) { return (n + 31) & ~31; }

}  // namespace

template <int MODE, int GPS>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_pair_kernel(const PairParams p, const __grid_constant__ CUtensorMap tmap_act) {
  static_assert(GPS == 2 || GPS == 4, "two or four quant groups per stage");
  constexpr int W_STAGE = GPS * W_BLOCK;   // packed weights of one stage of this SM's M-tile
  constexpr int A_COLS = GPS * 32;         // TMEM columns of one dequantised stage
  constexpr int KS = KG * GPS;             // K per stage
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int NB = p.nb, NW = p.nw, SB = p.sb, ND = p.nd, NA = p.na, HALF = p.half;
  const uint32_t atom_bytes = static_cast<uint32_t>(HALF) * 128u;
  const uint32_t off_w = static_cast<uint32_t>(NB * SB);
  const uint32_t off_bar = off_w + static_cast<uint32_t>(NW * W_STAGE);
  const uint32_t bar0 = sbase + off_bar;
  auto bar = [bar0](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + off_bar + BAR_BYTES);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + off_bar + BAR_BYTES + 4);
  uint8_t* s_stage = smem + off_bar + BAR_BYTES + MISC_BYTES;

  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = static_cast<int>(ptx::cluster_id_x()), ncl = static_cast<int>(ptx::cluster_count_x());
  // the even CTA's barrier i, as a cluster address (the odd CTA's arrivals go there)
  auto lead_bar = [&](int i) -> uint32_t { return ptx::mapa_shared(bar(i), 0); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = MODE == 0 ? p.H : p.F;
  const int KT = K / KG;
  const int NS = K / KS;                     // stages per unit
  const int MT = MODE == 0 ? (2 * p.F) / TC_M : p.H / TC_M;
  const int MGT = (MT + 1) / 2;              // M-tile pairs per tile
  const int A = p.T * p.k;
  const int DM = p.dm;
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
      ptx::mbar_init(bar(BAR_AFULL + s), 8);  // four dequant warps in each CTA (even CTA's barrier)
      ptx::mbar_init(bar(BAR_AEMPTY + s), 1);
    }
    for (int s = 0; s < NBMAX; ++s) {
      // this CTA's loads (gather threads, or one expect_tx arrival), plus the odd CTA's forwarded
      // completion on the even CTA's barrier
      const int own = MODE == 0 ? GATHER_T : 1;
      ptx::mbar_init(bar(BAR_BFULL + s), leader ? own + 1 : own);
      ptx::mbar_init(bar(BAR_BEMPTY + s), 1);
    }
    for (int d = 0; d < 2; ++d) {
      ptx::mbar_init(bar(BAR_DFULL + d), 1);
      ptx::mbar_init(bar(BAR_DEMPTY + d), 8);  // four epilogue warps in each CTA (even CTA's barrier)
    }
    ptx::mbar_init(bar(BAR_FIN), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(s_tmem), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised and the pair's TMEM allocated before any role starts
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const unsigned long long lim = p.wait_cycles;
  int prod_b = 0;  // activation TMA stages issued (down), for the drain after a timeout
  // Weight ring: the two dequant warpgroups take alternate stages (warpgroup it & 1), and each
  // owns every other slot -- warpgroup w's c-th stage goes to slot 2 (c % (NW / 2)) + w, fill
  // c / (NW / 2) -- so a slot's fills are always consumed by one warpgroup in order.  (With shared
  // slots a warpgroup could wait for a slot's next fill while the other's fill before it is still
  // landing, and a parity wait cannot tell those two phases apart.)
  int prod_wc[2] = {0, 0};  // weight stages issued per consuming warpgroup (also for the drain)

  if (warp == 0) {
    // ------------------------------------------------ weight producer: this SM's M-tile
    const int HW = NW / 2;
    int it = 0;  // stages of every unit, as the dequant warpgroups count them
    for (int u = cid; u < units; u += ncl) {
      Tile t;
      int grp;
      if (!unit_tile(p, u, MGT, &t, &grp)) continue;
      const int m = 2 * grp + static_cast<int>(rank);
      if (m >= MT) {  // odd M-tile count: the odd CTA has no rows in the last pair
        it += NS;
        continue;
      }
      const uint8_t* g0 = p.w + (static_cast<size_t>(t.expert) * MT + m) * KT * static_cast<size_t>(W_BLOCK);
      for (int ks = 0; ks < NS; ++ks, ++it) {
        const int wg = it & 1, c = prod_wc[wg]++;
        const int s = 2 * (c % HW) + wg, r = c / HW;
        if (r > 0 && !wait_warp(bar(BAR_WEMPTY + s), (r - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) goto wprod_done;
        ptx::mbar_arrive_expect_tx_elect(bar(BAR_WFULL + s), static_cast<uint32_t>(W_STAGE));
        ptx::bulk_g2s_elect(sbase + off_w + s * W_STAGE, g0 + static_cast<size_t>(ks) * GPS * W_BLOCK, W_STAGE,
                            bar(BAR_WFULL + s));
      }
    }
  wprod_done:;
  } else if (warp == 1) {
    if (leader) {
      // ------------------------------------------------ pair MMA issuer (even CTA)
      int ui = 0;
      int sa = 0, pa = 0, sb = 0, pb = 0;
      for (int u = cid; u < units; u += ncl) {
        Tile t;
        int grp;
        if (!unit_tile(p, u, MGT, &t, &grp)) continue;
        const uint32_t idesc = ptx::idesc_bf16_f32(2 * TC_M, round32(t.rows));
        const int d = ui % ND, rd = ui / ND;
        if (rd > 0 && !wait_warp(bar(BAR_DEMPTY + d), (rd - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
        ptx::tc_fence_after();
        const uint32_t dacc = tmem + d * DM;
        for (int ks = 0; ks < NS; ++ks) {
          if (!wait_warp(bar(BAR_AFULL + sa), pa, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
          if (!wait_warp(bar(BAR_BFULL + sb), pb, s_abort, p.err, lim, p.sleep_ns)) goto mma_done;
          if (MODE == 0) ptx::fence_proxy_async_smem();  // this CTA's cp.async rows, read by the tensor core
          ptx::tc_fence_after();
          const uint32_t a0 = tmem + A0 + sa * A_COLS;
          const uint32_t b0 = sbase + sb * SB;
#pragma unroll
          for (int g = 0; g < GPS; ++g)
            ptx::mma_group_pair_elect(dacc, a0 + g * 32, ptx::smem_desc_sw128(b0 + g * atom_bytes), idesc,
                                      g == 0 ? static_cast<uint32_t>(ks != 0) : 1u);
          ptx::mma_commit_pair_elect(bar(BAR_AEMPTY + sa));
          ptx::mma_commit_pair_elect(bar(BAR_BEMPTY + sb));
          if (++sa == NA) {
            sa = 0;
            pa ^= 1;
          }
          if (++sb == NB) {
            sb = 0;
            pb ^= 1;
          }
        }
        ptx::mma_commit_pair_elect(bar(BAR_DFULL + d));
        ++ui;
      }
    mma_done:
      ptx::mma_commit_pair_elect(bar(BAR_FIN));
      if (lane == 0) wait_drain(bar(BAR_FIN), 0, lim);
      __syncwarp();
    } else {
      // ------------------------------------------------ forwarder (odd CTA): this CTA's activation stage
      // has landed -> one arrival on the even CTA's barrier of the same stage
      int sb = 0, pb = 0;
      for (int u = cid; u < units; u += ncl) {
        Tile t;
        int grp;
        if (!unit_tile(p, u, MGT, &t, &grp)) continue;
        for (int ks = 0; ks < NS; ++ks) {
          if (!wait_warp(bar(BAR_BFULL + sb), pb, s_abort, p.err, lim, p.sleep_ns)) goto fwd_done;
          if (MODE == 0) ptx::fence_proxy_async_smem();  // cp.async rows, read by the pair's tensor core
          if (lane == 0) ptx::mbar_arrive_cluster(lead_bar(BAR_BFULL + sb));
          __syncwarp();
          if (++sb == NB) {
            sb = 0;
            pb ^= 1;
          }
        }
      }
    fwd_done:;
    }
  } else if (warp < 4) {
    if (MODE == 1) {
      // ------------------------------------------------ activation producer: TMA tiles of this CTA's h rows
      if (warp == 2) {
        int& it = prod_b;
        for (int u = cid; u < units; u += ncl) {
          Tile t;
          int grp;
          if (!unit_tile(p, u, MGT, &t, &grp)) continue;
          const int r0 = t.row0 + static_cast<int>(rank) * (round32(t.rows) / 2);
          for (int ks = 0; ks < NS; ++ks, ++it) {
            const int s = it % NB, r = it / NB;
            if (r > 0 && !wait_warp(bar(BAR_BEMPTY + s), (r - 1) & 1, s_abort, p.err, lim, p.sleep_ns)) goto bprod_done;
            const uint32_t dst = sbase + s * SB;
            ptx::mbar_arrive_expect_tx_elect(bar(BAR_BFULL + s), static_cast<uint32_t>(SB));
            for (int a = 0; a < GPS; ++a)
              ptx::tma_load_2d_elect(dst + a * atom_bytes, &tmap_act, ks * KS + a * KG, r0, bar(BAR_BFULL + s));
          }
        }
      bprod_done:;
      }
    } else {
      // ------------------------------------------------ activation gather: this CTA's half of the token rows
      const int gt = threadIdx.x - 64;  // 0..63
      const int chunk = gt & 7, row_a = gt >> 3;
      int it = 0;
      bool aborted = false;
      for (int u = cid; u < units && !aborted; u += ncl) {
        Tile t;
        int grp;
        if (!unit_tile(p, u, MGT, &t, &grp)) continue;
        const int hn = round32(t.rows) / 2;                     // rows per CTA in this tile
        const int i0 = static_cast<int>(rank) * hn;             // this CTA's first tile row
        int tok[HALF_MAX / 8];
#pragma unroll
        for (int j = 0; j < HALF_MAX / 8; ++j) {
          const int i = i0 + row_a + 8 * j;
          const int r = t.row0 + i;
          tok[j] = (row_a + 8 * j < hn && i < t.rows && r < A) ? __ldg(p.perm + r) : 0;
        }
        bool bad = false;
#pragma unroll
        for (int j = 0; j < HALF_MAX / 8; ++j) {
          const int i = i0 + row_a + 8 * j;
          const int r = t.row0 + i;
          int tk = -1;
          if (row_a + 8 * j < hn && i < t.rows) {
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
          for (int j = 0; j < HALF_MAX / 8; ++j) {
            const int i = row_a + 8 * j;  // row within this CTA's half
            if (tok[j] >= 0) {
              const uint16_t* src = p.act + static_cast<size_t>(tok[j]) * K + ks * KS + chunk * 8;
              const uint32_t dst = dst0 + (i >> 3) * 1024 + (i & 7) * 128 + ((chunk ^ (i & 7)) << 4);
#pragma unroll
              for (int g = 0; g < GPS; ++g) ptx::cp_async_16(dst + g * atom_bytes, src + g * KG);
            }
          }
          ptx::cp_async_mbar_arrive(bar(BAR_BFULL + s));
        }
      }
      ptx::cp_async_wait_all();
    }
  } else if (warp < 12) {
    // ------------------------------------------------ dequant: warpgroup wg expands the stages it with
    // it % 2 == wg of this SM's M-tile; each thread owns one weight row (= its TMEM lane)
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int L = 32 * q + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16) + A0;
    int it = 0;   // stages of every unit (A ring, warpgroup turn)
    int wc = 0;   // this warpgroup's stages with rows in this CTA (its half of the W ring)
    const int HW = NW / 2;
    for (int u = cid; u < units; u += ncl) {
      Tile t;
      int grp;
      if (!unit_tile(p, u, MGT, &t, &grp)) continue;
      const bool has = 2 * grp + static_cast<int>(rank) < MT;
      for (int ks = 0; ks < NS; ++ks, ++it) {
        if ((it & 1) != wg) continue;
        const int sa = it % NA;
        if (has) {
          const int c = wc++;
          const int sw = 2 * (c % HW) + wg;
          if (!wait_warp(bar(BAR_WFULL + sw), (c / HW) & 1, s_abort, p.err, lim, p.sleep_ns)) goto dequant_done;
          const uint8_t* ws = smem + off_w + sw * W_STAGE;
          uint4 pk[GPS][2];
          uint32_t sbw[GPS];
#pragma unroll
          for (int g = 0; g < GPS; ++g) {
            const uint8_t* blk = ws + g * W_BLOCK;
            pk[g][0] = *reinterpret_cast<const uint4*>(blk + L * 16);
            pk[g][1] = *reinterpret_cast<const uint4*>(blk + 2048 + L * 16);
            sbw[g] = *reinterpret_cast<const uint32_t*>(blk + W_PACKED + L * 4);
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(BAR_WEMPTY + sw));  // this warp's rows are in registers
          uint32_t v0[2][32];
#pragma unroll
          for (int g = 0; g < 2; ++g) expand_group(pk[g][0], pk[g][1], sbw[g], v0[g]);
          if (it >= NA && !wait_warp(bar(BAR_AEMPTY + sa), ((it / NA) - 1) & 1, s_abort, p.err, lim, p.sleep_ns))
            goto dequant_done;
          const uint32_t ta = trow + sa * A_COLS;
#pragma unroll
          for (int g = 0; g < 2; ++g) ptx::tmem_st_32x32b_x32(ta + g * 32, v0[g]);
#pragma unroll
          for (int g = 2; g < GPS; ++g) {
            uint32_t v[32];
            expand_group(pk[g][0], pk[g][1], sbw[g], v);
            ptx::tmem_st_32x32b_x32(ta + g * 32, v);
          }
          ptx::tmem_wait_st();
        } else {
          // no rows here in this pair: the slot's stale contents feed accumulator rows that are
          // never stored; only the hand-over is kept
          if (it >= NA && !wait_warp(bar(BAR_AEMPTY + sa), ((it / NA) - 1) & 1, s_abort, p.err, lim, p.sleep_ns))
            goto dequant_done;
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(lead_bar(BAR_AFULL + sa));
      }
    }
  dequant_done:;
  } else {
    // ------------------------------------------------ epilogue of this SM's 128 accumulator rows
    const int q = warp & 3;
    const int e = threadIdx.x - 12 * 32;  // 0..127
    int sbuf = 0;
    int ui = 0;
    for (int u = cid; u < units; u += ncl) {
      Tile t;
      int grp;
      if (!unit_tile(p, u, MGT, &t, &grp)) {
        if (threadIdx.x == 12 * 32 && leader) set_device_error(p.err, MOE_DEV_BAD_BLOCK);
        continue;
      }
      const int m = 2 * grp + static_cast<int>(rank);
      const int d = ui % ND;
      const bool ok = wait_warp(bar(BAR_DFULL + d), (ui / ND) & 1, s_abort, p.err, lim, p.sleep_ns);
      if (!ptx::named_bar_and(EPI_BAR, 128, ok)) break;
      ptx::tc_fence_after();
      const int N = round32(t.rows);
      const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16) + d * DM;  // this warp's lanes
      if (m < MT) {
        if (MODE == 0) {
          // features 64 m .. 64 m + 63 of h; g in lanes 0-63, u in lanes 64-127
          uint16_t* dst = static_cast<uint16_t*>(p.out) + static_cast<size_t>(t.row0) * p.F + GU_F * m;
          const int f = 32 * (q & 1) + lane;
          for (int c0 = 0; c0 < N; c0 += EPI_ROWS, sbuf ^= 1) {
            float* xu = reinterpret_cast<float*>(s_stage + sbuf * STAGE_BUF_GU);
            uint16_t* hs = reinterpret_cast<uint16_t*>(xu + EPI_ROWS * GU_F);
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tq + c0, v);
            ptx::tmem_wait_ld();
            if (q >= 2) {
#pragma unroll
              for (int j = 0; j < 32; ++j) xu[j * GU_F + f] = __uint_as_float(v[j]);
            }
            ptx::named_bar_sync(EPI_BAR, 128);
            if (q < 2) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                hs[j * GU_F + f] = float_to_bf16_bits(silu_fast(__uint_as_float(v[j])) * xu[j * GU_F + f]);
            }
            ptx::named_bar_sync(EPI_BAR, 128);
#pragma unroll
            for (int i = e; i < EPI_ROWS * 8; i += 128) {
              const int r = i >> 3, cc = i & 7;
              if (c0 + r < t.rows)
                *reinterpret_cast<uint4*>(dst + static_cast<size_t>(c0 + r) * p.F + 8 * cc) =
                    reinterpret_cast<const uint4*>(hs + r * GU_F)[cc];
            }
          }
        } else {
          // channels 128 m + (0..127) of y
          const int cc = e & 15, rr = e >> 4;
          uint16_t* dst = static_cast<uint16_t*>(p.out) + static_cast<size_t>(t.row0) * p.H + TC_M * m + 8 * cc;
          for (int c0 = 0; c0 < N; c0 += EPI_ROWS, sbuf ^= 1) {
            uint16_t* st = reinterpret_cast<uint16_t*>(s_stage + sbuf * STAGE_BUF_DOWN);
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tq + c0, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j * TC_M + 32 * q + lane] = float_to_bf16_bits(__uint_as_float(v[j]));
            ptx::named_bar_sync(EPI_BAR, 128);
            const uint4* src = reinterpret_cast<const uint4*>(st) + cc;
#pragma unroll
            for (int r = rr; r < EPI_ROWS; r += 8)
              if (c0 + r < t.rows) *reinterpret_cast<uint4*>(dst + static_cast<size_t>(c0 + r) * p.H) = src[r * 16];
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(lead_bar(BAR_DEMPTY + d));
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
    for (int w = 0; w < 2; ++w)
      for (int c = prod_wc[w] - NW / 2 < 0 ? 0 : prod_wc[w] - NW / 2; c < prod_wc[w]; ++c)
        wait_drain(bar(BAR_WFULL + 2 * (c % (NW / 2)) + w), (c / (NW / 2)) & 1, lim);
  }
  // neither CTA leaves (or releases the pair's TMEM) while the other may still use its shared or
  // tensor memory
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
}

// --------------------------------------------------------------------------
// host side
// --------------------------------------------------------------------------
namespace {

int max_dyn_smem_pair() {
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

cudaError_t launch_gemm_pair(int mode, const uint16_t* act, int T, int H, int F, int E, int k, const void* w,
                             const int32_t* perm, const int32_t* block_map, const int32_t* num_blocks, int bn, int cap,
                             void* out, cudaStream_t s) {
  PairParams prm;
  prm.act = act;
  prm.w = static_cast<const uint8_t*>(w);
  prm.perm = perm;
  prm.block_map = block_map;
  prm.num_blocks = num_blocks;
  prm.out = out;
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
  const int boxr = (bn + 31) & ~31;
  if (boxr > 2 * HALF_MAX) return cudaErrorInvalidValue;
  prm.half = boxr / 2;
  const int Kdim = mode == MOE_GATE_UP_SWIGLU ? H : F;
  // four quant groups per stage (16 MMAs per hand-over) while two accumulator buffers still fit
  const int GPS = (boxr <= 128 && Kdim % (4 * KG) == 0) ? 4 : 2;
  prm.sb = GPS * prm.half * 128;
  const int w_stage = GPS * W_BLOCK;
  const int a_cols = GPS * 32;
  const int fixed = BAR_BYTES + MISC_BYTES + (mode == MOE_GATE_UP_SWIGLU ? stage_bytes<0>() : stage_bytes<1>());
  const int total = max_dyn_smem_pair() - 1024 - fixed;
  int nbs = 0, nws = 0;
  for (int want = 3; want >= 2 && nws < 4; --want) {
    nbs = want;
    nws = (total - nbs * prm.sb) / w_stage;
  }
  if (nws < 4 || nbs < 2) return cudaErrorInvalidValue;
  if (nws > NWMAX) nws = NWMAX;
  nws &= ~1;  // an even depth: half of the slots for each dequant warpgroup
  nbs = (total - nws * w_stage) / prm.sb;
  if (nbs > NBMAX) nbs = NBMAX;
  prm.nb = nbs;
  prm.nw = nws;
  prm.dm = boxr;
  prm.nd = 2 * boxr + 2 * a_cols <= TMEM_COLS ? 2 : 1;
  prm.a0 = prm.nd * boxr;
  prm.na = (TMEM_COLS - prm.a0) / a_cols;
  if (prm.na > NAMAX) prm.na = NAMAX;
  if (prm.na < 2) return cudaErrorInvalidValue;
  const int smem = nbs * prm.sb + nws * w_stage + fixed + 1024;

  CUtensorMap tmap;
  memset(&tmap, 0, sizeof(tmap));
  if (mode == MOE_DOWN) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const int A = T * k;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(F), static_cast<cuuint64_t>(A + T)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(F) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(prm.half)};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(act), gdim, gstride, box,
                     estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  void (*kern)(const PairParams, const CUtensorMap) =
      mode == MOE_GATE_UP_SWIGLU ? (GPS == 4 ? gemm_pair_kernel<0, 4> : gemm_pair_kernel<0, 2>)
                                 : (GPS == 4 ? gemm_pair_kernel<1, 4> : gemm_pair_kernel<1, 2>);
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<size_t>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // one pair per two SMs, as many as can be resident at once (the kernel is persistent over units)
  int ncl = 0;
  cfg.gridDim = dim3(2);
  e = cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (ncl < 1) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(2 * ncl);
  e = cudaLaunchKernelEx(&cfg, kern, prm, tmap);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
