/*
 * moe_w4.h -- C ABI of libmoe_w4.so: the prefill/decode forward of a
 * mixture-of-experts FFN layer with groupwise-affine 4-bit expert weights and
 * GPU-resident routing, for NVIDIA GB300 (sm_103a).
 *
 * The layer follows "Perplexity Open Sources Lily" (aitrending.vip),
 * Technical Details: Model bullet (a router choosing 8 of 256 experts plus one
 * shared expert) and Prefill optimizations bullet (4-bit groupwise affine
 * weights, 64 weights per group, dequantised inside the grouped GEMM with FP32
 * accumulation; routing histogram, prefix scan, scatter and block map kept on
 * the GPU with no CPU synchronisation).  The Chinese section of the same page
 * ("预填充优化") adds that each group of 64 weights shares a bfloat16 scale.
 *
 * Conventions for every call:
 *  - Pointers named *_host are host pointers; every other pointer is a device
 *    pointer owned by the caller.  The library allocates nothing.
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - All tensors are dense row-major.  Device pointers must be 16-byte aligned.
 *  - Calls enqueue work on `stream` and return at once; no call synchronises
 *    the host except moe_get_device_error.
 *  - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  Argument errors
 *    are detected on the host before anything is enqueued.  Faults found by a
 *    kernel (a corrupt block map, an out-of-range index) are recorded in a
 *    device error word instead of trapping; read it with moe_get_device_error.
 *  - Behaviour for NaN or infinite logits is undefined.
 *
 * Sizes: T tokens, H hidden, E routed experts (the shared expert is index E of
 * every weight array), k experts per token, F expert FFN width, A = T*k
 * assignments, block_n rows per GEMM tile.  Limits: 1 <= k <= 32, k <= E,
 * E <= 1024, 1 <= T <= 2^20; the grouped GEMMs and the layer also need
 * H % 128 == 0 and F % 128 == 0.
 */
#ifndef MOE_W4_H
#define MOE_W4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
  MOE_OK = 0,
  MOE_ERR_NULL = -1,      /* a required pointer is NULL */
  MOE_ERR_ALIGN = -2,     /* a device pointer is not 16-byte aligned */
  MOE_ERR_SHAPE = -3,     /* sizes outside the limits above */
  MOE_ERR_WORKSPACE = -4, /* workspace smaller than moe_route_workspace_size() */
  MOE_ERR_CUDA = -5,      /* a CUDA launch or copy failed */
  MOE_ERR_DEVICE = -6,    /* moe_get_device_error found a kernel-side fault */
  MOE_ERR_MODE = -7       /* unknown mode or variant */
};

/* Device error word values (written by kernels, read by moe_get_device_error). */
enum {
  MOE_DEV_OK = 0,
  MOE_DEV_BAD_BLOCK = 1,  /* a block-map entry outside [0, E] x [0, A+T) */
  MOE_DEV_BAD_INDEX = 2,  /* a permutation entry outside [0, A) */
  MOE_DEV_TIMEOUT = 3,    /* a bounded device wait ran out */
  MOE_DEV_BAD_WORKSPACE = 4 /* a routing or decode workspace was not zero-filled when the call
                               began (a barrier counter already counted, or per-expert totals
                               that cannot come from this call); nothing was written from them */
};

/* GEMM modes. */
enum {
  MOE_GATE_UP_SWIGLU = 0, /* h = bf16(silu(x Wg^T) * (x Wu^T)) per routed row */
  MOE_DOWN = 1            /* y = bf16(h Wd^T) per routed row */
};

/* GEMM kernels.  The layer has two regimes and one kernel for each: the
 * tensor-core grouped GEMM for prefill-sized tiles and the GEMV for decode
 * tiles of at most 8 token rows.  Both read the same repacked weights and
 * compute the same values; AUTO picks by block_n, the others force one (the
 * tests run each kernel over every shape it accepts). */
enum {
  MOE_IMPL_AUTO = 0,      /* GEMV when block_n <= 8, else the tensor-core kernel */
  MOE_IMPL_TC = 2,        /* tcgen05 kernel, one CTA per work unit */
  MOE_IMPL_GEMV = 3,      /* decode GEMV kernel, mma.sync */
  MOE_IMPL_TC2 = 4,       /* tcgen05 kernel on CTA pairs (.cta_group::2): gate/up weights repacked
                             with gate_up = 2 (interleaved tiles); tiles of up to 256 rows */
  MOE_IMPL_TC_BF16 = 5    /* the unfused comparison path: the tcgen05 kernel over weights already
                             expanded to bf16 by moe_expand_w4 (3.6 times the bytes of the 4-bit
                             weights); same results as MOE_IMPL_TC */
};

/* ------------------------------------------------------------------------ */
/* Routing                                                                  */
/* ------------------------------------------------------------------------ */

/* Rows of the block map that moe_route may write: ceil(A/block_n) + E + ceil(T/block_n). */
int moe_block_map_capacity(int T, int E, int k, int block_n);

/* Bytes of scratch moe_route needs (per-chunk expert counts and the
 * counters of its grid barrier; 0 when one CTA routes everything). */
size_t moe_route_workspace_size(int T, int E, int k, int block_n);

/*
 * moe_route -- router softmax + top-k and GPU-resident routing
 * ("Perplexity Open Sources Lily", Technical Details, Model and Prefill
 * optimizations bullets).
 *
 * logits     float32 [T, E]   router logits (read only)
 * topk_ids   int32  [T, k]    chosen experts, by descending logit; equal
 *                             logits go to the lower index (-0.0 == +0.0)
 * topk_w     float32 [T, k]   exp(l_j - l_max) / sum over the k chosen
 *                             (the softmax renormalised over the top k)
 * counts     int32  [E]       histogram of the T*k assignments over experts
 * offsets    int32  [E+1]     exclusive prefix scan of counts; offsets[E] = A
 * perm       int32  [A]       assignment a = t*k + j at sorted position p,
 *                             sorted by (expert, a): perm[p] = a
 * inv_perm   int32  [A]       inv_perm[perm[p]] = p
 * block_map  int32  [cap, 3]  tiles (expert, first row, rows) for every expert
 *                             in ascending order, block_n rows per tile, then
 *                             the shared expert (index E) over rows A..A+T-1
 *                             (row A+t is token t); only the first
 *                             *num_blocks rows are written
 * num_blocks int32  [1]       number of tiles (device memory)
 * workspace  device scratch of at least moe_route_workspace_size() bytes,
 *            zero-filled by the caller before its first use: the per-chunk
 *            counts go at its start, and its last 16 bytes (of workspace_bytes)
 *            hold counters that every call leaves at zero, so one workspace
 *            serves calls with any T it is large enough for.  A workspace
 *            whose counters are not zero when a call begins is reported as
 *            MOE_DEV_BAD_WORKSPACE; no output is written from counts that do
 *            not add up.
 * block_n    1..1024.
 */
int moe_route(const float* logits, int T, int E, int k, int block_n,
              int32_t* topk_ids, float* topk_w, int32_t* counts, int32_t* offsets,
              int32_t* perm, int32_t* inv_perm, int32_t* block_map, int32_t* num_blocks,
              void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_route_x -- the router projection fused with the top-k, then the routing
 * of moe_route ("Perplexity Open Sources Lily", Technical Details, Model
 * bullet: a router chooses 8 of 256 experts per token).
 *
 * x        bf16 [T, H]   the tokens' activations
 * w_router bf16 [E, H]   the router's projection, one row per expert
 * logits   float32 [T, E] output: x w_router^T, products of the bf16 operands
 *                         accumulated in FP32 on the tensor cores
 * topk_ids ... workspace: as moe_route; the top-k (same selection, ties and
 *          weights as moe_route) is taken from these logits in the same
 *          kernel that computes them, then the histogram, scan, scatter and
 *          block map follow in moe_route's kernel.
 * Needs H % 64 == 0, E % 64 == 0 and E <= 512 (one cluster of E / 64 CTAs
 * per 128 tokens).  Two kernel launches on `stream`.
 */
int moe_route_x(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, int block_n,
                float* logits, int32_t* topk_ids, float* topk_w, int32_t* counts, int32_t* offsets,
                int32_t* perm, int32_t* inv_perm, int32_t* block_map, int32_t* num_blocks,
                void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_router -- the first kernel of moe_route_x alone: logits = x w_router^T
 * and the top-k ids and weights, one launch.  For callers that route
 * elsewhere, such as moe_layer_forward's fused decode kernel (which takes the
 * logits and recomputes the same top-k with the rest of the routing): a
 * batch-1 decode step through several layers is then two launches per layer,
 * each layer's output the next layer's x.  Same limits as moe_route_x.
 */
int moe_router(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, float* logits,
               int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/*
 * moe_route_noalloc -- moe_route for callers that may not allocate device
 * memory: code handed only its input and output buffers by a host engine
 * whose allocator owns the whole device (a serving process that reserves
 * memory up front), or code on a latency path where cudaMalloc's implicit
 * device-wide synchronisation is not acceptable.  The pages describe no such
 * entry point; it has no counterpart there.
 *
 * Same arguments, outputs and limits as moe_route, without the workspace:
 * the per-chunk expert counts live in one fixed 256 KiB device array of the
 * library (256 chunks x 256 experts of int32), held on every GPU that loads
 * the library until the process exits.  That covers every T for E <= 256;
 * a call whose counts need more than 256 KiB (moe_route_workspace_size
 * reports the need) returns MOE_ERR_WORKSPACE before enqueueing anything.
 * For T*k <= 1024 no scratch is used.  Nothing is allocated or freed.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Each call that uses the array first clears the
 * counters of its grid barrier (16 bytes, cudaMemsetAsync on `stream`), and
 * the routing kernel overwrites every count before reading it.  All calls
 * share the one array: calls that can overlap on the GPU (different streams,
 * or different host threads) race and must be serialised by the caller; a
 * call after such a race, on its own, gives correct results again.
 */
int moe_route_noalloc(const float* logits, int T, int E, int k, int block_n,
                      int32_t* topk_ids, float* topk_w, int32_t* counts, int32_t* offsets,
                      int32_t* perm, int32_t* inv_perm, int32_t* block_map, int32_t* num_blocks,
                      moe_stream_t stream);

/*
 * moe_rms_norm -- out[t] = bf16(x[t] / sqrt(mean_c x[t, c]^2 + eps)), unit
 * gain, FP32 sum of squares, each output rounded once: the glue that
 * normalises a layer's input when several layers run in sequence (the
 * decode chain).  x, out bf16 [T, H], H % 8 == 0; out may not overlap x.
 */
int moe_rms_norm(const uint16_t* x, uint16_t* out, int T, int H, float eps, moe_stream_t stream);

/*
 * moe_norm_router -- a decode step's layer input and router logits in one
 * launch (at most 8 tokens): x_norm = moe_rms_norm(x) (the same bits) and
 * logits = x_norm w_router^T (bf16 products, FP32 sums), one warp per expert.
 * x, x_norm bf16 [T, H]; w_router bf16 [E, H]; logits float32 [T, E].  The
 * decode chain feeds these to moe_layer_forward, whose fused decode kernel
 * takes the top-k from the logits.  Returns MOE_ERR_SHAPE for T > 8.
 */
int moe_norm_router(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, float eps, uint16_t* x_norm,
                    float* logits, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Weights                                                                  */
/* ------------------------------------------------------------------------ */

/*
 * Canonical weight layout (what moe_repack_w4 reads):
 *   packed uint32 [n_mat, rows, K/8]: K element 8*w+i in bits [4i, 4i+4) of word w
 *   scale, bias   bf16   [n_mat, rows, K/64]: w = bf16(q * scale + bias)
 * Gate/up matrices have rows = 2F (F gate rows, then F up rows) and K = H;
 * down matrices have rows = H and K = F.  n_mat = E + 1, shared expert last.
 */

/* Bytes of the repacked layout for n_mat matrices of rows x K. */
size_t moe_repacked_bytes(int n_mat, int rows, int K);

/*
 * moe_repack_w4 -- one-time conversion of canonical weights into the layout
 * the tensor-core kernel streams (not part of the layer's timed work).  Per
 * matrix, per 128-row tile, per 64-wide K group, one contiguous 4608-byte
 * block: [2 halves][128 rows][16 bytes] of packed nibbles (half h holds K
 * elements 32h..32h+31 of the group; within each word the nibbles are ordered
 * so that (word >> 4j) & 0x000f000f holds elements 2j and 2j+1 of its eight)
 * followed by [128 rows] x (scale bf16, bias bf16).  With gate_up = 1 the
 * tiles come in pairs: tile 2j holds the gate rows and tile 2j+1 the up rows
 * of features 128j .. 128j+127 (rows = 2F, F % 128 == 0).  With gate_up = 2
 * (the layout MOE_IMPL_TC2 reads) tile j holds the gate rows of features
 * 64j .. 64j+63 in its rows 0-63 and their up rows in rows 64-127 (F % 64 ==
 * 0).  gate_up = 0 is any other matrix (the down projection).  Needs rows %
 * 128 == 0 and K % 64 == 0; returns MOE_ERR_SHAPE otherwise.
 */
int moe_repack_w4(const uint32_t* packed, const uint16_t* scale, const uint16_t* bias,
                  int n_mat, int rows, int K, int gate_up, void* out, moe_stream_t stream);

/*
 * moe_expand_w4 -- the unfused path's first step: expand repacked 4-bit
 * weights (moe_repack_w4's output for n_mat matrices of rows x K) into a bf16
 * copy in HBM, in the same tile order (per matrix, 128-row tile, 64-wide K
 * group: 128 rows x 64 bf16, the 16-byte chunk i of row L stored at position
 * i ^ (L & 7)), each weight bf16(q * scale + bias) as the fused kernels
 * compute it.  moe_expert_gemm_w4 with MOE_IMPL_TC_BF16 reads this copy.
 * The pages credit fusing the dequantisation into the grouped GEMM, with no
 * full bf16 copy ever written, with +77.4% prefill throughput ("Perplexity
 * Open Sources Lily", TL;DR; the itinai.com post on the same engine,
 * paragraph 2); this pair of calls is the path that claim is measured against.
 * out: moe_expanded_bytes(n_mat, rows, K) bytes.
 */
size_t moe_expanded_bytes(int n_mat, int rows, int K);
int moe_expand_w4(const void* w_repacked, int n_mat, int rows, int K, void* out, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Grouped expert GEMM                                                      */
/* ------------------------------------------------------------------------ */

/*
 * moe_expert_gemm_w4 -- grouped SwiGLU expert GEMM over 4-bit groupwise-affine
 * weights with the dequantisation fused into the GEMM and FP32 accumulation
 * ("Perplexity Open Sources Lily", Technical Details, Prefill optimizations
 * bullet; itinai.com post on the Lily engine, paragraph 2: weights are expanded
 * only on chip, never as a full bf16 copy in memory).
 *
 * mode MOE_GATE_UP_SWIGLU:
 *   act  bf16 [T, H] tokens; row r of tile (e, r0, n) reads token perm[r]/k
 *        for r < A and token r-A for r >= A (shared expert);
 *   out  bf16 [A+T, F]: h[r] = bf16(silu(g) * u), g/u the gate/up projections
 *        accumulated in FP32 over the bf16-expanded weights.
 * mode MOE_DOWN:
 *   act  bf16 [A+T, F] the h of the gate/up call;
 *   out  bf16 [A+T, H]: y[r] = bf16(h[r] Wd^T) accumulated in FP32, in the
 *        same permuted row order (perm and topk_w are not read).
 * w_packed: the matrix set in the repacked layout of moe_repack_w4 (packed
 *        nibbles with each 64-group's bf16 scale and bias in the same block).
 * block_map / num_blocks: moe_route's outputs for the same block_n.
 * impl: MOE_IMPL_*.  AUTO takes GEMV for block_n <= 8 and TC otherwise.  TC
 * and TC_BF16 need block_n <= 128, TC2 block_n <= 256 (and gate/up weights
 * repacked with gate_up = 2); GEMV (decode: tiles of at most 8 token rows)
 * needs block_n <= 8; all need H % 128 == 0 and F % 128 == 0.  TC_BF16 reads
 * the bf16 copy of moe_expand_w4 instead of the 4-bit weights.  Returns
 * MOE_ERR_SHAPE when the chosen kernel cannot take the shape and
 * MOE_ERR_MODE for an unknown mode or impl.
 */
int moe_expert_gemm_w4(int mode, int impl, const uint16_t* act, int T, int H, int F, int E, int k,
                       const void* w_packed, const int32_t* perm, const float* topk_w,
                       const int32_t* block_map, const int32_t* num_blocks, int block_n,
                       void* out, moe_stream_t stream);

/*
 * moe_combine -- weighted gather-combine back to token order ("Perplexity
 * Open Sources Lily", Technical Details, Model bullet: 8 routed experts plus
 * one shared expert per token):
 *   out[t, c] = bf16( sum_{j<k} topk_w[t, j] * y[inv_perm[t*k + j], c]
 *                     + y[A + t, c] )
 * with the sum in FP32 in that fixed order (j = 0 .. k-1, then the shared
 * row), rounded once to nearest even.  y bf16 [A+T, H] is the down GEMM's
 * output, inv_perm int32 [A] and topk_w float32 [T, k] come from moe_route;
 * out bf16 [T, H].  H % 8 == 0.  An inv_perm entry outside [0, A) sets
 * MOE_DEV_BAD_INDEX and that term is skipped.
 */
int moe_combine(const uint16_t* y, const int32_t* inv_perm, const float* topk_w, uint16_t* out, int T, int H,
                int k, moe_stream_t stream);

/*
 * moe_expert_ffn_w4 -- both projections of every expert tile in one launch,
 * h kept on chip: for each block-map tile, the gate/up GEMM with SwiGLU writes
 * the tile's h into shared memory and the down GEMM of the same tile reads it
 * from there ("Perplexity Open Sources Lily", Technical Details, Prefill
 * optimizations bullet: the weights are expanded inside the GEMM; here h, too,
 * never leaves the chip).  x bf16 [T, H]; w13, w2 repacked as for
 * moe_expert_gemm_w4 (gate_up = 1 for w13); perm, block_map, num_blocks from
 * moe_route; y bf16 [A+T, H] (written; combine it with moe_combine).  The
 * same bits of y as MOE_GATE_UP_SWIGLU followed by MOE_DOWN; no h is written.
 * Needs block_n <= 64 (the tile's h must fit in shared memory),
 * H % 128 == 0 and F % 256 == 0, else MOE_ERR_SHAPE; argument errors are
 * returned before anything is enqueued.  moe_layer_forward uses it for the
 * tensor-core path whenever these hold (faster than the two GEMMs there).
 */
int moe_expert_ffn_w4(const uint16_t* x, int T, int H, int F, int E, int k, const void* w13, const void* w2,
                      const int32_t* perm, const int32_t* block_map, const int32_t* num_blocks, int block_n,
                      uint16_t* y, moe_stream_t stream);

/*
 * moe_down_combine -- MOE_DOWN and moe_combine in one launch of the
 * tensor-core kernel: the down projection writes its bf16 rows y as
 * moe_expert_gemm_w4 does, and every (token, 128-channel block) counts its
 * written rows in `workspace`; the epilogue that writes the last of a token's
 * k + 1 rows of a block combines them there, with moe_combine's arithmetic and
 * order (so out is bit for bit moe_combine's).  No thread waits for another.
 * ("Perplexity Open Sources Lily", Technical Details, Model bullet: 8 routed
 * experts plus one shared expert per token.)
 * h, perm, inv_perm, topk_w, block_map, num_blocks: as for MOE_DOWN and
 * moe_combine; y bf16 [A+T, H] (written); out bf16 [T, H].
 * workspace: moe_down_combine_workspace_size(T, H) bytes (an int32 per token
 * and 128 channels), zero-filled by the caller before the first call; every
 * call that completes leaves it zero (a counter found above k is reported as
 * MOE_DEV_BAD_WORKSPACE; after a call that reported a device error, zero it
 * again).  Needs block_n <= 128, H % 128 == 0, F % 128 == 0; argument errors
 * (MOE_ERR_SHAPE, _NULL, _ALIGN, _WORKSPACE) are returned before anything is
 * enqueued.  Measured slower than MOE_DOWN + moe_combine on this GPU (the
 * epilogue's counting and gathers lengthen every unit), so the layer uses it
 * only when buffers->combine_ws is set.
 */
size_t moe_down_combine_workspace_size(int T, int H);
int moe_down_combine(const uint16_t* h, int T, int H, int F, int E, int k, const void* w_packed,
                     const int32_t* perm, const int32_t* inv_perm, const float* topk_w,
                     const int32_t* block_map, const int32_t* num_blocks, int block_n,
                     uint16_t* y, uint16_t* out, void* workspace, size_t workspace_bytes,
                     moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Whole layer                                                              */
/* ------------------------------------------------------------------------ */

/* Device buffers of one layer call (all caller-owned; sizes for T, E, k, block_n). */
typedef struct {
  int32_t* topk_ids;   /* [T,k] */
  float* topk_w;       /* [T,k] */
  int32_t* counts;     /* [E] */
  int32_t* offsets;    /* [E+1] */
  int32_t* perm;       /* [A] */
  int32_t* inv_perm;   /* [A] */
  int32_t* block_map;  /* [moe_block_map_capacity, 3] */
  int32_t* num_blocks; /* [1] */
  uint16_t* h;         /* bf16 [A+T, F] */
  uint16_t* y;         /* bf16 [A+T, H] */
  void* workspace;     /* moe_route_workspace_size bytes */
  size_t workspace_bytes;
  void* decode_ws;      /* fused decode path: moe_decode_workspace_size bytes, zero before the
                           first call (every call leaves it zero); NULL: never fuse */
  size_t decode_ws_bytes;
  void* combine_ws;     /* moe_down_combine_workspace_size bytes, zero before the first call;
                           with the tensor-core kernel the layer then runs moe_down_combine
                           instead of MOE_DOWN + moe_combine; NULL: the two calls */
  size_t combine_ws_bytes;
} moe_buffers_t;

/*
 * moe_decode_workspace_size -- bytes of the fused decode path's counters for
 * T tokens and hidden size H (0 when T is above the fused path's limit of 8
 * tokens).  The workspace must be zero-filled once by the caller; each call
 * of the fused path returns it to zero.
 */
size_t moe_decode_workspace_size(int T, int H);

/* Weights of one layer: gate/up and down matrices of E+1 experts in the
 * repacked layout of moe_repack_w4 (gate_up = 1 for w13, 0 for w2). */
typedef struct {
  const void* w13;
  const void* w2;
} moe_weights_t;

/*
 * moe_layer_forward -- the whole hot path on one stream with no host sync:
 * moe_route, gate/up GEMM, down GEMM, moe_combine.  x bf16 [T,H], logits
 * float32 [T,E], out bf16 [T,H] are device pointers.  With the tensor-core
 * kernel, tiles of at most 64 rows and F % 256 == 0 the two GEMMs run as
 * moe_expert_ffn_w4 (h kept on chip, the same y); buffers->h is then not
 * written.
 *
 * Decode: when the GEMV kernel is chosen (impl MOE_IMPL_GEMV, or AUTO with
 * block_n <= 8), T <= 8, k <= 32 and buffers->decode_ws is set, the four steps
 * run as one fused kernel (cooperative launch; every CTA recomputes the
 * routing, then the gate/up and down work items hand over through counters
 * in decode_ws).  Its results are those of the four calls: the same routing
 * outputs, h, y and out.  Returns MOE_ERR_WORKSPACE when decode_ws_bytes is
 * below moe_decode_workspace_size(T, H).
 */
int moe_layer_forward(const uint16_t* x, const float* logits, uint16_t* out,
                      int T, int H, int F, int E, int k, int block_n, int impl,
                      const moe_weights_t* weights, const moe_buffers_t* buffers,
                      moe_stream_t stream);

/*
 * moe_layer_forward_host -- the same with x_host, logits_host and out_host in
 * host memory, all on `stream`: x is copied to the device staging buffer x_dev
 * first (the grouped GEMM reads each row k + 1 times).  When logits_host and
 * out_host are pinned (or registered) host memory, the kernels read the
 * logits and write the output there directly over the host link (each byte
 * crosses it once either way); otherwise they are copied through logits_dev
 * and out_dev.  Returns after enqueueing; the caller synchronises the stream
 * before reading out_host.
 */
int moe_layer_forward_host(const uint16_t* x_host, const float* logits_host, uint16_t* out_host,
                           uint16_t* x_dev, float* logits_dev, uint16_t* out_dev,
                           int T, int H, int F, int E, int k, int block_n, int impl,
                           const moe_weights_t* weights, const moe_buffers_t* buffers,
                           moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                              */
/* ------------------------------------------------------------------------ */

/* Synchronises the current device, returns the device error word in *code and
 * clears it.  Returns MOE_ERR_CUDA if the synchronisation itself failed. */
int moe_get_device_error(int32_t* code);

/* Time limit of every bounded wait inside the kernels (default 1 s): the
 * pipeline waits of the tensor-core kernel and the grid barriers of the
 * routing and fused decode kernels.  When a wait runs out the kernel records
 * MOE_DEV_TIMEOUT; the tensor-core kernel then leaves its loops, waits (at
 * least about 10 ms, whatever the limit) for its copies and MMAs in flight,
 * frees its tensor memory and returns; a grid barrier goes on.  Later kernels
 * validate every block-map and permutation entry they read, so a routing
 * result left incomplete by a timeout is reported, not followed.  Test hook. */
void moe_set_wait_limit_ns(uint64_t ns);

/* Wait statistics of the tensor-core kernels (moe_gemm_tc.cu, moe_ffn_tc.cu,
 * moe_gemm_pair.cu) in a trace build: libmoe_w4_trace.so, built by
 * `python -m bit_mixture_experts_gb300.build --trace` (-DMOE_TRACE), which
 * `python -m bit_mixture_experts_gb300.trace` loads and reports.  The product
 * library libmoe_w4.so records nothing.
 *
 * For each CTA (blockIdx.x mod 1024) and warp (32 slots), four uint64 words:
 * SM cycles spent in the kernel's bounded mbarrier waits, the number of such
 * waits, 2^64 - 1 - clock64 at the start of the warp's first wait (zero: no
 * wait), and clock64 at the end of its last -- word 4 (32 cta + warp) + i.
 * The words accumulate over launches until the next reset.
 *
 * moe_trace_words: the number of words (1024 x 32 x 4), or 0 in the product
 * library.
 * moe_trace_reset: zeroes them, ordered on `stream`.
 * moe_trace_read: synchronous copy of the first `words` words to `host`.
 * Both return MOE_ERR_MODE in the product library, MOE_ERR_NULL for a null
 * `host`, MOE_ERR_CUDA on a failed CUDA call. */
size_t moe_trace_words(void);
int moe_trace_reset(moe_stream_t stream);
int moe_trace_read(uint64_t* host, size_t words);

/* Library version, e.g. 0x000100 for 0.1.0. */
int moe_version(void);

/* Number of kernels this process has launched through the library so far
 * (all devices).  Used to count launches inside a timed region. */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_W4_H */
