// extern "C" entry points of libmoe_w4.so: argument checks, the device error
// word, and the launch sequence of the layer.  Every compute step runs in the
// kernels of moe_route.cu, moe_gemm_tc.cu, moe_gemm_gemv.cu, moe_decode.cu and
// moe_combine.cu; nothing here touches tensor data on the host.
#include <atomic>
#include <mutex>

#include "moe_common.cuh"
#ifdef MOE_TRACE
#include "moe_tc_dev.cuh"  // the trace words' layout (TRACE_ERR_INTS, TRACE_CTAS, trace_wait)
#endif

namespace moe {

#ifdef MOE_TRACE
// The trace build keeps the wait statistics of the tensor-core kernels right after the error word
// (TRACE_ERR_INTS ints, then TRACE_CTAS x 32 warps x 4 words; see trace_wait).
using tc_dev::TRACE_ERR_INTS;
constexpr size_t TRACE_WORDS = static_cast<size_t>(tc_dev::TRACE_CTAS) * 32 * 4;
struct TraceBlock {
  int err[TRACE_ERR_INTS];
  unsigned long long words[TRACE_WORDS];
};
__device__ TraceBlock g_trace_block;
#define MOE_ERROR_SYMBOL g_trace_block  // the error word is its first int
#else
__device__ int g_device_error = 0;
#define MOE_ERROR_SYMBOL g_device_error
#endif

// Per-device address of the device error word, looked up once per device.
int* device_error_ptr() {
  static std::mutex mu;
  static int* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, MOE_ERROR_SYMBOL) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

static std::atomic<uint64_t> g_launches{0};

void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

// defined in the kernel files
size_t route_workspace_bytes(int T, int E, int k);
cudaError_t launch_route(const float* logits, int T, int E, int k, int bn, int32_t* ids, float* w, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* bm, int32_t* nb, void* ws,
                         size_t ws_bytes, cudaStream_t s, int ids_given);
cudaError_t launch_rms_norm(const uint16_t* x, uint16_t* out, int T, int H, float eps, int num_sms, cudaStream_t s);
int norm_router_max_tokens();
cudaError_t launch_norm_router(const uint16_t* x, const uint16_t* wr, uint16_t* xn, float* logits, int T, int H,
                               int E, float eps, cudaStream_t s);
cudaError_t launch_router(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, float* logits,
                          int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_combine(const uint16_t* y, const int32_t* inv_perm, const float* topk_w, uint16_t* out, int T,
                           int H, int k, int num_sms, cudaStream_t s);
size_t repacked_bytes(int n_mat, int rows, int K);
cudaError_t launch_repack(const uint32_t* packed, const uint16_t* scale, const uint16_t* bias, int n_mat, int rows,
                          int K, int gate_up, void* out, cudaStream_t s);
cudaError_t launch_gemm_gemv(int mode, const uint16_t* act, int T, int H, int F, int E, int k, const void* w,
                             const int32_t* perm, const float* topk_w, const int32_t* block_map,
                             const int32_t* num_blocks, int bn, int cap, void* out, int num_sms, cudaStream_t s);
int gemv_max_rows();
int decode_max_tokens();
size_t decode_workspace_bytes(int T, int H);
cudaError_t launch_ffn_tc(const uint16_t* x, int T, int H, int F, int E, int k, const void* w13, const void* w2,
                          const int32_t* perm, const int32_t* block_map, const int32_t* num_blocks, int bn, int cap,
                          uint16_t* y, int num_sms, cudaStream_t s);
cudaError_t launch_decode(const uint16_t* x, const float* logits, const void* w13, const void* w2, int T, int H, int F,
                          int E, int k, int bn, int32_t* topk_ids, float* topk_w, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* inv_perm, int32_t* block_map, int32_t* num_blocks, uint16_t* h,
                          uint16_t* y, uint16_t* out, void* ws, unsigned long long wait_ns, int num_sms,
                          cudaStream_t s);
unsigned long long wait_limit_ns();
cudaError_t launch_gemm_tc(int mode, const uint16_t* act, int T, int H, int F, int E, int k, const void* w,
                           const int32_t* perm, const float* topk_w, const int32_t* block_map,
                           const int32_t* num_blocks, int bn, int cap, void* out, int num_sms, cudaStream_t s,
                           bool raw, uint16_t* cmb_out, const int32_t* inv_perm, int* cmb_cnt);
size_t expanded_bytes(int n_mat, int rows, int K);
cudaError_t launch_expand(const void* w4, int n_mat, int rows, int K, void* out, cudaStream_t s);
cudaError_t launch_gemm_pair(int mode, const uint16_t* act, int T, int H, int F, int E, int k, const void* w,
                             const int32_t* perm, const int32_t* block_map, const int32_t* num_blocks, int bn, int cap,
                             void* out, cudaStream_t s);
void set_wait_limit_ns(unsigned long long ns);

namespace {

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return 0x000100; }

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_block_map_capacity(int T, int E, int k, int block_n) {
  if (T < 1 || E < 1 || k < 1 || block_n < 1) return 0;
  const long long A = static_cast<long long>(T) * k;
  return static_cast<int>((A + block_n - 1) / block_n + E + (T + block_n - 1) / block_n);
}

size_t moe_route_workspace_size(int T, int E, int k, int block_n) {
  (void)block_n;
  if (T < 1 || E < 1 || k < 1) return 0;
  return route_workspace_bytes(T, E, k);
}

int moe_route(const float* logits, int T, int E, int k, int block_n, int32_t* topk_ids, float* topk_w,
              int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* block_map,
              int32_t* num_blocks, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  int rc = check_route_shape(T, E, k, block_n);
  if (rc) return rc;
  rc = check_ptrs(logits, topk_ids, topk_w, counts, offsets, perm, inv_perm, block_map, num_blocks);
  if (rc) return rc;
  const size_t need = route_workspace_bytes(T, E, k);
  if (need > 0) {
    if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
    rc = check_ptrs(workspace);
    if (rc) return rc;
  }
  if (!device_error_ptr()) return MOE_ERR_CUDA;
  return cuda_status(launch_route(logits, T, E, k, block_n, topk_ids, topk_w, counts, offsets, perm, inv_perm,
                                  block_map, num_blocks, workspace, workspace_bytes,
                                  reinterpret_cast<cudaStream_t>(stream), 0));
}

int moe_rms_norm(const uint16_t* x, uint16_t* out, int T, int H, float eps, moe_stream_t stream) {
  if (T < 1 || T > (1 << 20) || H < 8 || H % 8 != 0 || !(eps >= 0.0f)) return MOE_ERR_SHAPE;
  int rc = check_ptrs(x, out);
  if (rc) return rc;
  return cuda_status(launch_rms_norm(x, out, T, H, eps, num_sms(), reinterpret_cast<cudaStream_t>(stream)));
}

int moe_norm_router(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, float eps, uint16_t* x_norm,
                    float* logits, moe_stream_t stream) {
  if (T < 1 || T > norm_router_max_tokens() || H < 8 || H % 8 != 0 || E < 1 || E > 1024 || !(eps >= 0.0f))
    return MOE_ERR_SHAPE;
  int rc = check_ptrs(x, w_router, x_norm, logits);
  if (rc) return rc;
  return cuda_status(
      launch_norm_router(x, w_router, x_norm, logits, T, H, E, eps, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_router(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, float* logits,
               int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  int rc = check_route_shape(T, E, k, 1);
  if (rc) return rc;
  if (H < 64 || H % 64 != 0 || E % 64 != 0 || E > 512) return MOE_ERR_SHAPE;
  rc = check_ptrs(x, w_router, logits, topk_ids, topk_w);
  if (rc) return rc;
  if (!device_error_ptr()) return MOE_ERR_CUDA;
  return cuda_status(launch_router(x, w_router, T, H, E, k, logits, topk_ids, topk_w,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int moe_route_x(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, int block_n, float* logits,
                int32_t* topk_ids, float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm,
                int32_t* inv_perm, int32_t* block_map, int32_t* num_blocks, void* workspace,
                size_t workspace_bytes, moe_stream_t stream) {
  int rc = check_route_shape(T, E, k, block_n);
  if (rc) return rc;
  if (H < 64 || H % 64 != 0 || E % 64 != 0 || E > 512) return MOE_ERR_SHAPE;
  rc = check_ptrs(x, w_router, logits, topk_ids, topk_w, counts, offsets, perm, inv_perm, block_map, num_blocks);
  if (rc) return rc;
  const size_t need = route_workspace_bytes(T, E, k);
  if (need > 0) {
    if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
    rc = check_ptrs(workspace);
    if (rc) return rc;
  }
  if (!device_error_ptr()) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = cuda_status(launch_router(x, w_router, T, H, E, k, logits, topk_ids, topk_w, s));
  if (rc) return rc;
  return cuda_status(launch_route(logits, T, E, k, block_n, topk_ids, topk_w, counts, offsets, perm, inv_perm,
                                  block_map, num_blocks, workspace, workspace_bytes, s, 1));
}

int moe_expert_gemm_w4(int mode, int impl, const uint16_t* act, int T, int H, int F, int E, int k,
                       const void* w_packed, const int32_t* perm, const float* topk_w, const int32_t* block_map,
                       const int32_t* num_blocks, int block_n, void* out, moe_stream_t stream) {
  int rc = check_shape(T, H, F, E, k, block_n);
  if (rc) return rc;
  if (mode != MOE_GATE_UP_SWIGLU && mode != MOE_DOWN) return MOE_ERR_MODE;
  rc = check_ptrs(act, w_packed, perm, topk_w, block_map, num_blocks, out);
  if (rc) return rc;
  if (impl == MOE_IMPL_AUTO) impl = block_n <= gemv_max_rows() ? MOE_IMPL_GEMV : MOE_IMPL_TC;
  if (impl != MOE_IMPL_GEMV && impl != MOE_IMPL_TC && impl != MOE_IMPL_TC2 && impl != MOE_IMPL_TC_BF16)
    return MOE_ERR_MODE;
  // the kernels step K and M by 128; the GEMV takes tiles of at most 8 rows, the tensor-core kernels
  // 128, the CTA-pair kernel 256
  if (H % 128 != 0 || F % 128 != 0) return MOE_ERR_SHAPE;
  if (block_n > (impl == MOE_IMPL_GEMV ? gemv_max_rows() : impl == MOE_IMPL_TC2 ? 256 : 128)) return MOE_ERR_SHAPE;
  if (!device_error_ptr()) return MOE_ERR_CUDA;
  const int cap = moe_block_map_capacity(T, E, k, block_n);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (impl == MOE_IMPL_GEMV)
    return cuda_status(launch_gemm_gemv(mode, act, T, H, F, E, k, w_packed, perm, topk_w, block_map, num_blocks,
                                        block_n, cap, out, num_sms(), s));
  if (impl == MOE_IMPL_TC2)
    return cuda_status(launch_gemm_pair(mode, act, T, H, F, E, k, w_packed, perm, block_map, num_blocks, block_n,
                                        cap, out, s));
  return cuda_status(launch_gemm_tc(mode, act, T, H, F, E, k, w_packed, perm, topk_w, block_map, num_blocks,
                                    block_n, cap, out, num_sms(), s, impl == MOE_IMPL_TC_BF16, nullptr, nullptr,
                                    nullptr));
}

int moe_expert_ffn_w4(const uint16_t* x, int T, int H, int F, int E, int k, const void* w13, const void* w2,
                      const int32_t* perm, const int32_t* block_map, const int32_t* num_blocks, int block_n,
                      uint16_t* y, moe_stream_t stream) {
  int rc = check_shape(T, H, F, E, k, block_n);
  if (rc) return rc;
  if (H % 128 != 0 || F % 256 != 0 || block_n > 64) return MOE_ERR_SHAPE;
  rc = check_ptrs(x, w13, w2, perm, block_map, num_blocks, y);
  if (rc) return rc;
  if (!device_error_ptr()) return MOE_ERR_CUDA;
  const int cap = moe_block_map_capacity(T, E, k, block_n);
  return cuda_status(launch_ffn_tc(x, T, H, F, E, k, w13, w2, perm, block_map, num_blocks, block_n, cap, y, num_sms(),
                                   reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_down_combine_workspace_size(int T, int H) {
  if (T < 1 || T > (1 << 20) || H < 128 || H % 128 != 0) return 0;
  return static_cast<size_t>(T) * (H / 128) * sizeof(int32_t);
}

int moe_down_combine(const uint16_t* h, int T, int H, int F, int E, int k, const void* w_packed, const int32_t* perm,
                     const int32_t* inv_perm, const float* topk_w, const int32_t* block_map,
                     const int32_t* num_blocks, int block_n, uint16_t* y, uint16_t* out, void* workspace,
                     size_t workspace_bytes, moe_stream_t stream) {
  int rc = check_shape(T, H, F, E, k, block_n);
  if (rc) return rc;
  if (H % 128 != 0 || F % 128 != 0 || block_n > 128) return MOE_ERR_SHAPE;
  rc = check_ptrs(h, w_packed, perm, inv_perm, topk_w, block_map, num_blocks, y, out, workspace);
  if (rc) return rc;
  if (workspace_bytes < moe_down_combine_workspace_size(T, H)) return MOE_ERR_WORKSPACE;
  if (!device_error_ptr()) return MOE_ERR_CUDA;
  const int cap = moe_block_map_capacity(T, E, k, block_n);
  return cuda_status(launch_gemm_tc(MOE_DOWN, h, T, H, F, E, k, w_packed, perm, topk_w, block_map, num_blocks,
                                    block_n, cap, y, num_sms(), reinterpret_cast<cudaStream_t>(stream), false, out,
                                    inv_perm, static_cast<int*>(workspace)));
}

size_t moe_expanded_bytes(int n_mat, int rows, int K) {
  if (n_mat < 1 || rows < 128 || rows % 128 != 0 || K < 64 || K % 64 != 0) return 0;
  return expanded_bytes(n_mat, rows, K);
}

int moe_expand_w4(const void* w_repacked, int n_mat, int rows, int K, void* out, moe_stream_t stream) {
  if (n_mat < 1 || rows < 128 || rows % 128 != 0 || K < 64 || K % 64 != 0) return MOE_ERR_SHAPE;
  int rc = check_ptrs(w_repacked, out);
  if (rc) return rc;
  return cuda_status(launch_expand(w_repacked, n_mat, rows, K, out, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_combine(const uint16_t* y, const int32_t* inv_perm, const float* topk_w, uint16_t* out, int T, int H,
                int k, moe_stream_t stream) {
  if (T < 1 || T > (1 << 20) || H < 8 || H % 8 != 0 || k < 1 || k > 32) return MOE_ERR_SHAPE;
  int rc = check_ptrs(y, inv_perm, topk_w, out);
  if (rc) return rc;
  if (!device_error_ptr()) return MOE_ERR_CUDA;
  return cuda_status(
      launch_combine(y, inv_perm, topk_w, out, T, H, k, num_sms(), reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_decode_workspace_size(int T, int H) {
  if (T < 1 || T > decode_max_tokens() || H < 64 || H % 32 != 0) return 0;
  return decode_workspace_bytes(T, H);
}

int moe_layer_forward(const uint16_t* x, const float* logits, uint16_t* out, int T, int H, int F, int E, int k,
                      int block_n, int impl, const moe_weights_t* w, const moe_buffers_t* b, moe_stream_t stream) {
  if (!w || !b) return MOE_ERR_NULL;
  const bool gemv = impl == MOE_IMPL_GEMV || (impl == MOE_IMPL_AUTO && block_n <= gemv_max_rows());
  if (gemv && b->decode_ws && T <= decode_max_tokens() && k <= 32) {
    // the fused decode kernel: routing, both GEMVs and the combine in one launch
    int rc = check_shape(T, H, F, E, k, block_n);
    if (rc) return rc;
    if (block_n > gemv_max_rows() || H % 128 != 0 || F % 128 != 0) return MOE_ERR_SHAPE;
    rc = check_ptrs(x, logits, out, w->w13, w->w2, b->topk_ids, b->topk_w, b->counts, b->offsets, b->perm,
                    b->inv_perm, b->block_map, b->num_blocks, b->h, b->y, b->decode_ws);
    if (rc) return rc;
    if (b->decode_ws_bytes < decode_workspace_bytes(T, H)) return MOE_ERR_WORKSPACE;
    if (!device_error_ptr()) return MOE_ERR_CUDA;
    return cuda_status(launch_decode(x, logits, w->w13, w->w2, T, H, F, E, k, block_n, b->topk_ids, b->topk_w,
                                     b->counts, b->offsets, b->perm, b->inv_perm, b->block_map, b->num_blocks, b->h,
                                     b->y, out, b->decode_ws, wait_limit_ns(), num_sms(),
                                     reinterpret_cast<cudaStream_t>(stream)));
  }
  int rc = moe_route(logits, T, E, k, block_n, b->topk_ids, b->topk_w, b->counts, b->offsets, b->perm, b->inv_perm,
                     b->block_map, b->num_blocks, b->workspace, b->workspace_bytes, stream);
  if (rc) return rc;
  const int resolved = impl == MOE_IMPL_AUTO ? (block_n <= gemv_max_rows() ? MOE_IMPL_GEMV : MOE_IMPL_TC) : impl;
  if (resolved == MOE_IMPL_TC && !b->combine_ws && block_n <= 64 && H % 128 == 0 && F % 256 == 0) {
    // tiles of at most 64 rows: both projections of a tile in one launch, h kept in shared memory
    // (the same bits of y; measured faster than the two GEMMs at these tile heights)
    rc = moe_expert_ffn_w4(x, T, H, F, E, k, w->w13, w->w2, b->perm, b->block_map, b->num_blocks, block_n, b->y,
                           stream);
    if (rc) return rc;
    return moe_combine(b->y, b->inv_perm, b->topk_w, out, T, H, k, stream);
  }
  rc = moe_expert_gemm_w4(MOE_GATE_UP_SWIGLU, impl, x, T, H, F, E, k, w->w13, b->perm, b->topk_w, b->block_map,
                          b->num_blocks, block_n, b->h, stream);
  if (rc) return rc;
  if (resolved == MOE_IMPL_TC && b->combine_ws) {
    // the down GEMM with the combine in its epilogue (one launch fewer, y read back from L2 at once)
    return moe_down_combine(b->h, T, H, F, E, k, w->w2, b->perm, b->inv_perm, b->topk_w, b->block_map,
                            b->num_blocks, block_n, b->y, out, b->combine_ws, b->combine_ws_bytes, stream);
  }
  rc = moe_expert_gemm_w4(MOE_DOWN, impl, b->h, T, H, F, E, k, w->w2, b->perm, b->topk_w, b->block_map,
                          b->num_blocks, block_n, b->y, stream);
  if (rc) return rc;
  return moe_combine(b->y, b->inv_perm, b->topk_w, out, T, H, k, stream);
}

// The device's address of host memory it can read and write directly (pinned or registered, and
// mapped), or nullptr (pageable memory, or an address the runtime does not know).
static void* host_device_view(const void* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();  // an unknown pointer is not an error of this call
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int moe_layer_forward_host(const uint16_t* x_host, const float* logits_host, uint16_t* out_host, uint16_t* x_dev,
                           float* logits_dev, uint16_t* out_dev, int T, int H, int F, int E, int k, int block_n,
                           int impl, const moe_weights_t* w, const moe_buffers_t* b, moe_stream_t stream) {
  if (!x_host || !logits_host || !out_host) return MOE_ERR_NULL;
  int rc = check_shape(T, H, F, E, k, block_n);
  if (rc) return rc;
  rc = check_ptrs(x_dev, logits_dev, out_dev);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t xb = static_cast<size_t>(T) * H * sizeof(uint16_t);
  const size_t lb = static_cast<size_t>(T) * E * sizeof(float);
  // Pinned host buffers are read and written by the kernels over the host link where each byte
  // crosses it once anyway: the routing (or fused decode) kernel reads every logit once, and the
  // combine writes out straight to out_host, which saves two copy-engine operations and their
  // latency per call.  x, which the grouped GEMM gathers k + 1 times, is copied to x_dev first.
  // Pageable buffers go through logits_dev / out_dev with copies.
  const float* logits_view = static_cast<const float*>(host_device_view(logits_host));
  uint16_t* out_view = static_cast<uint16_t*>(host_device_view(out_host));
  if (logits_view && !aligned16(logits_view)) logits_view = nullptr;
  if (out_view && !aligned16(out_view)) out_view = nullptr;
  if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (!logits_view &&
      cudaMemcpyAsync(logits_dev, logits_host, lb, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  rc = moe_layer_forward(x_dev, logits_view ? logits_view : logits_dev, out_view ? out_view : out_dev, T, H, F, E, k,
                         block_n, impl, w, b, stream);
  if (rc) return rc;
  if (!out_view && cudaMemcpyAsync(out_host, out_dev, xb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_get_device_error(int32_t* code) {
  if (!code) return MOE_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, MOE_ERROR_SYMBOL, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(MOE_ERROR_SYMBOL, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  return MOE_OK;
}

size_t moe_repacked_bytes(int n_mat, int rows, int K) {
  if (n_mat < 1 || rows < 128 || rows % 128 != 0 || K < 64 || K % 64 != 0) return 0;
  return repacked_bytes(n_mat, rows, K);
}

int moe_repack_w4(const uint32_t* packed, const uint16_t* scale, const uint16_t* bias, int n_mat, int rows, int K,
                  int gate_up, void* out, moe_stream_t stream) {
  if (n_mat < 1 || rows < 128 || rows % 128 != 0 || K < 64 || K % 64 != 0) return MOE_ERR_SHAPE;
  if (gate_up < 0 || gate_up > 2) return MOE_ERR_MODE;
  if (gate_up == 1 && (rows / 2) % 128 != 0) return MOE_ERR_SHAPE;
  if (gate_up == 2 && (rows / 2) % 64 != 0) return MOE_ERR_SHAPE;
  int rc = check_ptrs(packed, scale, bias, out);
  if (rc) return rc;
  return cuda_status(launch_repack(packed, scale, bias, n_mat, rows, K, gate_up, out,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

void moe_set_wait_limit_ns(uint64_t ns) { set_wait_limit_ns(ns); }

size_t moe_trace_words(void) {
#ifdef MOE_TRACE
  return moe::TRACE_WORDS;
#else
  return 0;
#endif
}

int moe_trace_reset(moe_stream_t stream) {
#ifdef MOE_TRACE
  int* err = moe::device_error_ptr();
  if (!err) return MOE_ERR_CUDA;
  return moe::cuda_status(cudaMemsetAsync(err + moe::TRACE_ERR_INTS, 0,
                                          moe::TRACE_WORDS * sizeof(unsigned long long),
                                          reinterpret_cast<cudaStream_t>(stream)));
#else
  (void)stream;
  return MOE_ERR_MODE;
#endif
}

int moe_trace_read(uint64_t* host, size_t words) {
#ifdef MOE_TRACE
  if (!host) return MOE_ERR_NULL;
  int* err = moe::device_error_ptr();
  if (!err) return MOE_ERR_CUDA;
  const size_t n = words < moe::TRACE_WORDS ? words : moe::TRACE_WORDS;
  return cudaMemcpy(host, err + moe::TRACE_ERR_INTS, n * sizeof(uint64_t), cudaMemcpyDeviceToHost) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
#else
  (void)host;
  (void)words;
  return MOE_ERR_MODE;
#endif
}

}  // extern "C"
