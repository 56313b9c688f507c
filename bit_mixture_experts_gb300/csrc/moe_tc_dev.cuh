// Device helpers shared by the tensor-core grouped GEMMs (moe_gemm_tc.cu, one
// CTA per work unit, and moe_gemm_pair.cu, a CTA pair per work unit): the
// repacked weight block and its expansion to bf16.
#pragma once
#include "moe_common.cuh"
#include "moe_ptx.cuh"

namespace moe {
namespace tc_dev {

constexpr int TC_M = 128;              // weight rows per M-tile (the MMA's M on one SM)
constexpr int KG = 64;                 // one quantisation group
constexpr int W_PACKED = TC_M * 32;    // packed nibbles of one M-tile x K group
constexpr int W_BLOCK = W_PACKED + TC_M * 4;  // + (scale, bias) per row: one repacked block

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

// One quant group of one weight row: 64 nibbles (two uint4 of the repacked
// block) and its (scale, bias) bf16 pair -> 32 bf16x2 words of
// w = bf16(q * scale + bias).  128 + q is exact in bf16 (0x4300 | q), the
// subtraction of 128 is exact, and the fma rounds once.
__device__ __forceinline__ void expand_group(const uint4 p0, const uint4 p1, uint32_t sb, uint32_t (&v)[32]) {
  const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  const uint32_t s2 = (sb & 0xffffu) * 0x10001u;
  const uint32_t b2 = (sb >> 16) * 0x10001u;
  constexpr uint32_t MAGIC = 0x43004300u;  // bf16 pair (128, 128)
#pragma unroll
  for (int w = 0; w < 8; ++w) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // nibbles of K elements 8w+2j (low half) and 8w+2j+1 (high half): 128+q exactly
      const uint32_t x = ((words[w] >> (4 * j)) & 0x000f000fu) | MAGIC;
      v[4 * w + j] = ptx::bf16x2_fma(ptx::bf16x2_sub(x, MAGIC), s2, b2);
    }
  }
}

// Bounded waits.  The time limit is counted in SM clock cycles (clock64, cheap
// to read) from the first unsuccessful try; `limit` is in cycles.
//
// Bounded wait on phase `parity` of `bar` by a whole warp.  Returns false on
// timeout or when another role has already given up (s_abort); the decision
// is warp-uniform (lane 0's clock).
__device__ __forceinline__ bool wait_warp_untraced(uint32_t bar, uint32_t parity, volatile int* s_abort, int* err,
                                                   unsigned long long limit, uint32_t sleep_ns) {
  // the first probe does not block: a try_wait without a time hint may wait for a while inside the
  // instruction, past a short limit, without the limit being checked
  if (__all_sync(0xffffffffu, ptx::mbar_test_wait(bar, parity))) return true;
  const long long t0 = clock64();
  for (;;) {
    // sleep in hardware until the phase completes (or about 20 us pass) rather than polling; a limit
    // shorter than 20 us is polled without sleeping instead: the sleep time is only a hint, which
    // the hardware may exceed, and a short limit must be checked on time
    const bool done = sleep_ns >= 20000u ? ptx::mbar_try_wait_sleep(bar, parity, sleep_ns)
                                         : ptx::mbar_test_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    int give_up = *s_abort;
    if (!give_up && static_cast<unsigned long long>(clock64() - t0) > limit) give_up = 2;
    give_up = __shfl_sync(0xffffffffu, give_up, 0);
    if (give_up) {
      if (give_up == 2 && (threadIdx.x & 31) == 0) {
        set_device_error(err, MOE_DEV_TIMEOUT);
        *s_abort = 1;
      }
      return false;
    }
  }
}

#ifdef MOE_TRACE
// Trace build only (libmoe_w4_trace.so, moe_trace_read): per (CTA, warp) statistics of the waits
// above, in the words that follow the device error word there: cycles waited, waits, the complement
// (2^64 - 1 - t) of clock64 at the start of the first wait, and clock64 at the end of the last.  Lane
// 0 adds them with reductions whose result is not read, so a traced wait costs a few issued
// instructions and no round trip to memory.
constexpr int TRACE_CTAS = 1024;
constexpr int TRACE_ERR_INTS = 64;  // the error word's block before the trace words
__device__ __forceinline__ void trace_wait(int* err, long long t0, long long t1) {
  if ((threadIdx.x & 31) != 0) return;
  unsigned long long* w = reinterpret_cast<unsigned long long*>(err + TRACE_ERR_INTS) +
                          4 * ((blockIdx.x % TRACE_CTAS) * 32 + (threadIdx.x >> 5));
  atomicAdd(w, static_cast<unsigned long long>(t1 - t0));
  atomicAdd(w + 1, 1ull);
  atomicMax(w + 2, ~static_cast<unsigned long long>(t0));
  atomicMax(w + 3, static_cast<unsigned long long>(t1));
}
#endif

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* s_abort, int* err,
                                          unsigned long long limit, uint32_t sleep_ns) {
#ifdef MOE_TRACE
  const long long t0 = clock64();
  const bool r = wait_warp_untraced(bar, parity, s_abort, err, limit, sleep_ns);
  trace_wait(err, t0, clock64());
  return r;
#else
  return wait_warp_untraced(bar, parity, s_abort, err, limit, sleep_ns);
#endif
}

// Wait that ignores s_abort (used to drain copies and MMAs already in flight
// before the CTA exits).  Whatever the configured limit, it waits at least
// DRAIN_MIN_CYCLES (about 10 ms): a copy still landing in shared memory or an
// MMA still using TMEM must not outlive the CTA, even when a very short wait
// limit made the kernel give up early.
constexpr unsigned long long DRAIN_MIN_CYCLES = 20000000ull;

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  if (limit < DRAIN_MIN_CYCLES) limit = DRAIN_MIN_CYCLES;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (static_cast<unsigned long long>(clock64() - t0) > limit) return;
  }
}

// silu(g) = g / (1 + e^-g) with the fast exponential and division; the
// product with u is rounded to bf16 afterwards, which hides their few-ulp
// error except within a few FP32 ulps of a bf16 rounding boundary.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

}  // namespace tc_dev
}  // namespace moe
