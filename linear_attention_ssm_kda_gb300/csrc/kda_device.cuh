// kda_device.cuh -- device helpers shared by the verify and commit kernels:
// bulk-copy (TMA) and mbarrier wrappers in inline PTX, bounded waits, bf16
// conversions, the device error report, and the KDA gate.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"
#include "kda_params.h"

namespace kda {

// ----------------------------------------------------------------------------
// Error report
// ----------------------------------------------------------------------------
__device__ __forceinline__ void report(int* ws, int bits, int item) {
  if (ws != nullptr) {
    atomicOr(ws, bits);
    atomicExch(ws + 1, item);
  }
}

// ----------------------------------------------------------------------------
// Shared-memory addresses, mbarriers and bulk copies
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make the initialised barrier visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second

// Wait for phase `parity` of `bar` to complete, giving up after about a second.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - start > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Like mbar_wait_bounded, but also gives up as soon as *abort is set (another
// role of the CTA has timed out and the pipeline is being torn down).
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_timer_ns() - start > kWaitLimitNs) return false;
  }
  return true;
}

// Barrier over a subset of the CTA's warps (ids 1..15; `threads` a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Global -> shared bulk copy (TMA, non-tensor), completing on `bar`.
// dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared -> global bulk copy (TMA store), tracked by the issuing thread's bulk
// groups.  dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until the committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ----------------------------------------------------------------------------
// bf16 conversions
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Round to nearest even (hardware cvt.rn.bf16.f32).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Round a double straight to bf16 (nearest even): first to fp32 with
// round-to-odd (truncate, then set the last bit when inexact), which keeps
// the information the second rounding needs since fp32 carries more than two
// extra bits over bf16; then round that fp32 to bf16.
__device__ __forceinline__ uint16_t f64_to_bf16(double x) {
  float f = __double2float_rz(x);
  if (static_cast<double>(f) != x) f = __uint_as_float(__float_as_uint(f) | 1u);
  return f32_to_bf16(f);
}

// Error-free sum: a + b == s + e exactly (Knuth's TwoSum, any magnitudes).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// The rare fp64 evaluation of bf16_rne(silu(sum_j w_j x_j)), kept out of line.
static __device__ __noinline__ uint16_t conv_silu_bf16_fp64(float w0, float w1, float w2, float w3, float x0,
                                                             float x1, float x2, float x3) {
  double yd = 0.0;
  yd += static_cast<double>(w0) * static_cast<double>(x0);
  yd += static_cast<double>(w1) * static_cast<double>(x1);
  yd += static_cast<double>(w2) * static_cast<double>(x2);
  yd += static_cast<double>(w3) * static_cast<double>(x3);
  return f64_to_bf16(yd / (1.0 + exp(-yd)));
}

// bf16_rne(silu(y)) for y = sum_j w_j x_j (W = 4 taps), rounded from the exact
// value of y.  y is carried as an unevaluated pair y + yr: the products are
// exact in fp32 for bf16 weights (fp32 weights add their fma residuals), and
// TwoSum keeps every addition error, so y + yr is y to within 2^-44 of
// M = |p0 + p1| + |p2 + p3| (2^-40 sum|w_j x_j| for fp32 weights).
// silu(y) = y * sigma, sigma = 1 / (1 + expf(-y)) with expf within 2 ulp and
// __fdividef within 2 ulp: relative error below 5 ulp < 2^-20; the first-order
// term silu'(y) yr is added.  If [s - bound, s + bound] rounds to a single
// bf16 value (all but ~5e-4 of values) that is the answer; otherwise fp64.
__device__ __forceinline__ uint16_t conv_silu_bf16(const float w[4], const float x[4], bool exact_products) {
  const float p0 = __fmul_rn(w[0], x[0]), p1 = __fmul_rn(w[1], x[1]);
  const float p2 = __fmul_rn(w[2], x[2]), p3 = __fmul_rn(w[3], x[3]);
  float s01, e01, s23, e23, yh, e;
  two_sum(p0, p1, s01, e01);
  two_sum(p2, p3, s23, e23);
  two_sum(s01, s23, yh, e);
  float yl = __fadd_rn(__fadd_rn(e01, e23), e);
  float margin = (fabsf(s01) + fabsf(s23)) * 0x1p-44f;
  if (!exact_products) {
    const float r0 = __fmaf_rn(w[0], x[0], -p0), r1 = __fmaf_rn(w[1], x[1], -p1);
    const float r2 = __fmaf_rn(w[2], x[2], -p2), r3 = __fmaf_rn(w[3], x[3], -p3);
    yl = __fadd_rn(yl, __fadd_rn(__fadd_rn(r0, r1), __fadd_rn(r2, r3)));
    margin = (fabsf(p0) + fabsf(p1) + fabsf(p2) + fabsf(p3)) * 0x1p-40f;
  }
  float y, yr;
  two_sum(yh, yl, y, yr);
  if (fabsf(y) <= 80.0f) {
    const float sig = __fdividef(1.0f, 1.0f + expf(-y));
    float s = y * sig;
    const float dsilu = sig * (1.0f + y * (1.0f - sig));  // silu'(y)
    s = __fmaf_rn(dsilu, yr, s);
    const float bound = fabsf(s) * 0x1p-20f + margin + 0x1p-126f;
    const uint16_t lo = f32_to_bf16(__fsub_rd(s, bound));
    const uint16_t hi = f32_to_bf16(__fadd_ru(s, bound));
    if (lo == hi) return lo;
  }
  return conv_silu_bf16_fp64(w[0], w[1], w[2], w[3], x[0], x[1], x[2], x[3]);
}

// ----------------------------------------------------------------------------
// KDA gate ("vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py", _kda_gate)
// ----------------------------------------------------------------------------
__device__ __forceinline__ float kda_gate(float raw_g, float dt_bias, float A, int lower_bound_gate,
                                          float lower_bound) {
  const float u = raw_g + dt_bias;
  if (lower_bound_gate) return lower_bound / (1.0f + expf(-A * u));
  const float sp = (u > 20.0f) ? u : log1pf(expf(u));
  return -A * sp;
}

__device__ __forceinline__ float sigmoidf(float x) { return 1.0f / (1.0f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace kda
