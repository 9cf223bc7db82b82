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

// try_wait that lets the hardware suspend the thread for up to kSuspendNs
// while the phase is incomplete (it resumes as soon as the phase completes),
// so that a waiting warp does not spin on issue slots its neighbours need.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return done != 0;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second

// Wait for phase `parity` of `bar` to complete, giving up after about a second.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  while (!mbar_try_wait_suspend(bar, parity)) {
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
  while (!mbar_try_wait_suspend(bar, parity)) {
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

// Global -> shared tensor copies (TMA tiles) of a box at integer coordinates
// (innermost first), completing on `bar`.  The tensor map lives in kernel
// parameter space (a __grid_constant__ argument); rows outside the tensor
// arrive as zeros.  The innermost coordinate times the element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// ----------------------------------------------------------------------------
// Tensor cores (tcgen05), tensor memory
// ----------------------------------------------------------------------------
// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (8-row atoms of 128-byte rows, 1024-byte aligned): start
// address, leading byte offset 16 (unused for this layout), stride byte
// offset 1024 between 8-row atoms, descriptor version 1, swizzle mode 2.
// Advancing K by 8 fp32 (32 bytes) inside the atom adds 2 to the descriptor.
__device__ __forceinline__ uint64_t umma_desc_sw128(const void* tile) {
  const uint64_t addr = smem_u32(tile);
  return ((addr & 0x3FFFF) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::tf32: fp32 accumulate, tf32 A
// and B, both K-major, M x N (M in {64, 128}, N a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t umma_idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma this thread has issued so far completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Allocate `cols` tensor-memory columns (a power of two >= 32) for this CTA;
// the whole warp executes it and the base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

// 16 consecutive fp32 columns of the warp's 32 tensor-memory lanes: lane i of
// the warp gets row (lane base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of element (r, k), k < 32, of a K-major fp32 tile stored with
// the 128-byte swizzle: the 16-byte chunk k / 4 of row r sits at chunk
// (k / 4) xor (r mod 8) of its 128-byte row.
__device__ __forceinline__ int sw128_offset(int r, int k) {
  return (r >> 3) * 1024 + (r & 7) * 128 + (((k >> 2) ^ (r & 7)) << 4) + (k & 3) * 4;
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

// ----------------------------------------------------------------------------
// The convolution output code.  The conv runs in fp32, as causal_conv1d_update
// does, and the code stored for every later step is bf16(SiLU(y)).  So that
// the code does not depend on how a compiler or a math library evaluates it,
// every step is an IEEE-754 fp32 add, multiply or fma, or integer arithmetic
// on the bits, in a fixed order, with no branch:
//   y = w0 x0, then y = fma(wj, xj, y) for the newer taps j = 1 .. W-1;
//   z = e^-|y|: x = max(-|y|, -104) (e^-104 rounds to 0); n = x log2 e rounded
//     to nearest even, from the exact product, by one fma with 1.5 * 2^23
//     (whose ulp is 1, so n sits in the low mantissa bits); Cody-Waite
//     reduction r = x - n ln2 with ln2 split in a 15-bit head (n times it is
//     exact) and a tail; e^r by its Taylor series to r^7/7! in Horner form
//     (|r| <= 0.347, truncation under 1e-8 relative); z = e^r 2^n1 2^n2 with
//     n1 = floor(n/2), n2 = n - n1 (the first scaling is exact, the second
//     rounds once);
//   1/(1+z), 1+z in [1, 2]: r0 = 24/17 - (8/17)(1+z), then three Newton steps;
//   SiLU(y) = y sigma with sigma = 1/(1+z) for y >= 0 and z/(1+z) below.
// e^x is within one fp32 ulp of exact, SiLU within four.
// ----------------------------------------------------------------------------
// Two codes at once (tokens a and b of one channel) on the packed fp32x2 unit:
// every half runs exactly the sequence described above, operation by
// operation (fma(-n, c, x) is computed as fma(n, -c, x), the same exact value).
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

__device__ __forceinline__ float2 silu_f32x2(float2 y) {
  constexpr float kLog2e = 0x1.715476p+0f;
  constexpr float kShifter = 0x1.8p+23f;
  constexpr float kLn2Hi = 0x1.62e4p-1f;
  constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
  // z = e^x, x = max(-|y|, -104)
  const float2 x = make_float2(fmaxf(-fabsf(y.x), -104.0f), fmaxf(-fabsf(y.y), -104.0f));
  // n = rint(x log2 e) through the shifter, lane by lane on the scalar unit
  const float ta = __fmaf_rn(x.x, kLog2e, kShifter), tb = __fmaf_rn(x.y, kLog2e, kShifter);
  const float2 nf = make_float2(__fsub_rn(ta, kShifter), __fsub_rn(tb, kShifter));
  const int na = __float_as_int(ta) - __float_as_int(kShifter);
  const int nb = __float_as_int(tb) - __float_as_int(kShifter);
  float2 r = __ffma2_rn(nf, f2(-kLn2Hi), x);
  r = __ffma2_rn(nf, f2(-kLn2Lo), r);
  // 1/k! rounded to fp32, k = 7 .. 2
  float2 q = f2(0x1.a01a02p-13f);
  q = __ffma2_rn(q, r, f2(0x1.6c16c2p-10f));
  q = __ffma2_rn(q, r, f2(0x1.111112p-7f));
  q = __ffma2_rn(q, r, f2(0x1.555556p-5f));
  q = __ffma2_rn(q, r, f2(0x1.555556p-3f));
  q = __ffma2_rn(q, r, f2(0.5f));
  q = __ffma2_rn(q, r, f2(1.0f));
  q = __ffma2_rn(q, r, f2(1.0f));
  const int na1 = na >> 1, nb1 = nb >> 1;  // arithmetic shift: floor(n / 2)
  q = __fmul2_rn(q, make_float2(__int_as_float((na1 + 127) << 23), __int_as_float((nb1 + 127) << 23)));
  const float2 z =
      __fmul2_rn(q, make_float2(__int_as_float((na - na1 + 127) << 23), __int_as_float((nb - nb1 + 127) << 23)));
  // 1/(1+z), 1+z in [1, 2]: linear start, three Newton steps
  const float2 d = __fadd2_rn(f2(1.0f), z);
  const float2 dn = make_float2(-d.x, -d.y);
  float2 rc = __ffma2_rn(f2(-0x1.e1e1e2p-2f), d, f2(0x1.69696ap+0f));
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const float2 e = __ffma2_rn(dn, rc, f2(1.0f));
    rc = __ffma2_rn(rc, e, rc);
  }
  const float2 sigma = __fmul2_rn(make_float2(y.x >= 0.0f ? 1.0f : z.x, y.y >= 0.0f ? 1.0f : z.y), rc);
  return __fmul2_rn(y, sigma);
}

// bf16 codes of SiLU(sum_j w_j x_j) for two windows xa, xb of one channel
// (W = 4 taps, oldest first): the low half holds a, the high half b.
__device__ __forceinline__ uint32_t conv_silu_bf16x2(const float w[4], const float xa[4], const float xb[4]) {
  float2 y = __fmul2_rn(f2(w[0]), make_float2(xa[0], xb[0]));
  y = __ffma2_rn(f2(w[1]), make_float2(xa[1], xb[1]), y);
  y = __ffma2_rn(f2(w[2]), make_float2(xa[2], xb[2]), y);
  y = __ffma2_rn(f2(w[3]), make_float2(xa[3], xb[3]), y);
  const float2 s = silu_f32x2(y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(s.x, s.y);
  return *reinterpret_cast<const uint32_t*>(&b);
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

// e^g for the KDA gate with the hardware approximations (ex2 / lg2): g feeds
// only the decay, where a few 1e-7 of relative error is far below the bf16
// outputs' resolution.  softplus(u) = log(1 + e^u) below 20, u above.
__device__ __forceinline__ float kda_decay_fast(float raw_g, float dt_bias, float A, int lower_bound_gate,
                                                float lower_bound) {
  const float u = raw_g + dt_bias;
  float g;
  if (lower_bound_gate)
    g = __fdividef(lower_bound, 1.0f + __expf(-A * u));
  else
    g = -A * ((u > 20.0f) ? u : __logf(1.0f + __expf(u)));
  return __expf(g);
}

__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace kda
