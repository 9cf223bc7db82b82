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

// try_wait: while the phase is incomplete the hardware may suspend the
// thread, up to its own time limit (it resumes as soon as the phase
// completes), so a waiting warp does not spin on issue slots its neighbours
// need.  An explicit 20 us suspend hint measured slower: about 0.6 % on the
// C2 and C4 verify, 4 % on the C3 (tensor-core) verify; 1 us and 100 us
// were no different from 20 us.
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

// Wait for phase `parity` of `bar` to complete, giving up after limit_ns
// (about a second unless a caller sets a shorter limit).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - start > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Like mbar_wait_bounded, but also gives up as soon as *abort is set (another
// role of the CTA has timed out and the pipeline is being torn down).
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                                   uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_timer_ns() - start > limit_ns) return false;
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

// Programmatic dependent launch: wait until the grid launched before this one
// in the stream has completed with its memory visible (a no-op when this grid
// was launched without the attribute), then order that view before this
// thread's later bulk copies, which read through the async proxy.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ----------------------------------------------------------------------------
// bf16 conversions
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Round to nearest even (hardware cvt.rn.bf16.f32).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ----------------------------------------------------------------------------
// The convolution output code: bf16_rne(SiLU(y)), y = sum_j w_j x_j over the
// W = 4 taps, rounded once from the mathematical value
// ("vllm.models.kimi_k3.nvidia.specialized_decode.recoverssm.state",
// deferred_recoverssm_verify: causal_conv1d_update with activation "silu",
// output in the activation dtype).  Three tiers decide it:
//   1. fp32 (conv_silu_bf16x2, two codes at once on the packed fp32x2
//      unit): y by an fma chain, SiLU on the special-function unit
//      (silu_f32x2), and a
//      bound E on |computed - exact|.  When no bf16 rounding boundary lies
//      within E of the computed value, the hardware rounding of it is the
//      correctly rounded code.  Otherwise the code is marked doubtful (about
//      6 in 10^4 codes on the decode workloads' data, 2 in 10^3 with
//      outliers).
//   2. float-float (conv_code_ff): y exactly as a pair of floats, e^-|y| by a
//      32-entry table and a short series, SiLU by a pair-of-floats quotient,
//      relative error far below 2^-36; for |y| <= 87 it decides every code
//      not within 2^-36 of a boundary.
//   3. double (conv_code_f64): the definition evaluated in fp64 (exact
//      products, the sum in tap order, y / (1 + e^-y)) and rounded once, for
//      what tier 2 leaves.  conv_code_exact runs tiers 2 and 3.
// ----------------------------------------------------------------------------
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// SiLU(y) = y sigma(y), sigma = 1 / (1 + e^-y), on the special-function unit:
//   e^-y = 2^(-y log2 e) with the argument split exactly: th = RN(-y L) for
//     L = log2 e rounded to fp32, r = fma(-y, L, -th) (the product's exact
//     rounding error) and tl = r - y (log2 e - L); then e^-y =
//     ex2(th) (1 + tl ln 2) (tl is below 2^-16 |th|, so the series' next term
//     is far below the unit's own error).  y is clamped at 104, past which
//     e^-y is below the fp32 range and sigma is 1;
//   sigma by the unit's reciprocal of 1 + e^-y, SiLU = y sigma.
// Its relative error against the exact SiLU of the fp32 input is at most
// kSiluRelErr for every y >= -80 (checked over all fp32 inputs on GB300).
// sigma is returned for the error bound.
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float2 silu_f32x2(float2 y, float2& sigma) {
  constexpr float kL = 0x1.715476p+0f;     // log2 e to fp32
  constexpr float kLlo = 0x1.4ae0cp-26f;   // log2 e - kL
  constexpr float kLn2 = 0x1.62e43p-1f;
  const float2 yc = make_float2(fminf(y.x, 104.0f), fminf(y.y, 104.0f));
  const float2 th = __fmul2_rn(yc, f2(-kL));
  const float2 r = __ffma2_rn(yc, f2(-kL), make_float2(-th.x, -th.y));
  const float2 tl = __ffma2_rn(yc, f2(-kLlo), r);
  float2 e = make_float2(ex2_approx(th.x), ex2_approx(th.y));
  e = __ffma2_rn(e, __fmul2_rn(tl, f2(kLn2)), e);
  const float2 d = __fadd2_rn(f2(1.0f), e);
  sigma = make_float2(rcp_approx(d.x), rcp_approx(d.y));
  return __fmul2_rn(y, sigma);
}

// Relative error bound of silu_f32x2 (in units of 2^-24, with margin over the
// largest error seen across all fp32 inputs >= -80: 5.58) and the lowest y
// tier 1 serves (below it e^-|y| nears the subnormal range).
constexpr float kSiluRelErr = 6.0f * 0x1p-24f;
constexpr float kTier1MinY = -80.0f;

// Tier 1: the bf16 codes of SiLU(sum_j w_j x_j) for two windows a and b,
// each with its own weights (W = 4 taps, oldest first): two channels at one
// token, or two tokens of one channel.  The low half of the result holds a,
// the high half b; bits 0 / 1 of *doubt tell whether the code of a / b must
// be decided by the exact tiers.
//
// The fma chain starts from +0, so an exactly zero sum is +0 (SiLU(0) = +0).
// Its error dy is at most u (|y_2| + |y_3| + |y_4|) over the partial sums y_k,
// u = 2^-24, plus u |y_1| for fp32 weights (a bf16 weight times a bf16 input
// is exact; e0 is 1 for fp32 weights (kW32) and 0 for bf16), so
// dy^2 <= 4 u^2 (e0 y_1^2 + y_2^2 + y_3^2 + y_4^2).  The conv error moves s by
// at most slope dy, where |SiLU'| <= 1.1 everywhere and |SiLU'(t)| =
// |sigma(t) + SiLU(t)(1 - sigma(t))| <= sigma + |SiLU|, which over
// [y - dy, y + dy] stays below sigma + |s| + 1.35 dy; hence
// slope^2 <= min(1.21, 4 (sigma^2 + s^2) + 4 dy^2).  With the evaluation error
// kSiluRelErr |s|, the total error E obeys E^2 <= 2 kSiluRelErr^2 s^2 +
// 2 slope^2 dy^2.  The code is certain when the square of the distance from s
// to the midpoint of its bf16 interval exceeds that bound, and the bound stays
// below 2^-20 s^2 (the next midpoint is at least 2^-10 |s| away).  The
// constants carry slack for the bound's own rounding; the 2^-126 term makes
// every |s| below 2^-63 doubtful, where the squares leave the normal range.
template <bool kW32>
__device__ __forceinline__ uint32_t conv_silu_bf16x2(const float wa[4], const float wb[4], const float xa[4],
                                                     const float xb[4], uint32_t* doubt) {
  constexpr float k4U2 = 0x1.0001p-46f;                            // 4 u^2
  constexpr float k2Eps2 = 2.0f * 36.0f * 0x1p-48f * 1.0001f;       // 2 kSiluRelErr^2
  const float2 y1 = __ffma2_rn(make_float2(wa[0], wb[0]), make_float2(xa[0], xb[0]), f2(0.0f));
  const float2 y2 = __ffma2_rn(make_float2(wa[1], wb[1]), make_float2(xa[1], xb[1]), y1);
  const float2 y3 = __ffma2_rn(make_float2(wa[2], wb[2]), make_float2(xa[2], xb[2]), y2);
  const float2 y = __ffma2_rn(make_float2(wa[3], wb[3]), make_float2(xa[3], xb[3]), y3);
  float2 sigma;
  const float2 s = silu_f32x2(y, sigma);
  // dy^2 bound
  float2 q;
  if constexpr (kW32)
    q = __ffma2_rn(y2, y2, __fmul2_rn(y1, y1));
  else
    q = __fmul2_rn(y2, y2);
  q = __ffma2_rn(y3, y3, q);
  q = __ffma2_rn(y, y, q);
  const float2 dy2 = __fmul2_rn(f2(k4U2), q);
  const float2 s2 = __fmul2_rn(s, s);
  const float2 sl = __ffma2_rn(f2(4.001f), __ffma2_rn(sigma, sigma, s2), __fmul2_rn(f2(4.001f), dy2));
  const float2 sl2 = make_float2(fminf(1.2101f, sl.x), fminf(1.2101f, sl.y));
  const float2 bound = __ffma2_rn(f2(k2Eps2), s2, __ffma2_rn(f2(2.001f), __fmul2_rn(sl2, dy2), f2(0x1p-126f)));
  const float2 mid = make_float2(__uint_as_float((__float_as_uint(s.x) & 0xFFFF0000u) | 0x8000u),
                                 __uint_as_float((__float_as_uint(s.y) & 0xFFFF0000u) | 0x8000u));
  const float2 dist = __fadd2_rn(s, make_float2(-mid.x, -mid.y));  // exact: s and mid lie within a factor 2
  const float2 d2 = __fmul2_rn(dist, dist);
  const float2 reach = __fmul2_rn(f2(0x1p-20f), s2);
  const bool da = !(d2.x > bound.x) || !(bound.x < reach.x) || !(y.x >= kTier1MinY);
  const bool db = !(d2.y > bound.y) || !(bound.y < reach.y) || !(y.y >= kTier1MinY);
  *doubt = (da ? 1u : 0u) | (db ? 2u : 0u);
  const __nv_bfloat162 b = __floats2bfloat162_rn(s.x, s.y);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// ---- tiers 2 and 3 ----
namespace exact_conv {

struct FF {  // h + l, |l| well below ulp(h) after normalisation
  float h, l;
};

// error-free transforms (every operation rounds exactly once: no contraction)
__device__ __forceinline__ FF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FF fast_two_sum(float a, float b) {  // needs |a| >= |b| or a == 0
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const FF p = two_prod(a.h, b.h);
  float e = __fmaf_rn(a.h, b.l, p.l);
  e = __fmaf_rn(a.l, b.h, e);
  return fast_two_sum(p.h, e);
}

// 2^(j/32), j = 0 .. 31, as hi = the nearest fp32 and lo = the nearest fp32
// to the remainder (Tang's table-driven exponential).
static __device__ __constant__ float kExp2Hi[32] = {
    0x1.000000p+0f, 0x1.059b0ep+0f, 0x1.0b5586p+0f, 0x1.11301ep+0f, 0x1.172b84p+0f, 0x1.1d4874p+0f,
    0x1.2387a6p+0f, 0x1.29e9e0p+0f, 0x1.306fe0p+0f, 0x1.371a74p+0f, 0x1.3dea64p+0f, 0x1.44e086p+0f,
    0x1.4bfdaep+0f, 0x1.5342b6p+0f, 0x1.5ab07ep+0f, 0x1.6247ecp+0f, 0x1.6a09e6p+0f, 0x1.71f75ep+0f,
    0x1.7a1148p+0f, 0x1.82589ap+0f, 0x1.8ace54p+0f, 0x1.93737cp+0f, 0x1.9c4918p+0f, 0x1.a5503cp+0f,
    0x1.ae89fap+0f, 0x1.b7f770p+0f, 0x1.c199bep+0f, 0x1.cb720ep+0f, 0x1.d5818ep+0f, 0x1.dfc974p+0f,
    0x1.ea4afap+0f, 0x1.f50766p+0f};
static __device__ __constant__ float kExp2Lo[32] = {
    0.0f,             -0x1.9d4f52p-25f, 0x1.9f3122p-25f,  -0x1.fdb496p-25f, -0x1.c15742p-27f, -0x1.d2e8cap-25f,
    0x1.ceac48p-25f,  -0x1.5c0424p-25f, 0x1.4636e2p-25f,  -0x1.18aac6p-25f, 0x1.824684p-25f,  0x1.8624b4p-30f,
    -0x1.593abcp-25f, -0x1.2c5610p-25f, -0x1.5bd5ecp-27f, -0x1.f8b550p-25f, 0x1.9fcef4p-26f,  0x1.1d8beep-25f,
    -0x1.829fd0p-25f, -0x1.accc7cp-26f, 0x1.15506ep-27f,  -0x1.e64744p-25f, 0x1.51f848p-27f,  -0x1.b83b54p-25f,
    -0x1.a94b14p-26f, -0x1.a09438p-25f, -0x1.3d56b2p-27f, -0x1.8837ccp-27f, -0x1.822dbcp-27f, -0x1.908c94p-25f,
    0x1.52486cp-27f,  -0x1.246eb0p-26f};

// Tier 2.  Returns the code, or -1 when tier 3 must decide.
//   y = sum_j w_j x_j as a pair (h, l): each product split exactly
//     (two_prod), the high parts summed with two_sum, the seven low parts
//     summed with two_sum and their rounding errors gathered; |y - (h + l)|
//     <= 2^-47 |h| + 2^-61 sum_j |w_j x_j| (+ 2^-145 for subnormal products).
//   e^x, x = -|y| >= -87 (|y| > 87 goes to tier 3): n = rint(32 x / ln2), r = x - n ln2/32 with
//     ln2/32 = C1 + C2 + C3 (C1 has 12 significant bits, so n C1 is exact for
//     |n| < 4096), |r| <= ln2/64; e^r = 1 + r + r^2/2 + r^3 (1/6 + r/24 +
//     r^2/120) with the first three terms as pairs (truncation < 2^-48);
//     e^x = z' 2^m, z' = e^r 2^((n mod 32)/32), m = floor(n/32).
//   s = y / (1 + z) (y >= 0), or y z / (1 + z) = 2^m (y z' / (1 + z)) (y < 0),
//     z = e^-|y|, as a pair: q1 = RN(num / d), q2 from the exact residual
//     num - q1 d.  For y < 0 the rounding is decided on the unscaled quotient
//     and the code rescaled by 2^m (|s| >= 87 e^-87 > 2^-126: a normal bf16,
//     where rounding commutes with the power-of-two scaling).
//   The code is the rounding of s.h + s.l, decided when the pair lies farther
//   from the bf16 midpoint than 2^-36 |s| plus the effect of the conv error.
static __device__ __noinline__ int conv_code_ff(float w0, float w1, float w2, float w3, float x0, float x1, float x2,
                                                float x3) {
  const FF p0 = two_prod(w0, x0), p1 = two_prod(w1, x1), p2 = two_prod(w2, x2), p3 = two_prod(w3, x3);
  const FF a = two_sum(p0.h, p1.h), b = two_sum(p2.h, p3.h), c = two_sum(a.h, b.h);
  FF t = two_sum(p0.l, p1.l);
  float err = t.l;
  t = two_sum(t.h, p2.l);
  err = __fadd_rn(err, t.l);
  t = two_sum(t.h, p3.l);
  err = __fadd_rn(err, t.l);
  t = two_sum(t.h, a.l);
  err = __fadd_rn(err, t.l);
  t = two_sum(t.h, b.l);
  err = __fadd_rn(err, t.l);
  t = two_sum(t.h, c.l);
  err = __fadd_rn(err, t.l);
  FF y = two_sum(c.h, t.h);
  y = two_sum(y.h, __fadd_rn(y.l, err));
  const float mag = fabsf(p0.h) + fabsf(p1.h) + fabsf(p2.h) + fabsf(p3.h);
  const float dy = __fmaf_rn(0x1p-46f, fabsf(y.h), __fmaf_rn(0x1p-60f, mag, 0x1p-144f));
  if (y.h == 0.0f) return mag == 0.0f ? 0 : -1;  // an exactly zero sum: SiLU = +0
  if (!(fabsf(y.h) <= 87.0f)) return -1;  // e^-|y| (and its scale 2^m) must stay normal fp32
  const bool neg = y.h < 0.0f;
  const FF x = neg ? y : FF{-y.h, -y.l};  // -|y|
  // z' and m
  constexpr float kShifter = 0x1.8p+23f;
  constexpr float k32Log2e = 0x1.715476p+5f;
  constexpr float kC1 = 0x1.62ep-6f, kC2 = 0x1.0bfbe8p-20f, kC3 = 0x1.cf79acp-45f;
  const float tt = __fmaf_rn(x.h, k32Log2e, kShifter);
  const float nf = __fsub_rn(tt, kShifter);
  const int n = __float_as_int(tt) - __float_as_int(kShifter);
  const float r1 = __fmaf_rn(-nf, kC1, x.h);  // exact: n C1 lies within a factor 2 of x.h
  const FF pc2 = two_prod(-nf, kC2);
  FF r = two_sum(r1, pc2.h);
  r = two_sum(r.h, __fadd_rn(r.l, __fadd_rn(pc2.l, __fmaf_rn(-nf, kC3, x.l))));
  const FF sq = two_prod(r.h, r.h);
  const float sql = __fmaf_rn(__fmul_rn(2.0f, r.h), r.l, sq.l);
  const float poly = __fmaf_rn(__fmaf_rn(r.h, 0x1.111112p-7f, 0x1.555556p-5f), r.h, 0x1.555556p-3f);
  const float t3 = __fmul_rn(__fmul_rn(sq.h, r.h), poly);
  const FF e1 = fast_two_sum(1.0f, r.h);
  const FF e2 = two_sum(e1.h, __fmul_rn(0.5f, sq.h));
  const float el = __fadd_rn(__fadd_rn(e1.l, e2.l), __fadd_rn(r.l, __fmaf_rn(0.5f, sql, t3)));
  const FF er = fast_two_sum(e2.h, el);
  const int j = n & 31;
  const int m = n >> 5;  // n >= -4020: m >= -126
  const FF zp = ff_mul(er, FF{kExp2Hi[j], kExp2Lo[j]});
  const float scale = __int_as_float((m + 127) << 23);
  // d = 1 + z (z below 2^-24 only touches the low part)
  FF d = fast_two_sum(1.0f, __fmul_rn(zp.h, scale));
  d.l = __fadd_rn(d.l, __fmul_rn(zp.l, scale));
  const FF num = neg ? ff_mul(y, zp) : y;
  // 1/d.h for d.h in [1, 2]: the hardware approximation and one Newton step;
  // q1 = num.h / d.h to a few ulp, so num.h - q1 d.h is exact (two_prod and
  // a subtraction within a factor 2) and q2 = res rc carries the rest
  float rc;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(d.h));
  rc = __fmaf_rn(rc, __fmaf_rn(-d.h, rc, 1.0f), rc);
  const float q1 = __fmul_rn(num.h, rc);
  const FF pq = two_prod(q1, d.h);
  const float res = __fadd_rn(__fsub_rn(__fsub_rn(num.h, pq.h), pq.l), __fsub_rn(num.l, __fmul_rn(q1, d.l)));
  const FF s = two_sum(q1, __fmul_rn(res, rc));
  if (s.h == 0.0f) return -1;
  // rounding of s.h + s.l to bf16
  const uint32_t sb = __float_as_uint(s.h);
  const float ah = __uint_as_float(sb & 0x7FFFFFFFu);
  const float al = (sb >> 31) ? -s.l : s.l;
  const uint32_t tb = sb & 0x7FFF0000u;
  const float mid = __uint_as_float(tb | 0x8000u);
  const float diff = __fadd_rn(__fsub_rn(ah, mid), al);  // ah - mid is exact
  // the conv error's effect on the decided quotient: slope dy, with
  // |SiLU'| <= 1.1 for y >= 0 and <= sigma + |SiLU| + 2 dy below; for y < 0
  // the quotient is SiLU 2^-m, so its share is (z'/d + |quotient| + 2 dy 2^-m) dy
  const float slope = neg ? __fmul_rn(zp.h, rc) * 1.001f + ah + 2.0f * __fmul_rn(dy, __int_as_float((127 - m) << 23))
                          : 1.1f;
  const float e = __fmaf_rn(0x1p-36f, ah, __fmaf_rn(__fmul_rn(slope, 1.001f), dy, 0x1p-140f));
  if (!(fabsf(diff) > e)) return -1;
  uint32_t code = (tb >> 16) + (diff > 0.0f ? 1u : 0u);  // magnitude bits of the unscaled code
  if (neg) code += static_cast<uint32_t>(m) << 7;        // times 2^m: exponent field of bf16 (m <= 0)
  return static_cast<int>(code | ((sb >> 16) & 0x8000u));
}

// Tier 3: the definition in fp64.  Every product of a bf16 input and a bf16
// or fp32 weight is exact in double; the sum runs in tap order from +0; the
// result is rounded once to bf16 (nearest, subnormal quantum 2^-133).  For
// y > 0, SiLU(y) lies strictly below y; beyond y of about 37, 1 + e^-y is 1
// in double and s comes out as y itself, so a y exactly halfway between two
// codes takes the one nearer zero (the exact value's side), not the even one.
static __device__ __noinline__ uint32_t conv_code_f64(float w0, float w1, float w2, float w3, float x0, float x1, float x2,
                                               float x3) {
  double y = 0.0;
  y += static_cast<double>(w0) * static_cast<double>(x0);
  y += static_cast<double>(w1) * static_cast<double>(x1);
  y += static_cast<double>(w2) * static_cast<double>(x2);
  y += static_cast<double>(w3) * static_cast<double>(x3);
  const double s = y / (1.0 + exp(-y));
  const double a = fabs(s);
  if (a == 0.0) return signbit(s) ? 0x8000u : 0u;
  int e2;
  (void)frexp(a, &e2);                                   // a = f 2^e2, f in [1/2, 1)
  const double q = ldexp(1.0, max(e2 - 8, -133));       // bf16 quantum at a
  const double sc = a / q;                               // exact (a power-of-two scaling)
  const double k = (y > 0.0 && s == y && sc - floor(sc) == 0.5) ? floor(sc) : rint(sc);
  const double r = k * q;                                // at most 8 significant bits
  const uint32_t bits = __float_as_uint(static_cast<float>(r)) >> 16;
  return bits | (signbit(s) ? 0x8000u : 0u);
}

// The code of one (channel, token) that tier 1 left doubtful.
static __device__ __noinline__ uint32_t conv_code_exact(float w0, float w1, float w2, float w3, float x0, float x1, float x2,
                                                 float x3) {
  const int c = conv_code_ff(w0, w1, w2, w3, x0, x1, x2, x3);
  return c >= 0 ? static_cast<uint32_t>(c) : conv_code_f64(w0, w1, w2, w3, x0, x1, x2, x3);
}

}  // namespace exact_conv

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
