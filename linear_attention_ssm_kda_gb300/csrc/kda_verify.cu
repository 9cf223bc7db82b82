// kda_verify.cu -- the KDA RecoverSSM speculative verify for sm_103a.
//
// Computes what "vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py"
// (_kda_recoverssm_verify_kernel with _kda_recurrent_step and _kda_gate)
// computes, with the short causal conv of
// "vllm.models.kimi_k3.nvidia.recoverssm.kernels" (CuteRecoverSSMVerify:
// conv fused into the verify, rolled conv state of Q + W - 2 taps) in front.
//
// Math.  The window is applied in closed form rather than step by step.
// With D_t = prod_{j<=t} e^{g_j} (per key channel),
//   P_t = S0 (D_t * k^_t),  R_t = S0 (D_t * q^_t)                (one pass over S0)
//   M_tu = sum_k k^_u D_{u+1..t} k^_t (u < t),  N_tu = sum_k k^_u D_{u+1..t} q^_t (u <= t)
//   c_t = beta_t (v_t - P_t - sum_{u<t} M_tu c_u),   o_t = R_t + sum_{u<=t} N_tu c_u,
// which is the recurrence S <- S diag(e^g), c = beta (v - S k^), S <- S + c k^T,
// o = S q^ expanded: the checkpoint S0 is read once (2n FMAs per element) and
// never written.
//
// Schedule.  One persistent CTA per SM walks the (request, head) items
// blockIdx.x + i * gridDim.x (local index i).  Two producer warps feed it
// through mbarrier rings in shared memory:
//   inputs (1 warp)    reads request metadata 32 items per round trip and
//                      bulk-copies (TMA) each item's small inputs into a
//                      ring: the 16-byte hulls of its activation and gate row
//                      segments (rows may start anywhere), its conv taps,
//                      conv weights and dt_bias;
//   state (1 warp)     streams each live item's 64 KB fp32 state as eight row
//                      chunks into a ring of chunk slots, so the HBM stream
//                      runs ahead of the arithmetic by ~2.5 items;
// and twelve compute warps take each item through three phases:
//   conv   one channel per thread (3K = 384 threads): conv + SiLU (bf16,
//          rounded from the exact value) of the window and the key record;
//          the v-channel threads also evaluate the gates and the gate
//          record; the rolled conv taps are written into the shared-memory
//          copy of the item's conv state and leave by bulk stores (TMA);
//   gates  one key channel per thread: norms and the closed-form operands
//          X_t, Y_t, M, N (one warp reduce-scatter);
//   gemv   eight warps, each on its own row chunk of the state: P | R, then
//          the corrections and outputs of its rows.
// Every wait is bounded; a timeout sets KDA_DEVERR_TIMEOUT and an abort flag
// that stops the other roles.
#include <cuda_runtime.h>

#include "kda_device.cuh"

namespace kda {

namespace {

constexpr int kConvWidth = 4;
constexpr int kComputeWarps = 12;  // 3K channels of a K = 128 head, one per thread
constexpr int kGemvWarps = 8;      // one state row chunk each
constexpr int kGateWarps = 4;      // one key channel per thread (K = 128)
constexpr int kThreads = 32 * (2 + kComputeWarps);
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kBarCompute = 1;
constexpr int kSmemLimit = 227 * 1024;

constexpr int ru(int x, int a) { return (x + a - 1) / a * a; }

enum : int { kLive = 1, kNull = 2 };

// Inputs warp -> prep, per item.
template <int QMAX>
struct SmallMeta {
  int flags, bos, n, a;
  long long s, r;
  float A, pad;
  float beta[QMAX];
};

template <int KD, int QMAX>
struct Layout {
  static_assert(7 * QMAX + 10 <= 96, "small-input copies per item exceed three per lane");
  static constexpr int RW = KD / 8;           // state rows per gemv warp (one chunk)
  static constexpr int kChunk = RW * KD * 4;  // bytes per state chunk
  static constexpr int kLcMax = QMAX + kConvWidth - 2;
  static constexpr int kSeg = KD * 2 + 16;    // hull of one row segment
  static constexpr int kNumSmall = QMAX <= 4 ? 3 : 2;  // small-input ring
  // small slot
  static constexpr int kAct = ru(int(sizeof(SmallMeta<QMAX>)), 128);  // [QMAX][3] hulls
  static constexpr int kGate = kAct + QMAX * 3 * kSeg;                 // [QMAX] hulls
  static constexpr int kConv = ru(kGate + QMAX * kSeg, 16);            // the head's conv taps
  static constexpr int kW = ru(kConv + 3 * KD * kLcMax * 2, 16);       // [3][KD][W] weights
  static constexpr int kDt = kW + 3 * KD * kConvWidth * 4;             // [KD] dt_bias
  static constexpr int kSmall = ru(kDt + KD * 4, 128);
  // per-item scratch
  static constexpr int kXs = 3 * QMAX * KD * 4;                        // [3][QMAX][KD] q | k | v
  static constexpr int kVec = 2 * QMAX * KD * 4;                       // [2n][KD] X_t | Y_t
  static constexpr int kEg = QMAX * KD * 4;                            // [QMAX][KD] e^g
  static constexpr int kMN = ru(QMAX * QMAX * 4, 16);
  static constexpr int kRedPerWarp = 2 * QMAX * RW;                    // floats
  static constexpr int kPart = ru(2 * QMAX + QMAX * QMAX, 32);         // reduced values per gate warp
  static constexpr int kFixed = kNumSmall * kSmall + kXs + kVec + kEg + kMN + kGemvWarps * kRedPerWarp * 4 +
                                kGateWarps * kPart * 4 + 32 + 2 * kNumSmall * 8;
  static constexpr int kChunkFit = (kSmemLimit - kFixed - 64 * 2 * 8) / kChunk;
  static constexpr int kNumChunk = kChunkFit > 64 ? 64 : kChunkFit;
  // CTA layout
  static constexpr int oChunks = 0;
  static constexpr int oSmall = oChunks + kNumChunk * kChunk;
  static constexpr int oXs = oSmall + kNumSmall * kSmall;
  static constexpr int oVec = oXs + kXs;
  static constexpr int oEg = oVec + kVec;
  static constexpr int oMN = oEg + kEg;
  static constexpr int oRed = oMN + kMN;
  static constexpr int oPart = oRed + kGemvWarps * kRedPerWarp * 4;
  static constexpr int oMisc = oPart + kGateWarps * kPart * 4;  // int[8]: abort, compute ok, chunk failure
  static constexpr int oBars = ru(oMisc + 32, 8);
  static constexpr int kNumBars = 2 * kNumChunk + 2 * kNumSmall;
  static constexpr int kBytes = oBars + kNumBars * 8;
  static_assert(kBytes <= kSmemLimit, "shared memory budget");
  static_assert(kNumChunk >= 2 * kGemvWarps, "at least two items of state in flight");
};

template <int KD, int QMAX>
struct Bars {
  uint64_t *ch_full, *ch_empty, *sm_full, *sm_empty;
  __device__ explicit Bars(unsigned char* smem) {
    using Lay = Layout<KD, QMAX>;
    uint64_t* b = reinterpret_cast<uint64_t*>(smem + Lay::oBars);
    ch_full = b;
    ch_empty = b + Lay::kNumChunk;
    sm_full = b + 2 * Lay::kNumChunk;
    sm_empty = sm_full + Lay::kNumSmall;
  }
};

// Acquire a barrier phase another lane or thread has already seen complete.
__device__ __forceinline__ void mbar_acquire_seen(uint64_t* bar, uint32_t parity) {
  for (int i = 0; i < 1 << 20 && !mbar_try_wait(bar, parity); ++i) {
  }
}

__device__ __forceinline__ long long shfl_ll(long long v, int src) {
  return static_cast<long long>(__shfl_sync(0xffffffffu, static_cast<unsigned long long>(v), src));
}

// Warp-wide bounded wait by lane 0; every lane then holds the acquire.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane, const volatile int* abort_flag) {
  bool ok = true;
  if (lane == 0) ok = mbar_wait_or_abort(bar, parity, abort_flag);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok && lane != 0) mbar_acquire_seen(bar, parity);
  return ok;
}

// Number of local items of this CTA.
__device__ __forceinline__ int local_items(int items) {
  const int base = static_cast<int>(blockIdx.x);
  return base < items ? (items - base + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) : 0;
}

// Per-item request metadata, decoded by one lane (both producer warps decode
// identically; only the inputs warp reports device errors).
template <int QMAX>
struct ItemMeta {
  int flags, h, bos, n, a;
  long long s, r;
};

template <int QMAX>
__device__ __forceinline__ ItemMeta<QMAX> decode_item(const VerifyParams& p, int it, bool valid, bool report_errors) {
  ItemMeta<QMAX> m{0, 0, 0, 0, 1, 0, 0};
  if (!valid) return m;
  const int b = it / p.H;
  m.h = it - b * p.H;
  m.bos = p.qsl[b];
  const int len = p.qsl[b + 1] - m.bos;
  m.s = p.state_indices[b];
  m.r = p.record_indices ? static_cast<long long>(p.record_indices[b]) : m.s;
  m.a = p.num_accepted_prev ? min(max(p.num_accepted_prev[b], 1), p.Q) : 1;
  m.n = min(max(len, 0), p.Q);
  if (len < 0 || (m.n > 0 && (m.bos < 0 || m.bos + m.n > p.T))) {
    if (report_errors) report(p.workspace, KDA_DEVERR_TOKEN_RANGE, it);
  } else if (m.n > 0) {
    if (m.s <= p.null_block_id) {
      m.flags = kNull;
    } else if (m.s < 0 || m.s >= p.num_slots) {
      if (report_errors) report(p.workspace, KDA_DEVERR_SLOT_RANGE, it);
    } else if (m.r < 0 || m.r >= p.num_record_rows) {
      if (report_errors) report(p.workspace, KDA_DEVERR_ROW_RANGE, it);
    } else {
      m.flags = kLive;
    }
  }
  return m;
}

// Byte offset of a row segment inside its 16-byte-aligned hull.
__device__ __forceinline__ int hull_offset(const void* src) {
  return static_cast<int>(reinterpret_cast<uintptr_t>(src) & 15);
}

// The q-th bulk copy of a live item's small inputs: source, shared-memory
// destination and size (the 16-byte hull of the region).  Copies are, in
// order: 3n activation row segments (token t, group g), n gate row segments,
// the head's conv taps (3 blocks dim-first, 3 (Q+W-2) rows seq-first), three
// conv-weight blocks and dt_bias.  Returns false past the last copy.
template <int KD, int QMAX>
__device__ __forceinline__ bool small_copy(const VerifyParams& p, int q, int n, int bos, long long s, int h,
                                           unsigned char* sl, const void** src, void** dst, uint32_t* bytes) {
  using Lay = Layout<KD, QMAX>;
  const long long HK = static_cast<long long>(p.H) * KD;
  const int Lc = p.Q + kConvWidth - 2;
  const unsigned char* ptr;
  int len;
  if (q < 3 * n) {
    const int t = q / 3, g = q - 3 * (q / 3);
    ptr = reinterpret_cast<const unsigned char*>(p.mixed_qkv + static_cast<long long>(bos + t) * p.qkv_stride +
                                                 g * HK + static_cast<long long>(h) * KD);
    *dst = sl + Lay::kAct + q * Lay::kSeg;
    len = KD * 2;
  } else if (q < 4 * n) {
    const int t = q - 3 * n;
    ptr = reinterpret_cast<const unsigned char*>(p.raw_gate + static_cast<long long>(bos + t) * p.gate_stride +
                                                 static_cast<long long>(h) * KD);
    *dst = sl + Lay::kGate + t * Lay::kSeg;
    len = KD * 2;
  } else {
    q -= 4 * n;
    const int nconv = p.conv_dim_first ? 3 : 3 * Lc;
    const uint16_t* cs = p.conv_state + s * p.conv_slot_stride;
    if (q < nconv) {
      if (p.conv_dim_first) {
        ptr = reinterpret_cast<const unsigned char*>(cs + (q * HK + static_cast<long long>(h) * KD) * Lc);
        *dst = sl + Lay::kConv + q * KD * Lc * 2;
        len = KD * Lc * 2;
      } else {
        const int j = q / 3, g = q - 3 * (q / 3);
        ptr = reinterpret_cast<const unsigned char*>(cs + j * 3 * HK + g * HK + static_cast<long long>(h) * KD);
        *dst = sl + Lay::kConv + q * KD * 2;
        len = KD * 2;
      }
    } else if (q < nconv + 3) {
      const int g = q - nconv;
      const int wb = p.conv_weight_fp32 ? 4 : 2;
      ptr = static_cast<const unsigned char*>(p.conv_weight) + (g * HK + static_cast<long long>(h) * KD) * kConvWidth * wb;
      *dst = sl + Lay::kW + g * KD * kConvWidth * wb;
      len = KD * kConvWidth * wb;
    } else if (q == nconv + 3) {
      ptr = reinterpret_cast<const unsigned char*>(p.dt_bias + static_cast<long long>(h) * KD);
      *dst = sl + Lay::kDt;
      len = KD * 4;
    } else {
      return false;
    }
  }
  const int off = hull_offset(ptr);
  *src = ptr - off;
  *bytes = static_cast<uint32_t>((off + len + 15) & ~15);
  return true;
}

// ---------------------------------------------------------------- inputs warp

template <int KD, int QMAX>
__device__ void produce_inputs(const VerifyParams& p, unsigned char* smem, int lane, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX>;
  Bars<KD, QMAX> bars(smem);
  const int nloc = local_items(p.B * p.H);
  bool ok = true;
  for (int i0 = 0; i0 < nloc && ok; i0 += 32) {
    // metadata of up to 32 items, one per lane, in two round trips
    const int it = static_cast<int>(blockIdx.x) + (i0 + lane) * static_cast<int>(gridDim.x);
    const ItemMeta<QMAX> im = decode_item<QMAX>(p, it, i0 + lane < nloc, true);
    const float A = (i0 + lane < nloc) ? expf(p.A_log[im.h]) : 0.0f;
    float beta[QMAX];
#pragma unroll
    for (int t = 0; t < QMAX; ++t)
      beta[t] = (im.flags == kLive && t < im.n)
                    ? sigmoid_fast(bf16_to_f32(p.raw_beta[static_cast<long long>(im.bos + t) * p.beta_stride + im.h]))
                    : 0.0f;
    const int count = min(32, nloc - i0);
    for (int j = 0; j < count && ok; ++j) {
      const int i = i0 + j;
      SmallMeta<QMAX> mj;
      mj.flags = __shfl_sync(0xffffffffu, im.flags, j);
      mj.bos = __shfl_sync(0xffffffffu, im.bos, j);
      mj.n = __shfl_sync(0xffffffffu, im.n, j);
      mj.a = __shfl_sync(0xffffffffu, im.a, j);
      mj.s = shfl_ll(im.s, j);
      mj.r = shfl_ll(im.r, j);
      mj.A = __shfl_sync(0xffffffffu, A, j);
      mj.pad = 0.0f;
#pragma unroll
      for (int t = 0; t < QMAX; ++t) mj.beta[t] = __shfl_sync(0xffffffffu, beta[t], j);
      const int jh = __shfl_sync(0xffffffffu, im.h, j);
      const int slot = i % Lay::kNumSmall;
      ok = warp_wait(&bars.sm_empty[slot], ((i / Lay::kNumSmall) & 1) ^ 1, lane, abort_flag);
      if (!ok) break;
      unsigned char* sl = smem + Lay::oSmall + slot * Lay::kSmall;
      if (lane == 0) *reinterpret_cast<SmallMeta<QMAX>*>(sl) = mj;
      if (mj.flags & kLive) {
        // at most 7 QMAX + 10 copies, three per lane; the barrier expects every
        // byte before the first copy can land
        const void* src[3];
        void* dst[3];
        uint32_t bytes[3];
        uint32_t mine = 0;
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          if (!small_copy<KD, QMAX>(p, lane + 32 * c, mj.n, mj.bos, mj.s, jh, sl, &src[c], &dst[c], &bytes[c]))
            bytes[c] = 0;
          mine += bytes[c];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
        if (lane == 0) mbar_arrive_expect_tx(&bars.sm_full[slot], mine);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 3; ++c)
          if (bytes[c]) bulk_g2s(dst[c], src[c], bytes[c], &bars.sm_full[slot]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.sm_full[slot]);
      }
    }
  }
  if (!ok && lane == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

// ---------------------------------------------------------------- state warp

template <int KD, int QMAX>
__device__ void produce_state(const VerifyParams& p, unsigned char* smem, int lane, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX>;
  Bars<KD, QMAX> bars(smem);
  const int nloc = local_items(p.B * p.H);
  uint32_t ch_cnt = 0;
  bool ok = true;
  for (int i0 = 0; i0 < nloc && ok; i0 += 32) {
    const int it = static_cast<int>(blockIdx.x) + (i0 + lane) * static_cast<int>(gridDim.x);
    const ItemMeta<QMAX> im = decode_item<QMAX>(p, it, i0 + lane < nloc, false);
    const int count = min(32, nloc - i0);
    for (int j = 0; j < count && ok; ++j) {
      if (!(__shfl_sync(0xffffffffu, im.flags, j) & kLive)) continue;
      const int jh = __shfl_sync(0xffffffffu, im.h, j);
      const long long js = shfl_ll(im.s, j);
      // lane c streams row chunk c into the next free chunk slot
      if (lane < kGemvWarps) {
        const uint32_t cc = ch_cnt + lane;
        const int pos = cc % Lay::kNumChunk;
        ok = mbar_wait_or_abort(&bars.ch_empty[pos], ((cc / Lay::kNumChunk) & 1) ^ 1, abort_flag);
        if (ok) {
          const float* src = p.state + js * p.state_slot_stride + static_cast<long long>(jh) * KD * KD;
          mbar_arrive_expect_tx(&bars.ch_full[pos], Lay::kChunk);
          bulk_g2s(smem + Lay::oChunks + pos * Lay::kChunk, src + lane * Lay::RW * KD, Lay::kChunk,
                   &bars.ch_full[pos]);
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      ch_cnt += kGemvWarps;
    }
  }
  if (!ok && lane == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

// ---------------------------------------------------------------- compute

// One reduce-scatter stage over the lanes `mask` apart: each lane keeps the
// half of its W values selected by its lane bit and adds the partner's copy.
template <int W>
__device__ __forceinline__ void reduce_scatter_stage(float* acc, int mask, bool upper) {
#pragma unroll
  for (int i = 0; i < W / 2; ++i) {
    const float send = upper ? acc[i] : acc[i + W / 2];
    const float keep = upper ? acc[i + W / 2] : acc[i];
    acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
  }
}

// Dot products of a warp's RW state rows with NCG operand vectors.  Lane =
// 8 rs + kq covers rows 4i + rs (i < RW/4) and the float4 key chunks
// 4kq + 32j (j < KD/32): a warp-wide LDS.128 reads 4 rows x 128 contiguous
// bytes, and the 8 lanes of a row share a broadcast operand load.  The 8
// partial sums of a row meet in a three-stage reduce-scatter.
template <int KD, int NCG>
__device__ __forceinline__ void gemv_chunk(const float* __restrict__ st, const float* __restrict__ vec,
                                           float* __restrict__ red, int lane) {
  constexpr int RW = KD / 8;
  constexpr int R = RW / 4;
  constexpr int J = KD / 32;
  constexpr int NV = R * NCG;
  constexpr int NVP = (NV + 7) / 8 * 8;
  const int kq = lane & 7;
  const int rs = lane >> 3;
  float acc[NVP];
#pragma unroll
  for (int i = 0; i < NVP; ++i) acc[i] = 0.0f;
#pragma unroll 2
  for (int j = 0; j < J; ++j) {
    const int kk = 4 * kq + 32 * j;
    float4 vv[NCG];
#pragma unroll
    for (int c = 0; c < NCG; ++c) vv[c] = *reinterpret_cast<const float4*>(vec + c * KD + kk);
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const float4 sv = *reinterpret_cast<const float4*>(st + (4 * i + rs) * KD + kk);
#pragma unroll
      for (int c = 0; c < NCG; ++c) {
        float x = acc[i * NCG + c];
        x = fmaf(sv.x, vv[c].x, x);
        x = fmaf(sv.y, vv[c].y, x);
        x = fmaf(sv.z, vv[c].z, x);
        x = fmaf(sv.w, vv[c].w, x);
        acc[i * NCG + c] = x;
      }
    }
  }
  reduce_scatter_stage<NVP>(acc, 4, (kq & 4) != 0);
  reduce_scatter_stage<NVP / 2>(acc, 2, (kq & 2) != 0);
  reduce_scatter_stage<NVP / 4>(acc, 1, (kq & 1) != 0);
#pragma unroll
  for (int i = 0; i < NVP / 8; ++i) {
    const int v = (NVP / 8) * kq + i;
    if (v < NV) {
      const int row = v / NCG;
      const int c = v - row * NCG;
      red[c * RW + 4 * row + rs] = acc[i];
    }
  }
}

template <int KD, int QMAX>
__device__ void compute(const VerifyParams& p, unsigned char* smem, int ct, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX>;
  constexpr int RW = Lay::RW;
  constexpr int NREDP = Lay::kPart;  // |q_t|^2, |k_t|^2, raw M / N grid, padded to 32
  constexpr int PER = NREDP / 32;
  Bars<KD, QMAX> bars(smem);
  volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::oMisc);
  float* xs = reinterpret_cast<float*>(smem + Lay::oXs);    // [3][QMAX][KD]
  float* vec = reinterpret_cast<float*>(smem + Lay::oVec);  // [2n][KD]
  float* mn = reinterpret_cast<float*>(smem + Lay::oMN);    // [QMAX][QMAX]
  float* part = reinterpret_cast<float*>(smem + Lay::oPart);
  const int warp = ct >> 5;
  const int lane = ct & 31;
  float* red = reinterpret_cast<float*>(smem + Lay::oRed) + warp * Lay::kRedPerWarp;
  const int nloc = local_items(p.B * p.H);
  const long long HK = static_cast<long long>(p.H) * KD;
  const int Lc = p.Q + kConvWidth - 2;
  const uint32_t qkv_lo = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.mixed_qkv));
  const uint32_t gate_lo = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.raw_gate));
  const uint32_t hk2 = static_cast<uint32_t>(HK) * 2u;
  uint32_t live = 0;
  bool alive = true;
  for (int i = 0; i < nloc; ++i) {
    const int it = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int h = it - (it / p.H) * p.H;
    const int slot = i % Lay::kNumSmall;
    const uint32_t ph = (i / Lay::kNumSmall) & 1;
    const unsigned char* sl = smem + Lay::oSmall + slot * Lay::kSmall;
    if (ct == 0) misc[1] = mbar_wait_or_abort(&bars.sm_full[slot], ph, abort_flag) ? 1 : 0;
    named_barrier(kBarCompute, kComputeThreads);
    if (!misc[1]) {
      alive = false;
      break;
    }
    if (ct != 0) mbar_acquire_seen(&bars.sm_full[slot], ph);
    const SmallMeta<QMAX> m = *reinterpret_cast<const SmallMeta<QMAX>*>(sl);
    const int n = m.n;
    const int bos = m.bos;
    const uint32_t hoff = static_cast<uint32_t>(h) * KD * 2u;
    if (!(m.flags & kLive)) {
      if (m.flags & kNull) {  // null slot: zero outputs, nothing else
        for (int e = ct; e < n * KD; e += kComputeThreads) {
          const int t = e / KD;
          p.out[static_cast<long long>(bos + t) * p.out_stride + static_cast<long long>(h) * KD + (e - t * KD)] = 0;
        }
      }
      named_barrier(kBarCompute, kComputeThreads);
      if (ct == 0) mbar_arrive(&bars.sm_empty[slot]);
      continue;
    }
    uint16_t* kg = p.key_gate + m.r * p.kg_stride + static_cast<long long>(h) * p.Q * 2 * KD;

    // ---- conv: thread ct owns channel k of group g (q | k | v) ----
    if (ct < 3 * KD) {
      const int g = ct / KD;
      const int k = ct - g * KD;
      uint16_t* conv = reinterpret_cast<uint16_t*>(const_cast<unsigned char*>(sl) + Lay::kConv);
      float w[kConvWidth];
      if (p.conv_weight_fp32) {
        const float4 wv = reinterpret_cast<const float4*>(sl + Lay::kW)[g * KD + k];
        w[0] = wv.x; w[1] = wv.y; w[2] = wv.z; w[3] = wv.w;
      } else {
        const uint2 wv = reinterpret_cast<const uint2*>(sl + Lay::kW)[g * KD + k];
        w[0] = bf16_to_f32(wv.x & 0xffff); w[1] = bf16_to_f32(wv.x >> 16);
        w[2] = bf16_to_f32(wv.y & 0xffff); w[3] = bf16_to_f32(wv.y >> 16);
      }
      uint16_t seq[kConvWidth - 1 + QMAX + 1];
#pragma unroll
      for (int j = 0; j < kConvWidth - 1; ++j)
        seq[j] = p.conv_dim_first ? conv[(g * KD + k) * Lc + m.a - 1 + j] : conv[((m.a - 1 + j) * 3 + g) * KD + k];
#pragma unroll
      for (int t = 0; t < QMAX + 1; ++t) {
        seq[kConvWidth - 1 + t] = 0;
        if (t < n) {
          const uint32_t off =
              (qkv_lo + static_cast<uint32_t>(bos + t) * static_cast<uint32_t>(p.qkv_stride) * 2u + g * hk2 + hoff) &
              15u;
          seq[kConvWidth - 1 + t] =
              *reinterpret_cast<const uint16_t*>(sl + Lay::kAct + (t * 3 + g) * Lay::kSeg + off + 2 * k);
        }
      }
      float* xg = xs + g * QMAX * KD;
#pragma unroll
      for (int t = 0; t < QMAX; t += 2) {  // tokens in pairs: two independent chains
        if (t < n) {
          const float x0[kConvWidth] = {bf16_to_f32(seq[t]), bf16_to_f32(seq[t + 1]), bf16_to_f32(seq[t + 2]),
                                        bf16_to_f32(seq[t + 3])};
          const float x1[kConvWidth] = {bf16_to_f32(seq[t + 1]), bf16_to_f32(seq[t + 2]), bf16_to_f32(seq[t + 3]),
                                        bf16_to_f32(seq[t + 4])};
          const uint16_t y0 = conv_silu_bf16(w, x0);
          const uint16_t y1 = conv_silu_bf16(w, x1);
          xg[t * KD + k] = bf16_to_f32(y0);
          if (g == 1) kg[t * 2 * KD + k] = y0;  // key record: the bf16 conv output
          if (t + 1 < n && t + 1 < QMAX) {
            xg[(t + 1) * KD + k] = bf16_to_f32(y1);
            if (g == 1) kg[(t + 1) * 2 * KD + k] = y1;
          }
        }
      }
      // rolled conv state, into the slot's copy: taps 0 .. W-3+n <- seq[1 .. W-2+n]
#pragma unroll
      for (int j = 0; j < kConvWidth - 2 + QMAX; ++j) {
        if (j < kConvWidth - 2 + n) {
          if (p.conv_dim_first)
            conv[(g * KD + k) * Lc + j] = seq[j + 1];
          else
            conv[(j * 3 + g) * KD + k] = seq[j + 1];
        }
      }
      if (g == 2) {  // gates and the gate record, on the v-channel threads
        const float dtb = reinterpret_cast<const float*>(sl + Lay::kDt)[k];
        float* egs = reinterpret_cast<float*>(smem + Lay::oEg);
#pragma unroll
        for (int t = 0; t < QMAX; ++t) {
          if (t < n) {
            const uint32_t goff =
                (gate_lo + static_cast<uint32_t>(bos + t) * static_cast<uint32_t>(p.gate_stride) * 2u + hoff) & 15u;
            const uint16_t rg = *reinterpret_cast<const uint16_t*>(sl + Lay::kGate + t * Lay::kSeg + goff + 2 * k);
            kg[t * 2 * KD + KD + k] = rg;  // gate record: bit copy
            egs[t * KD + k] = kda_decay_fast(bf16_to_f32(rg), dtb, m.A, p.lower_bound_gate, p.lower_bound);
          }
        }
      }
    }
    fence_async_shared();
    named_barrier(kBarCompute, kComputeThreads);
    if (ct == 0) {  // the rolled conv state leaves by bulk stores from the slot
      uint16_t* cs = p.conv_state + m.s * p.conv_slot_stride;
      if (p.conv_dim_first) {
#pragma unroll
        for (int g = 0; g < 3; ++g)
          bulk_s2g(cs + (g * HK + static_cast<long long>(h) * KD) * Lc, sl + Lay::kConv + g * KD * Lc * 2, KD * Lc * 2);
      } else {
        for (int j = 0; j < kConvWidth - 2 + n; ++j)
#pragma unroll
          for (int g = 0; g < 3; ++g)
            bulk_s2g(cs + j * 3 * HK + g * HK + static_cast<long long>(h) * KD, sl + Lay::kConv + (j * 3 + g) * KD * 2,
                     KD * 2);
      }
      bulk_commit();
    }

    // ---- gates, gate record, norms and closed-form scalars: key channel k = ct ----
    float qv[QMAX], kv[QMAX], eg[QMAX];
    if (ct < KD) {
      const int k = ct;
      const float* egs = reinterpret_cast<const float*>(smem + Lay::oEg);
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        qv[t] = kv[t] = eg[t] = 0.0f;
        if (t < n) {
          qv[t] = xs[t * KD + k];
          kv[t] = xs[QMAX * KD + t * KD + k];
          eg[t] = egs[t * KD + k];
        }
      }
      // vals: [t] |q_t|^2, [QMAX + t] |k_t|^2, [2QMAX + t QMAX + u] k_u D_{u+1..t} k_t (u < t),
      //       [2QMAX + u QMAX + t] k_u D_{u+1..t} q_t (u <= t); zero past n.
      float vals[NREDP];
#pragma unroll
      for (int v = 0; v < NREDP; ++v) vals[v] = 0.0f;
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        vals[t] = qv[t] * qv[t];
        vals[QMAX + t] = kv[t] * kv[t];
      }
#pragma unroll
      for (int u = 0; u < QMAX; ++u) {
        float wu = kv[u];
#pragma unroll
        for (int t = u; t < QMAX; ++t) {
          if (t > u) {
            wu *= eg[t];
            vals[2 * QMAX + t * QMAX + u] = wu * kv[t];
          }
          vals[2 * QMAX + u * QMAX + t] = wu * qv[t];
        }
      }
      reduce_scatter_stage<NREDP>(vals, 16, (lane & 16) != 0);
      reduce_scatter_stage<NREDP / 2>(vals, 8, (lane & 8) != 0);
      reduce_scatter_stage<NREDP / 4>(vals, 4, (lane & 4) != 0);
      reduce_scatter_stage<NREDP / 8>(vals, 2, (lane & 2) != 0);
      reduce_scatter_stage<NREDP / 16>(vals, 1, (lane & 1) != 0);
#pragma unroll
      for (int v = 0; v < PER; ++v) part[warp * NREDP + lane * PER + v] = vals[v];
    }
    named_barrier(kBarCompute, kComputeThreads);
    if (ct < KD) {
      float rq[QMAX], rk[QMAX];
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        float qq = 0.0f, kk = 0.0f;
#pragma unroll
        for (int w = 0; w < KD / 32; ++w) {
          qq += part[w * NREDP + t];
          kk += part[w * NREDP + QMAX + t];
        }
        rq[t] = rsqrtf(qq + 1e-6f) * p.k_scale;  // q^ = q rsqrt(|q|^2 + eps) K^-1/2
        rk[t] = rsqrtf(kk + 1e-6f);              // k^ = k rsqrt(|k|^2 + eps)
      }
      float D = 1.0f;
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        if (t < n) {
          D *= eg[t];
          vec[t * KD + ct] = D * (kv[t] * rk[t]);        // X_t = D_t k^_t
          vec[(n + t) * KD + ct] = D * (qv[t] * rq[t]);  // Y_t = D_t q^_t
        }
      }
      if (ct < QMAX * QMAX) {
        const int i2 = ct / QMAX, j2 = ct - (ct / QMAX) * QMAX;
        float raw = 0.0f;
#pragma unroll
        for (int w = 0; w < KD / 32; ++w) raw += part[w * NREDP + 2 * QMAX + ct];
        // i2 > j2: M = raw rk_j rk_i (t = i2, u = j2); i2 <= j2: N = raw rk_i rq_j (u = i2, t = j2)
        float ri = 0.0f, rj = 0.0f;
#pragma unroll
        for (int t = 0; t < QMAX; ++t) {
          if (t == i2) ri = rk[t];
          if (t == j2) rj = (i2 > j2) ? rk[t] : rq[t];
        }
        mn[ct] = raw * ri * rj;
      }
    }
    named_barrier(kBarCompute, kComputeThreads);
    if (ct == 0) {  // the small inputs are consumed once the bulk stores have read them
      bulk_wait_read();
      mbar_arrive(&bars.sm_empty[slot]);
    }

    // ---- gemv on the warp's row chunk, then its rows' corrections and outputs ----
    if (warp < kGemvWarps) {
      const uint32_t pc = live * kGemvWarps + warp;
      const int pos = pc % Lay::kNumChunk;
      const uint32_t cph = (pc / Lay::kNumChunk) & 1;
      if (warp_wait(&bars.ch_full[pos], cph, lane, abort_flag)) {
        const float* st = reinterpret_cast<const float*>(smem + Lay::oChunks + pos * Lay::kChunk);
        for (int cg = 0; cg < 2 * n; cg += 8) {
          switch (min(8, 2 * n - cg)) {
            case 2: gemv_chunk<KD, 2>(st, vec + cg * KD, red + cg * RW, lane); break;
            case 4: gemv_chunk<KD, 4>(st, vec + cg * KD, red + cg * RW, lane); break;
            case 6: gemv_chunk<KD, 6>(st, vec + cg * KD, red + cg * RW, lane); break;
            default: gemv_chunk<KD, 8>(st, vec + cg * KD, red + cg * RW, lane); break;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.ch_empty[pos]);
        if (lane < RW) {
          const int row = warp * RW + lane;
          float* corr = p.corr + m.r * p.corr_stride + static_cast<long long>(h) * p.Q * KD;
          const float* xv = xs + 2 * QMAX * KD;
          float cv[QMAX];
#pragma unroll
          for (int t = 0; t < QMAX; ++t) {
            if (t < n) {
              float x = xv[t * KD + row] - red[t * RW + lane];
#pragma unroll
              for (int u = 0; u < t; ++u) x = fmaf(-mn[t * QMAX + u], cv[u], x);
              const float c = x * m.beta[t];
              cv[t] = c;
              float o = red[(n + t) * RW + lane];
#pragma unroll
              for (int u = 0; u <= t; ++u) o = fmaf(mn[u * QMAX + t], cv[u], o);
              corr[t * KD + row] = c;
              p.out[static_cast<long long>(bos + t) * p.out_stride + static_cast<long long>(h) * KD + row] =
                  f32_to_bf16(o);
            }
          }
        }
      } else if (lane == 0) {
        misc[2] = 1;
      }
    }
    ++live;
    named_barrier(kBarCompute, kComputeThreads);
    if (misc[2]) {
      alive = false;
      break;
    }
  }
  if (ct == 0) bulk_wait_all();
  if (!alive && ct == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

template <int KD, int QMAX>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const VerifyParams p) {
  using Lay = Layout<KD, QMAX>;
  extern __shared__ __align__(1024) unsigned char smem[];
  volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::oMisc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  if (tid == 0) {
    Bars<KD, QMAX> bars(smem);
    for (int i = 0; i < Lay::kNumChunk; ++i) {
      mbar_init(&bars.ch_full[i], 1);
      mbar_init(&bars.ch_empty[i], 1);
    }
    for (int i = 0; i < Lay::kNumSmall; ++i) {
      mbar_init(&bars.sm_full[i], 1);
      mbar_init(&bars.sm_empty[i], 1);
    }
    for (int i = 0; i < 8; ++i) misc[i] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) {
    produce_inputs<KD, QMAX>(p, smem, tid & 31, misc);
  } else if (warp == 1) {
    produce_state<KD, QMAX>(p, smem, tid & 31, misc);
  } else {
    compute<KD, QMAX>(p, smem, tid - 64, misc);
  }
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int KD, int QMAX>
cudaError_t launch(const VerifyParams& p, cudaStream_t stream) {
  constexpr int bytes = Layout<KD, QMAX>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<KD, QMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const int items = p.B * p.H;
  const int grid = items < sm_count() ? items : sm_count();
  verify_kernel<KD, QMAX><<<grid, kThreads, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& p, int K, cudaStream_t stream) {
  if (K == 128) return p.Q <= 4 ? launch<128, 4>(p, stream) : launch<128, 8>(p, stream);
  return p.Q <= 4 ? launch<64, 4>(p, stream) : launch<64, 8>(p, stream);
}

}  // namespace kda
