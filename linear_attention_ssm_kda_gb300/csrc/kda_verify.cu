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
// blockIdx.x, blockIdx.x + gridDim.x, ... with three warp roles linked by
// mbarrier rings in shared memory:
//   producer (1 warp)  reads request metadata 32 items per round trip and
//                      issues bulk copies (TMA): each item's small inputs
//                      (activation and gate rows, conv taps, conv weights,
//                      dt_bias) into a 2-slot ring, and its 64 KB state as
//                      eight row chunks into a chunk ring of ~20 slots, so
//                      ~100 KB of HBM reads per SM stay in flight;
//   prep (4 warps)     conv + SiLU (bf16, rounded from the exact value), the
//                      rolled conv state and key/gate records, norms, gates,
//                      and the closed-form operands, into a 2-slot ring;
//   gemv (8 warps)     each consumes its own row chunk of the state: P | R,
//                      the corrections and outputs of its rows.
// Rows of an activation buffer may start anywhere: the producer copies the
// 16-byte-aligned hull of each row segment and the consumer reads at the
// offset (a 16-byte block never straddles a page, so the hull is mapped).
// Every wait is bounded; a timeout sets KDA_DEVERR_TIMEOUT and an abort flag
// that stops the other roles.
#include <cuda_runtime.h>

#include "kda_device.cuh"

namespace kda {

namespace {

constexpr int kConvWidth = 4;
constexpr int kPrepWarps = 4;
constexpr int kGemvWarps = 8;
constexpr int kThreads = 32 * (1 + kPrepWarps + kGemvWarps);
constexpr int kPrepThreads = 32 * kPrepWarps;
constexpr int kGemvThreads = 32 * kGemvWarps;
constexpr int kBarPrep = 1;
constexpr int kBarGemv = 2;
constexpr int kSmemLimit = 227 * 1024;

constexpr int ru(int x, int a) { return (x + a - 1) / a * a; }

enum : int { kLive = 1, kNull = 2, kEnd = 4 };

// Producer -> prep, per item.
template <int QMAX>
struct SmallMeta {
  int flags, bos, n, a;
  long long s, r;
  float A, pad;
  float beta[QMAX];
  uint8_t act_off[QMAX * 3];  // byte offset of each row segment inside its hull
  uint8_t gate_off[QMAX];
};

// Prep -> gemv, per live item.
template <int QMAX>
struct OpMeta {
  int flags, bos, n, h;
  long long r;
  float beta[QMAX];
};

template <int KD, int QMAX>
struct Layout {
  static constexpr int RW = KD / 8;                 // state rows per gemv warp (one chunk)
  static constexpr int kChunk = RW * KD * 4;        // bytes per state chunk
  static constexpr int kLcMax = QMAX + kConvWidth - 2;
  static constexpr int kSeg = KD * 2 + 16;          // hull of one row segment
  // small slot
  static constexpr int kAct = ru(int(sizeof(SmallMeta<QMAX>)), 128);  // [QMAX][3] hulls
  static constexpr int kGate = kAct + QMAX * 3 * kSeg;                 // [QMAX] hulls
  static constexpr int kConv = ru(kGate + QMAX * kSeg, 16);            // the head's conv taps
  static constexpr int kW = ru(kConv + 3 * KD * kLcMax * 2, 16);       // [3][KD][W] weights
  static constexpr int kDt = kW + 3 * KD * kConvWidth * 4;             // [KD] dt_bias
  static constexpr int kSmall = ru(kDt + KD * 4, 128);
  static constexpr int kNumSmall = 2;
  // operand slot
  static constexpr int kOpMN = ru(int(sizeof(OpMeta<QMAX>)), 16);      // [QMAX][QMAX]
  static constexpr int kOpVec = ru(kOpMN + QMAX * QMAX * 4, 16);       // [2n][KD]: X_t | Y_t
  static constexpr int kOpV = kOpVec + 2 * QMAX * KD * 4;              // [QMAX][KD] v_t
  static constexpr int kOp = ru(kOpV + QMAX * KD * 4, 128);
  static constexpr int kNumOp = 2;
  // scratch
  static constexpr int kRedPerWarp = 2 * QMAX * RW;                    // floats
  static constexpr int kPartPerWarp = 2 * QMAX + QMAX * QMAX;          // floats
  static constexpr int kFixed = kNumSmall * kSmall + kNumOp * kOp + kGemvWarps * kRedPerWarp * 4 +
                                kPrepWarps * kPartPerWarp * 4 + 32 + (2 * kNumSmall + 2 * kNumOp) * 8;
  static constexpr int kChunkFit = (kSmemLimit - kFixed - 64 * 2 * 8) / kChunk;
  static constexpr int kNumChunk = kChunkFit > 64 ? 64 : kChunkFit;
  // CTA layout
  static constexpr int oChunks = 0;
  static constexpr int oSmall = oChunks + kNumChunk * kChunk;
  static constexpr int oOp = oSmall + kNumSmall * kSmall;
  static constexpr int oRed = oOp + kNumOp * kOp;
  static constexpr int oPart = oRed + kGemvWarps * kRedPerWarp * 4;
  // int[8]: abort, prep small-slot ok, gemv op ok, gemv chunk failure, prep op-slot ok
  static constexpr int oMisc = oPart + kPrepWarps * kPartPerWarp * 4;
  static constexpr int oBars = ru(oMisc + 32, 8);
  static constexpr int kNumBars = 2 * kNumChunk + 2 * kNumSmall + 2 * kNumOp;
  static constexpr int kBytes = oBars + kNumBars * 8;
  static_assert(kBytes <= kSmemLimit, "shared memory budget");
  static_assert(kNumChunk >= 2 * kGemvWarps, "at least two items of state in flight");
};

template <int KD, int QMAX>
struct Bars {
  uint64_t *ch_full, *ch_empty, *sm_full, *sm_empty, *op_full, *op_empty;
  __device__ explicit Bars(unsigned char* smem) {
    using Lay = Layout<KD, QMAX>;
    uint64_t* b = reinterpret_cast<uint64_t*>(smem + Lay::oBars);
    ch_full = b;
    ch_empty = b + Lay::kNumChunk;
    sm_full = b + 2 * Lay::kNumChunk;
    sm_empty = sm_full + Lay::kNumSmall;
    op_full = sm_empty + Lay::kNumSmall;
    op_empty = op_full + Lay::kNumOp;
  }
};

// Acquire a barrier phase another thread of the group has already seen complete.
__device__ __forceinline__ void mbar_acquire_seen(uint64_t* bar, uint32_t parity) {
  for (int i = 0; i < 1 << 20 && !mbar_try_wait(bar, parity); ++i) {
  }
}

__device__ __forceinline__ long long shfl_ll(long long v, int src) {
  return static_cast<long long>(__shfl_sync(0xffffffffu, static_cast<unsigned long long>(v), src));
}

// Bulk-copy the 16-byte-aligned hull of `bytes` bytes at `src`; returns the
// offset of src inside the hull and adds the hull size to *total (issue=false
// only measures).
__device__ __forceinline__ int hull_copy(void* dst, const void* src, int bytes, uint64_t* bar, bool issue,
                                         uint32_t* total) {
  const uintptr_t g = reinterpret_cast<uintptr_t>(src);
  const uintptr_t start = g & ~static_cast<uintptr_t>(15);
  const int off = static_cast<int>(g - start);
  const uint32_t size = static_cast<uint32_t>((off + bytes + 15) & ~15);
  if (issue) bulk_g2s(dst, reinterpret_cast<const void*>(start), size, bar);
  *total += size;
  return off;
}

// ---------------------------------------------------------------- producer

template <int KD, int QMAX>
__device__ void issue_small(const VerifyParams& p, unsigned char* sl, SmallMeta<QMAX>* m, int h, uint64_t* bar,
                            bool issue, uint32_t* total) {
  using Lay = Layout<KD, QMAX>;
  const long long HK = static_cast<long long>(p.H) * KD;
  const int Lc = p.Q + kConvWidth - 2;
  for (int t = 0; t < m->n; ++t) {
    const long long row = static_cast<long long>(m->bos + t);
#pragma unroll
    for (int g = 0; g < 3; ++g) {
      const uint16_t* src = p.mixed_qkv + row * p.qkv_stride + g * HK + static_cast<long long>(h) * KD;
      m->act_off[t * 3 + g] =
          static_cast<uint8_t>(hull_copy(sl + Lay::kAct + (t * 3 + g) * Lay::kSeg, src, KD * 2, bar, issue, total));
    }
    const uint16_t* gsrc = p.raw_gate + row * p.gate_stride + static_cast<long long>(h) * KD;
    m->gate_off[t] = static_cast<uint8_t>(hull_copy(sl + Lay::kGate + t * Lay::kSeg, gsrc, KD * 2, bar, issue, total));
  }
  const uint16_t* cs = p.conv_state + m->s * p.conv_slot_stride;
  if (p.conv_dim_first) {
#pragma unroll
    for (int g = 0; g < 3; ++g)
      hull_copy(sl + Lay::kConv + g * KD * Lc * 2, cs + (g * HK + static_cast<long long>(h) * KD) * Lc, KD * Lc * 2,
                bar, issue, total);
  } else {
    for (int j = 0; j < Lc; ++j)
#pragma unroll
      for (int g = 0; g < 3; ++g)
        hull_copy(sl + Lay::kConv + (j * 3 + g) * KD * 2, cs + j * 3 * HK + g * HK + static_cast<long long>(h) * KD,
                  KD * 2, bar, issue, total);
  }
  const int wb = p.conv_weight_fp32 ? 4 : 2;
  const unsigned char* w = static_cast<const unsigned char*>(p.conv_weight);
#pragma unroll
  for (int g = 0; g < 3; ++g)
    hull_copy(sl + Lay::kW + g * KD * kConvWidth * wb, w + (g * HK + static_cast<long long>(h) * KD) * kConvWidth * wb,
              KD * kConvWidth * wb, bar, issue, total);
  hull_copy(sl + Lay::kDt, p.dt_bias + static_cast<long long>(h) * KD, KD * 4, bar, issue, total);
}

template <int KD, int QMAX>
__device__ void produce(const VerifyParams& p, unsigned char* smem, int lane, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX>;
  Bars<KD, QMAX> bars(smem);
  const int items = p.B * p.H;
  uint32_t sm_cnt = 0, ch_cnt = 0;
  bool ok = true;
  for (int base = blockIdx.x; base < items && ok; base += 32 * gridDim.x) {
    // ---- metadata of up to 32 items, one per lane, in two round trips ----
    const int it = base + lane * static_cast<int>(gridDim.x);
    const bool valid = it < items;
    int b = 0, h = 0, bos = 0, len = 0, a = 1;
    long long s = 0, r = 0;
    float A = 0.0f;
    if (valid) {
      b = it / p.H;
      h = it - b * p.H;
      bos = p.qsl[b];
      len = p.qsl[b + 1] - bos;
      s = p.state_indices[b];
      r = p.record_indices ? static_cast<long long>(p.record_indices[b]) : s;
      a = p.num_accepted_prev ? min(max(p.num_accepted_prev[b], 1), p.Q) : 1;
      A = expf(p.A_log[h]);
    }
    const int n = min(max(len, 0), p.Q);
    int flags = 0;
    if (valid) {
      if (len < 0 || (n > 0 && (bos < 0 || bos + n > p.T))) {
        report(p.workspace, KDA_DEVERR_TOKEN_RANGE, it);
      } else if (n > 0) {
        if (s <= p.null_block_id) {
          flags = kNull;
        } else if (s < 0 || s >= p.num_slots) {
          report(p.workspace, KDA_DEVERR_SLOT_RANGE, it);
        } else if (r < 0 || r >= p.num_record_rows) {
          report(p.workspace, KDA_DEVERR_ROW_RANGE, it);
        } else {
          flags = kLive;
        }
      }
    }
    float beta[QMAX];
#pragma unroll
    for (int t = 0; t < QMAX; ++t)
      beta[t] = (flags == kLive && t < n)
                    ? sigmoidf(bf16_to_f32(p.raw_beta[static_cast<long long>(bos + t) * p.beta_stride + h]))
                    : 0.0f;

    // ---- issue the items in order ----
    const int count = min(32, (items - base + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x));
    for (int j = 0; j < count; ++j) {
      const int jf = __shfl_sync(0xffffffffu, flags, j);
      const int jb = __shfl_sync(0xffffffffu, bos, j);
      const int jn = __shfl_sync(0xffffffffu, n, j);
      const int ja = __shfl_sync(0xffffffffu, a, j);
      const int jh = __shfl_sync(0xffffffffu, h, j);
      const long long js = shfl_ll(s, j);
      const long long jr = shfl_ll(r, j);
      const float jA = __shfl_sync(0xffffffffu, A, j);
      float jbeta[QMAX];
#pragma unroll
      for (int t = 0; t < QMAX; ++t) jbeta[t] = __shfl_sync(0xffffffffu, beta[t], j);
      if (lane == 0) {
        const int slot = sm_cnt % Lay::kNumSmall;
        const uint32_t ph = (sm_cnt / Lay::kNumSmall) & 1;
        ok = mbar_wait_or_abort(&bars.sm_empty[slot], ph ^ 1, abort_flag);
        if (ok) {
          unsigned char* sl = smem + Lay::oSmall + slot * Lay::kSmall;
          SmallMeta<QMAX>* m = reinterpret_cast<SmallMeta<QMAX>*>(sl);
          m->flags = jf;
          m->bos = jb;
          m->n = jn;
          m->a = ja;
          m->s = js;
          m->r = jr;
          m->A = jA;
#pragma unroll
          for (int t = 0; t < QMAX; ++t) m->beta[t] = jbeta[t];
          if (jf & kLive) {
            uint32_t total = 0;
            issue_small<KD, QMAX>(p, sl, m, jh, &bars.sm_full[slot], false, &total);
            mbar_arrive_expect_tx(&bars.sm_full[slot], total);
            uint32_t again = 0;
            issue_small<KD, QMAX>(p, sl, m, jh, &bars.sm_full[slot], true, &again);
          } else {
            mbar_arrive(&bars.sm_full[slot]);
          }
          ++sm_cnt;
          if (jf & kLive) {
            const float* src = p.state + js * p.state_slot_stride + static_cast<long long>(jh) * KD * KD;
            for (int c = 0; c < kGemvWarps && ok; ++c) {
              const int pos = ch_cnt % Lay::kNumChunk;
              const uint32_t cph = (ch_cnt / Lay::kNumChunk) & 1;
              ok = mbar_wait_or_abort(&bars.ch_empty[pos], cph ^ 1, abort_flag);
              if (ok) {
                mbar_arrive_expect_tx(&bars.ch_full[pos], Lay::kChunk);
                bulk_g2s(smem + Lay::oChunks + pos * Lay::kChunk, src + c * Lay::RW * KD, Lay::kChunk,
                         &bars.ch_full[pos]);
                ++ch_cnt;
              }
            }
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
    }
  }
  if (!ok && lane == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

// ---------------------------------------------------------------- prep

template <int KD, int QMAX>
__device__ void prep(const VerifyParams& p, unsigned char* smem, int pt, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX>;
  Bars<KD, QMAX> bars(smem);
  volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::oMisc);
  float* part = reinterpret_cast<float*>(smem + Lay::oPart);
  const int pw = pt >> 5;
  const int lane = pt & 31;
  const int items = p.B * p.H;
  const long long HK = static_cast<long long>(p.H) * KD;
  const int Lc = p.Q + kConvWidth - 2;
  uint32_t sm_cnt = 0, op_cnt = 0;
  bool alive = true;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int slot = sm_cnt % Lay::kNumSmall;
    const uint32_t ph = (sm_cnt / Lay::kNumSmall) & 1;
    if (pt == 0) misc[1] = mbar_wait_or_abort(&bars.sm_full[slot], ph, abort_flag) ? 1 : 0;
    named_barrier(kBarPrep, kPrepThreads);
    if (!misc[1]) {
      alive = false;
      break;
    }
    if (pt != 0) mbar_acquire_seen(&bars.sm_full[slot], ph);
    const unsigned char* sl = smem + Lay::oSmall + slot * Lay::kSmall;
    const SmallMeta<QMAX>& m = *reinterpret_cast<const SmallMeta<QMAX>*>(sl);
    const int flags = m.flags;
    const int n = m.n;
    const int bos = m.bos;
    const int h = it - (it / p.H) * p.H;
    if (!(flags & kLive)) {
      if (flags & kNull) {  // null slot: zero outputs, nothing else
        for (int i = pt; i < n * KD; i += kPrepThreads) {
          const int t = i / KD;
          p.out[static_cast<long long>(bos + t) * p.out_stride + static_cast<long long>(h) * KD + (i - t * KD)] = 0;
        }
      }
      named_barrier(kBarPrep, kPrepThreads);
      if (pt == 0) mbar_arrive(&bars.sm_empty[slot]);
      ++sm_cnt;
      continue;
    }
    const int os = op_cnt % Lay::kNumOp;
    const uint32_t oph = (op_cnt / Lay::kNumOp) & 1;
    if (pt == 0) misc[4] = mbar_wait_or_abort(&bars.op_empty[os], oph ^ 1, abort_flag) ? 1 : 0;
    named_barrier(kBarPrep, kPrepThreads);
    if (!misc[4]) {
      alive = false;
      break;
    }
    unsigned char* op = smem + Lay::oOp + os * Lay::kOp;
    float* op_vec = reinterpret_cast<float*>(op + Lay::kOpVec);
    float* op_v = reinterpret_cast<float*>(op + Lay::kOpV);
    float* op_mn = reinterpret_cast<float*>(op + Lay::kOpMN);
    const long long s = m.s;
    const long long r = m.r;
    const int a = m.a;

    // ---- conv + SiLU: thread k owns channels q_k, k_k and v_k of the head ----
    float qv[QMAX], kv[QMAX], eg[QMAX];
#pragma unroll
    for (int t = 0; t < QMAX; ++t) qv[t] = kv[t] = eg[t] = 0.0f;
    if (pt < KD) {
      const int k = pt;
      const uint16_t* conv = reinterpret_cast<const uint16_t*>(sl + Lay::kConv);
      uint16_t* kg = p.key_gate + r * p.kg_stride + static_cast<long long>(h) * p.Q * 2 * KD;
#pragma unroll
      for (int g = 0; g < 3; ++g) {
        float w[kConvWidth];
        if (p.conv_weight_fp32) {
          const float4 wv = reinterpret_cast<const float4*>(sl + Lay::kW)[g * KD + k];
          w[0] = wv.x; w[1] = wv.y; w[2] = wv.z; w[3] = wv.w;
        } else {
          const uint2 wv = reinterpret_cast<const uint2*>(sl + Lay::kW)[g * KD + k];
          w[0] = bf16_to_f32(wv.x & 0xffff); w[1] = bf16_to_f32(wv.x >> 16);
          w[2] = bf16_to_f32(wv.y & 0xffff); w[3] = bf16_to_f32(wv.y >> 16);
        }
        uint16_t seq[kConvWidth - 1 + QMAX];
#pragma unroll
        for (int j = 0; j < kConvWidth - 1; ++j)
          seq[j] = p.conv_dim_first ? conv[(g * KD + k) * Lc + a - 1 + j] : conv[((a - 1 + j) * 3 + g) * KD + k];
#pragma unroll
        for (int t = 0; t < QMAX; ++t)
          seq[kConvWidth - 1 + t] =
              (t < n) ? *reinterpret_cast<const uint16_t*>(sl + Lay::kAct + (t * 3 + g) * Lay::kSeg +
                                                           m.act_off[t * 3 + g] + 2 * k)
                      : 0;
#pragma unroll
        for (int t = 0; t < QMAX; ++t) {
          if (t < n) {
            const float x[kConvWidth] = {bf16_to_f32(seq[t]), bf16_to_f32(seq[t + 1]), bf16_to_f32(seq[t + 2]),
                                         bf16_to_f32(seq[t + 3])};
            const uint16_t y = conv_silu_bf16(w, x, !p.conv_weight_fp32);
            const float yf = bf16_to_f32(y);
            if (g == 0) qv[t] = yf;
            if (g == 1) {
              kv[t] = yf;
              kg[t * 2 * KD + k] = y;  // key record: the bf16 conv output
            }
            if (g == 2) op_v[t * KD + k] = yf;
          }
        }
        // rolled conv state, in place: taps 0 .. W-3+n <- seq[1 .. W-2+n]
        uint16_t* cs = p.conv_state + s * p.conv_slot_stride;
        const long long ch = g * HK + static_cast<long long>(h) * KD + k;
#pragma unroll
        for (int j = 0; j < kConvWidth - 2 + QMAX; ++j) {
          if (j < kConvWidth - 2 + n) {
            if (p.conv_dim_first)
              cs[ch * Lc + j] = seq[j + 1];
            else
              cs[static_cast<long long>(j) * 3 * HK + ch] = seq[j + 1];
          }
        }
      }
      // gate record (bit copy) and decay factors
      const float dtb = reinterpret_cast<const float*>(sl + Lay::kDt)[k];
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        if (t < n) {
          const uint16_t rg = *reinterpret_cast<const uint16_t*>(sl + Lay::kGate + t * Lay::kSeg + m.gate_off[t] + 2 * k);
          kg[t * 2 * KD + KD + k] = rg;
          eg[t] = expf(kda_gate(bf16_to_f32(rg), dtb, m.A, p.lower_bound_gate, p.lower_bound));
        }
      }
    }
    // ---- norms ----
#pragma unroll
    for (int t = 0; t < QMAX; ++t) {
      if (t < n) {
        const float qq = warp_sum(qv[t] * qv[t]);
        const float kk = warp_sum(kv[t] * kv[t]);
        if (lane == 0) {
          part[pw * Lay::kPartPerWarp + t] = qq;
          part[pw * Lay::kPartPerWarp + QMAX + t] = kk;
        }
      }
    }
    named_barrier(kBarPrep, kPrepThreads);
    float kn[QMAX], qn[QMAX];
#pragma unroll
    for (int t = 0; t < QMAX; ++t) {
      kn[t] = qn[t] = 0.0f;
      if (t < n) {
        float qq = 0.0f, kk = 0.0f;
#pragma unroll
        for (int w = 0; w < kPrepWarps; ++w) {
          qq += part[w * Lay::kPartPerWarp + t];
          kk += part[w * Lay::kPartPerWarp + QMAX + t];
        }
        kn[t] = kv[t] * rsqrtf(kk + 1e-6f);
        qn[t] = qv[t] * (rsqrtf(qq + 1e-6f) * p.k_scale);
      }
    }
    // ---- closed-form operands: X_t = D_t k^_t, Y_t = D_t q^_t, M, N ----
    if (pt < KD) {
      float D = 1.0f;
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        if (t < n) {
          D *= eg[t];
          op_vec[t * KD + pt] = D * kn[t];
          op_vec[(n + t) * KD + pt] = D * qn[t];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < QMAX; ++u) {
      float wu = kn[u];  // k^_u * D_{u+1..t}
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        if (t > u) wu *= eg[t];
        float mval = 0.0f, nval = 0.0f;
        if (u < n && t < n && t >= u) {
          if (t > u) mval = warp_sum(wu * kn[t]);
          nval = warp_sum(wu * qn[t]);
        }
        if (lane == 0) {
          if (t > u) part[pw * Lay::kPartPerWarp + 2 * QMAX + t * QMAX + u] = mval;  // M_tu
          if (t >= u) part[pw * Lay::kPartPerWarp + 2 * QMAX + u * QMAX + t] = nval;  // N_tu
        }
      }
    }
    named_barrier(kBarPrep, kPrepThreads);
    if (pt < QMAX * QMAX) {
      float acc = 0.0f;
#pragma unroll
      for (int w = 0; w < kPrepWarps; ++w) acc += part[w * Lay::kPartPerWarp + 2 * QMAX + pt];
      op_mn[pt] = acc;
    }
    if (pt == 0) {
      OpMeta<QMAX>* om = reinterpret_cast<OpMeta<QMAX>*>(op);
      om->flags = kLive;
      om->bos = bos;
      om->n = n;
      om->h = h;
      om->r = r;
#pragma unroll
      for (int t = 0; t < QMAX; ++t) om->beta[t] = m.beta[t];
    }
    named_barrier(kBarPrep, kPrepThreads);
    if (pt == 0) {
      mbar_arrive(&bars.sm_empty[slot]);
      mbar_arrive(&bars.op_full[os]);
    }
    ++sm_cnt;
    ++op_cnt;
  }
  if (pt == 0) {
    if (alive) {  // end marker for the gemv warps
      const int os = op_cnt % Lay::kNumOp;
      const uint32_t oph = (op_cnt / Lay::kNumOp) & 1;
      if (mbar_wait_or_abort(&bars.op_empty[os], oph ^ 1, abort_flag)) {
        reinterpret_cast<OpMeta<QMAX>*>(smem + Lay::oOp + os * Lay::kOp)->flags = kEnd;
        mbar_arrive(&bars.op_full[os]);
      } else {
        alive = false;
      }
    }
    if (!alive) {
      report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
      *abort_flag = 1;
    }
  }
}

// ---------------------------------------------------------------- gemv

// Dot products of a warp's RW state rows with NCG operand vectors.  Lane =
// 8 rs + kq covers rows 4i + rs (i < RW/4) and the float4 key chunks
// 4kq + 32j (j < KD/32): a warp-wide LDS.128 reads 4 rows x 128 contiguous
// bytes, and the 8 lanes of a row share a broadcast operand load.  The 8
// partial sums of a row meet in a three-stage reduce-scatter.
template <int W>
__device__ __forceinline__ void reduce_scatter_stage(float* acc, int mask, bool upper) {
#pragma unroll
  for (int i = 0; i < W / 2; ++i) {
    const float send = upper ? acc[i] : acc[i + W / 2];
    const float keep = upper ? acc[i + W / 2] : acc[i];
    acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
  }
}

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
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int k0 = 4 * kq + 32 * j;
    float4 vv[NCG];
#pragma unroll
    for (int c = 0; c < NCG; ++c) vv[c] = *reinterpret_cast<const float4*>(vec + c * KD + k0);
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const float4 sv = *reinterpret_cast<const float4*>(st + (4 * i + rs) * KD + k0);
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
__device__ void gemv(const VerifyParams& p, unsigned char* smem, int gw, int lane, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX>;
  constexpr int RW = Lay::RW;
  Bars<KD, QMAX> bars(smem);
  volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::oMisc);
  float* red = reinterpret_cast<float*>(smem + Lay::oRed) + gw * Lay::kRedPerWarp;
  const bool leader = gw == 0 && lane == 0;
  uint32_t op_cnt = 0, live = 0;
  bool alive = true;
  for (;;) {
    const int os = op_cnt % Lay::kNumOp;
    const uint32_t oph = (op_cnt / Lay::kNumOp) & 1;
    if (leader) misc[2] = mbar_wait_or_abort(&bars.op_full[os], oph, abort_flag) ? 1 : 0;
    named_barrier(kBarGemv, kGemvThreads);
    if (!misc[2]) {
      alive = false;
      break;
    }
    if (!leader) mbar_acquire_seen(&bars.op_full[os], oph);
    const unsigned char* op = smem + Lay::oOp + os * Lay::kOp;
    const OpMeta<QMAX>& om = *reinterpret_cast<const OpMeta<QMAX>*>(op);
    if (om.flags & kEnd) break;
    const float* op_vec = reinterpret_cast<const float*>(op + Lay::kOpVec);
    const float* op_v = reinterpret_cast<const float*>(op + Lay::kOpV);
    const float* op_mn = reinterpret_cast<const float*>(op + Lay::kOpMN);
    const int n = om.n;
    const uint32_t pc = live * kGemvWarps + gw;
    const int pos = pc % Lay::kNumChunk;
    const uint32_t cph = (pc / Lay::kNumChunk) & 1;
    bool got = true;
    if (lane == 0) got = mbar_wait_or_abort(&bars.ch_full[pos], cph, abort_flag);
    got = __shfl_sync(0xffffffffu, got, 0);
    if (got) {
      if (lane != 0) mbar_acquire_seen(&bars.ch_full[pos], cph);
      const float* st = reinterpret_cast<const float*>(smem + Lay::oChunks + pos * Lay::kChunk);
      for (int cg = 0; cg < 2 * n; cg += 8) {
        switch (min(8, 2 * n - cg)) {
          case 2: gemv_chunk<KD, 2>(st, op_vec + cg * KD, red + cg * RW, lane); break;
          case 4: gemv_chunk<KD, 4>(st, op_vec + cg * KD, red + cg * RW, lane); break;
          case 6: gemv_chunk<KD, 6>(st, op_vec + cg * KD, red + cg * RW, lane); break;
          default: gemv_chunk<KD, 8>(st, op_vec + cg * KD, red + cg * RW, lane); break;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.ch_empty[pos]);
      // ---- corrections and outputs of the warp's rows ----
      if (lane < RW) {
        const int row = gw * RW + lane;
        float* corr = p.corr + om.r * p.corr_stride + static_cast<long long>(om.h) * p.Q * KD;
        float cv[QMAX];
#pragma unroll
        for (int t = 0; t < QMAX; ++t) {
          if (t < n) {
            float x = op_v[t * KD + row] - red[t * RW + lane];
#pragma unroll
            for (int u = 0; u < t; ++u) x = fmaf(-op_mn[t * QMAX + u], cv[u], x);
            const float c = x * om.beta[t];
            cv[t] = c;
            float o = red[(n + t) * RW + lane];
#pragma unroll
            for (int u = 0; u <= t; ++u) o = fmaf(op_mn[u * QMAX + t], cv[u], o);
            corr[t * KD + row] = c;
            p.out[static_cast<long long>(om.bos + t) * p.out_stride + static_cast<long long>(om.h) * KD + row] =
                f32_to_bf16(o);
          }
        }
      }
    } else if (lane == 0) {
      misc[3] = 1;
    }
    named_barrier(kBarGemv, kGemvThreads);
    if (misc[3]) {
      alive = false;
      break;
    }
    if (leader) mbar_arrive(&bars.op_empty[os]);
    ++op_cnt;
    ++live;
  }
  if (!alive && leader) {
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
    for (int i = 0; i < Lay::kNumOp; ++i) {
      mbar_init(&bars.op_full[i], 1);
      mbar_init(&bars.op_empty[i], 1);
    }
    for (int i = 0; i < 8; ++i) misc[i] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) {
    produce<KD, QMAX>(p, smem, tid & 31, misc);
  } else if (warp <= kPrepWarps) {
    prep<KD, QMAX>(p, smem, tid - 32, misc);
  } else {
    gemv<KD, QMAX>(p, smem, warp - 1 - kPrepWarps, tid & 31, misc);
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
