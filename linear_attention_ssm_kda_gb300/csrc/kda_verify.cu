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
// never written (except by the fold variant, which writes the folded state).
//
// Schedule.  One persistent CTA per SM walks the (request, head) items
// blockIdx.x + i * gridDim.x (local index i) with four roles that meet only
// at mbarrier rings in shared memory, so the stages of consecutive items
// overlap:
//   inputs (1 warp)  reads request metadata 32 items per round trip and
//                    copies each item's small inputs into a ring: TMA tiles
//                    of its q | k | v (| gate) rows, conv taps and conv
//                    weights when they are 16-byte aligned, otherwise bulk
//                    copies of the 16-byte hulls of each row segment (rows
//                    may start anywhere); dt_bias by a bulk copy;
//   state (1 warp)   streams each live item's 64 KB fp32 state as eight row
//                    chunks into a ring of chunk slots, running ahead of the
//                    arithmetic by two to three items;
//   prep (6 warps)   conv + SiLU of two channels per thread over the window
//                    (the bf16 codes, the key record, the rolled conv taps
//                    stored straight to the slot), then one key channel per
//                    thread: the gates and gate record, the norms and the
//                    closed-form operands X_t, Y_t, M, N, handed on through a
//                    ring of operand slots;
//   gemv (8 warps)   each on its own row chunk of the state: P | R with
//                    packed fp32x2 FMAs, then the corrections and outputs of
//                    its rows.
// Two more variants share the roles: the tcgen05 variant (K = 128) replaces
// the gemv warps by four split warps and one MMA thread (products on the
// tensor cores, tensor-core path below), and the fold variant first folds
// each item's pending records of the previous step into its state chunk and
// stores the folded checkpoint back (fold_chunk).
// Every wait is bounded; a timeout sets KDA_DEVERR_TIMEOUT and an abort flag
// that stops the other roles.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "kda_device.cuh"

namespace kda {

namespace {

constexpr int kConvWidth = 4;
constexpr int kPrepWarps = 6;  // two conv channels per thread, then one key channel per thread
constexpr int kGemvWarps = 8;  // one state row chunk (16 rows at K = 128) each
constexpr int kPrepConvThreads = 32 * kPrepWarps;
constexpr int kBarPrep = 1;
constexpr int kSmemLimit = 227 * 1024;
// misc ints in shared memory
constexpr int kMiscAbort = 0;
constexpr int kMiscPrepFail = 1;
constexpr int kMiscTaddr = 4;  // tensor-memory base of the tensor-core path
constexpr int kSplitWarps = 4;  // tensor-core path: warps 8 .. 11 form the low parts and read out the products
constexpr int kMmaWarp = 2 + kPrepWarps + kSplitWarps;  // warp 12 issues the MMAs

constexpr int ru(int x, int a) { return (x + a - 1) / a * a; }

// Kernel variants: the CUDA-core verify, the tcgen05 verify (K = 128: the
// default for windows of 8, forced by KDA_VERIFY_TCGEN05), and the
// CUDA-core verify that first folds each request's pending records of the
// previous step into its checkpoint.
enum : int { kVarPlain = 0, kVarTcgen05 = 1, kVarFold = 2 };

enum : int { kLive = 1, kNull = 2 };

// Inputs warp -> prep, per item.
template <int QMAX>
struct SmallMeta {
  int flags, bos, n, a;
  long long s, r;
  float A, pad;
  float beta[QMAX];
  int fold_m, pad2;  // fold variant: pending records to fold, their row
  long long fold_r;
};

// Prep -> gemv, per item (head of an operand slot).
template <int QMAX>
struct OpMeta {
  int flags, bos, n, pad;
  long long r;
  float beta[QMAX];
  int fold_m, pad2;   // fold variant: pending records folded into the chunk,
  long long s;        // the slot the folded state goes back to,
  float rkf[QMAX];    // and 1 / |k_u| (with the eps) of each pending key
};

template <int KD, int QMAX, int VAR>
struct Layout {
  static_assert(7 * QMAX + 10 <= 96, "small-input copies per item exceed three per lane");
  // Tensor-core instantiation (K = 128, windows of 4 or 8 tokens): the state
  // streams as K-slices of 32 (128 rows x 128 bytes, 128-byte swizzle) and the
  // products S0 [X | Y] come from tcgen05 MMAs; otherwise CUDA-core gemv warps.
  static_assert(VAR != kVarTcgen05 || (KD == 128 && (QMAX == 4 || QMAX == 8)), "the tensor-core path covers K = 128");
  static_assert(VAR != kVarFold || QMAX <= 4, "the fold variant covers windows up to 4");
  static constexpr bool kTC = VAR == kVarTcgen05;
  static constexpr bool kFold = VAR == kVarFold;
  static constexpr int kThreads = 32 * (kTC ? kMmaWarp + 1 : 2 + kPrepWarps + kGemvWarps);
  static constexpr int RW = KD / kGemvWarps;  // state rows per gemv warp (one chunk)
  static constexpr int kChunk = kTC ? 128 * 32 * 4 : RW * KD * 4;  // bytes per state unit (chunk or K-slice)
  static constexpr int kLcMax = QMAX + kConvWidth - 2;
  static constexpr int kSeg = KD * 2 + 16;    // hull of one row segment
  static constexpr int kNumSmall = QMAX <= 4 ? 3 : 2;  // small-input ring
  // small slot
  static constexpr int kAct = ru(int(sizeof(SmallMeta<QMAX>)), 128);  // [QMAX][3] hulls
  static constexpr int kGate = ru(kAct + QMAX * 3 * kSeg, 128);       // [QMAX] hulls
  static constexpr int kConv = ru(kGate + QMAX * kSeg, 128);           // the head's conv taps
  static constexpr int kW = ru(kConv + 3 * KD * kLcMax * 2, 128);      // [3][KD][W] weights
  static constexpr int kDt = ru(kW + 3 * KD * kConvWidth * 4, 128);    // [KD] dt_bias
  // fold variant: the pending records of the item, [QMAX][2K] bf16 key/gate
  // and [QMAX][V] fp32 corrections (V == K)
  static constexpr int kFoldKg = ru(kDt + KD * 4, 128);
  static constexpr int kFoldC = kFoldKg + (kFold ? QMAX * 2 * KD * 2 : 0);
  static constexpr int kSmall = ru(kFoldC + (kFold ? QMAX * KD * 4 : 0), 128);
  // operand slot (prep -> gemv).  Tensor-core path: first the MMA's B operand,
  // [X | Y]_hi rows 0..7 and [X | Y]_lo rows 8..15, as four K-slices of
  // [16][32] fp32 with the 128-byte swizzle (8 KB), then the rest.
  static constexpr int kMmaN = 4 * QMAX;          // MMA N: the 2 QMAX vectors' hi rows, then their lo rows
  static constexpr int kBSlice = kMmaN * 128;     // bytes of the B operand per K-slice of 32
  static constexpr int kDCols = kMmaN;            // tensor-memory columns per D buffer (two buffers)
  static constexpr int kTmemCols = 2 * kDCols < 32 ? 32 : 2 * kDCols;
  static_assert(kTmemCols >= 2 * kDCols && kTmemCols <= 512, "two D buffers fit the tensor-memory allocation");
  static constexpr int kOpMeta = kTC ? 4 * kBSlice : 0;
  static constexpr int kOpVec = ru(kOpMeta + int(sizeof(OpMeta<QMAX>)), 16);  // [2 QMAX][KD] X_t | Y_t
  static constexpr int kOpV = kTC ? kOpVec : kOpVec + 2 * QMAX * KD * 4;        // [QMAX][KD] v_t
  static constexpr int kOpMN = kOpV + QMAX * KD * 4;                            // [QMAX][QMAX] M | N
  // fold variant: prod_u e^{g_u} [K], the pending k_u prod_{w>u} e^{g_w}
  // (unnormalised) [QMAX][K] and the pending corrections [QMAX][V]
  static constexpr int kOpDall = ru(kOpMN + QMAX * QMAX * 4, 16);
  static constexpr int kOpKd = kOpDall + (kFold ? KD * 4 : 0);
  static constexpr int kOpFc = kOpKd + (kFold ? QMAX * KD * 4 : 0);
  static constexpr int kOp = ru(kOpFc + (kFold ? QMAX * KD * 4 : 0), kTC ? 1024 : 128);
  // prep runs up to two items ahead of the gemv team; on the tensor-core path
  // an item's slot is also held until its readout, one item later
  static constexpr int kNumOp = kTC ? (QMAX <= 4 ? 4 : 3) : QMAX <= 4 ? 3 : 2;
  // per-item scratch of the prep team
  static constexpr int kXs = 2 * QMAX * KD * 4;                        // [2][QMAX][KD] q | k conv outputs
  // per-warp scratch
  static constexpr int kRedPerWarp = kTC ? 0 : 2 * QMAX * RW;         // floats
  static constexpr int kFoldIdx = 2 * QMAX + QMAX * QMAX;  // fold variant: |k_u|^2 of the pending keys
  static constexpr int kPart = ru(kFoldIdx + (kFold ? QMAX : 0), 32);         // reduced values per prep warp
  static constexpr int kFixed = kNumSmall * kSmall + kNumOp * kOp + kXs + kGemvWarps * kRedPerWarp * 4 +
                                kPrepWarps * kPart * 4 + 32 + (2 * kNumSmall + 2 * kNumOp + 4) * 8 +
                                (kTC ? 1024 : 0);
  static constexpr int kBarsPerChunk = kTC ? 4 : 2;
  static constexpr int kChunkFit = (kSmemLimit - kFixed - 64 * kBarsPerChunk * 8) / kChunk;
  static constexpr int kNumChunk = kChunkFit > 64 ? 64 : kChunkFit;
  // CTA layout
  static constexpr int oChunks = 0;
  static constexpr int oSmall = oChunks + kNumChunk * kChunk;
  static constexpr int oOp = ru(oSmall + kNumSmall * kSmall, kTC ? 1024 : 128);
  static constexpr int oXs = oOp + kNumOp * kOp;
  static constexpr int oRed = oXs + kXs;
  static constexpr int oPart = oRed + kGemvWarps * kRedPerWarp * 4;
  static constexpr int oMisc = oPart + kPrepWarps * kPart * 4;  // int[8]
  static constexpr int oBars = ru(oMisc + 32, 8);
  static constexpr int kNumBars = kBarsPerChunk * kNumChunk + 2 * kNumSmall + 2 * kNumOp + 4;
  static constexpr int kBytes = oBars + kNumBars * 8;
  static_assert(kBytes <= kSmemLimit, "shared memory budget");
  // at least six K-slices (tensor cores), 1.5 items of chunks (fold variant,
  // whose slots carry the pending records) or two items of chunks in flight
  static_assert(kNumChunk >= (kTC ? 6 : kFold ? 3 * kGemvWarps / 2 : 2 * kGemvWarps), "state in flight");
};

template <int KD, int QMAX, int VAR>
struct Bars {
  uint64_t *ch_full, *ch_empty, *sm_full, *sm_empty, *op_full, *op_empty, *d_full, *d_empty, *hi_done, *lo_full;
  __device__ explicit Bars(unsigned char* smem) {
    using Lay = Layout<KD, QMAX, VAR>;
    uint64_t* b = reinterpret_cast<uint64_t*>(smem + Lay::oBars);
    ch_full = b;
    ch_empty = b + Lay::kNumChunk;
    sm_full = b + 2 * Lay::kNumChunk;
    sm_empty = sm_full + Lay::kNumSmall;
    op_full = sm_empty + Lay::kNumSmall;
    op_empty = op_full + Lay::kNumOp;
    d_full = op_empty + Lay::kNumOp;   // [2] tensor-core path
    d_empty = d_full + 2;              // [2]
    hi_done = d_empty + 2;             // [kNumChunk]
    lo_full = hi_done + Lay::kNumChunk;  // [kNumChunk]
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
  ok = __all_sync(0xffffffffu, ok);
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
  int fold_m;
  long long fold_r;
};

template <int QMAX>
__device__ __forceinline__ ItemMeta<QMAX> decode_item(const VerifyParams& p, int it, bool valid, bool report_errors) {
  ItemMeta<QMAX> m{0, 0, 0, 0, 1, 0, 0, 0, 0};
  if (!valid) return m;
  const int b = it / p.H;
  m.h = it - b * p.H;
  m.bos = p.qsl[b];
  const int len = p.qsl[b + 1] - m.bos;
  m.s = p.state_indices[b];
  m.r = p.record_indices ? static_cast<long long>(p.record_indices[b]) : m.s;
  m.a = p.num_accepted_prev ? min(max(p.num_accepted_prev[b], 1), p.Q) : 1;
  m.n = min(max(len, 0), p.Q);
  if (p.fold_qsl != nullptr) {  // the previous step's pending records, folded first
    const int plen = p.fold_qsl[b + 1] - p.fold_qsl[b];
    m.fold_m = min(max(p.fold_num_accepted[b], 0), min(max(plen, 0), p.Q));
    m.fold_r = p.fold_record_indices ? static_cast<long long>(p.fold_record_indices[b]) : m.s;
  }
  if (len < 0 || (m.n > 0 && (m.bos < 0 || m.bos + m.n > p.T))) {
    if (report_errors) report(p.workspace, KDA_DEVERR_TOKEN_RANGE, it);
  } else if (m.n > 0 || m.fold_m > 0) {
    if (m.s <= p.null_block_id) {
      m.flags = m.n > 0 ? kNull : 0;
    } else if (m.s < 0 || m.s >= p.num_slots) {
      if (report_errors) report(p.workspace, KDA_DEVERR_SLOT_RANGE, it);
    } else if ((m.n > 0 && (m.r < 0 || m.r >= p.num_record_rows)) ||
               (m.fold_m > 0 && (m.fold_r < 0 || m.fold_r >= p.num_record_rows))) {
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
template <int KD, int QMAX, bool DF, int VAR>
__device__ __forceinline__ bool small_copy(const VerifyParams& p, int q, int n, int bos, long long s, int h,
                                           unsigned char* sl, const void** src, void** dst, uint32_t* bytes) {
  using Lay = Layout<KD, QMAX, VAR>;
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
    const int nconv = DF ? 3 : 3 * Lc;
    const uint16_t* cs = p.conv_state + s * p.conv_slot_stride;
    if (q < nconv) {
      if (DF) {
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

// The same copies for the dim-first conv layout when they fit one per lane
// (4n + 7 <= 32): every lane computes its copy without branches, by
// selecting a base, a row, a row stride and a column per kind of copy.
// Kinds by lane q: activation (t = q / 3, g = q % 3) for q < 3n, gate
// (t = q - 3n) for q < 4n, conv taps of group q - 4n, conv weights of group
// q - 4n - 3, dt_bias at q = 4n + 6.  Returns false for lanes past the last copy.
template <int KD, int QMAX, int VAR>
__device__ __forceinline__ bool small_copy_lane(const VerifyParams& p, int q, int n, int bos, long long s, int h,
                                                unsigned char* sl, const void** src, void** dst, uint32_t* bytes) {
  using Lay = Layout<KD, QMAX, VAR>;
  const long long HK = static_cast<long long>(p.H) * KD;
  const int Lc = p.Q + kConvWidth - 2;
  const int wb = p.conv_weight_fp32 ? 4 : 2;
  const int n3 = 3 * n, n4 = 4 * n;
  const bool is_act = q < n3, is_gate = !is_act && q < n4, is_conv = q >= n4 && q < n4 + 3;
  const bool is_w = q >= n4 + 3 && q < n4 + 6, is_dt = q == n4 + 6;
  const int t_act = q / 3;
  const int g = is_act ? q - 3 * t_act : (is_conv ? q - n4 : q - n4 - 3);
  const long long hk = static_cast<long long>(h) * KD;
  const unsigned char* base = is_act    ? reinterpret_cast<const unsigned char*>(p.mixed_qkv)
                              : is_gate ? reinterpret_cast<const unsigned char*>(p.raw_gate)
                              : is_conv ? reinterpret_cast<const unsigned char*>(p.conv_state)
                              : is_w    ? static_cast<const unsigned char*>(p.conv_weight)
                                        : reinterpret_cast<const unsigned char*>(p.dt_bias);
  const long long row = is_act ? bos + t_act : (is_gate ? bos + q - n3 : (is_conv ? s : 0));
  const long long row_bytes = is_act ? p.qkv_stride * 2 : (is_gate ? p.gate_stride * 2 : (is_conv ? p.conv_slot_stride * 2 : 0));
  const long long col = is_act ? (g * HK + hk) * 2
                      : is_gate ? hk * 2
                      : is_conv ? (g * HK + hk) * Lc * 2
                      : is_w    ? (g * HK + hk) * kConvWidth * wb
                                : hk * 4;
  const int dst_off = is_act    ? Lay::kAct + q * Lay::kSeg
                      : is_gate ? Lay::kGate + (q - n3) * Lay::kSeg
                      : is_conv ? Lay::kConv + g * KD * Lc * 2
                      : is_w    ? Lay::kW + g * KD * kConvWidth * wb
                                : Lay::kDt;
  const int len = (is_act || is_gate) ? KD * 2 : (is_conv ? KD * Lc * 2 : (is_w ? KD * kConvWidth * wb : KD * 4));
  const unsigned char* ptr = base + row * row_bytes + col;
  const int off = hull_offset(ptr);
  *src = ptr - off;
  *dst = sl + dst_off;
  *bytes = static_cast<uint32_t>((off + len + 15) & ~15);
  return is_act || is_gate || is_conv || is_w || is_dt;
}

// ---------------------------------------------------------------- inputs warp

// Fold variant: bulk copies of an item's pending records (the first m tokens'
// key/gate rows and corrections of head h in record row r) into its
// small-input slot; the barrier's expected bytes already count them.
template <int KD, int QMAX, int VAR>
__device__ __forceinline__ void fold_copies(const VerifyParams& p, unsigned char* sl, int h, int m, long long r,
                                            uint64_t* bar) {
  using Lay = Layout<KD, QMAX, VAR>;
  const uint16_t* kg = p.key_gate + r * p.kg_stride + static_cast<long long>(h) * p.Q * 2 * KD;
  const float* c = p.corr + r * p.corr_stride + static_cast<long long>(h) * p.Q * KD;
  bulk_g2s(sl + Lay::kFoldKg, kg, static_cast<uint32_t>(m) * 2 * KD * 2, bar);
  bulk_g2s(sl + Lay::kFoldC, c, static_cast<uint32_t>(m) * KD * 4, bar);
}

template <int KD, int QMAX, bool DF, int VAR>
__device__ void produce_inputs(const VerifyParams& p, unsigned char* smem, int lane, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX, VAR>;
  Bars<KD, QMAX, VAR> bars(smem);
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
    // lane j's own item: the per-item header the prep team reads
    SmallMeta<QMAX> own;
    own.flags = im.flags;
    own.bos = im.bos;
    own.n = im.n;
    own.a = im.a;
    own.s = im.s;
    own.r = im.r;
    own.A = A;
    own.pad = 0.0f;
#pragma unroll
    for (int t = 0; t < QMAX; ++t) own.beta[t] = beta[t];
    own.fold_m = im.fold_m;
    own.pad2 = 0;
    own.fold_r = im.fold_r;
    const int count = min(32, nloc - i0);
    for (int j = 0; j < count && ok; ++j) {
      const int i = i0 + j;
      const int jflags = __shfl_sync(0xffffffffu, im.flags, j);
      const int jbos = __shfl_sync(0xffffffffu, im.bos, j);
      const int jn = __shfl_sync(0xffffffffu, im.n, j);
      const long long js = shfl_ll(im.s, j);
      const int jh = __shfl_sync(0xffffffffu, im.h, j);
      const int jfm = Lay::kFold ? __shfl_sync(0xffffffffu, im.fold_m, j) : 0;
      const long long jfr = Lay::kFold ? shfl_ll(im.fold_r, j) : 0;
      // fold variant: the item's pending key/gate and correction records
      const uint32_t fold_bytes = (jflags & kLive) ? static_cast<uint32_t>(jfm) * (2 * KD * 2 + KD * 4) : 0u;
      const int slot = i % Lay::kNumSmall;
      ok = warp_wait(&bars.sm_empty[slot], ((i / Lay::kNumSmall) & 1) ^ 1, lane, abort_flag);
      if (!ok) break;
      unsigned char* sl = smem + Lay::oSmall + slot * Lay::kSmall;
      if (lane == j) *reinterpret_cast<SmallMeta<QMAX>*>(sl) = own;
      __syncwarp();  // orders lane j's header before lane 0's arrival on sm_full
      if ((jflags & kLive) && p.act_mode != 0) {
        // four or five tensor / bulk copies, all from lane 0
        if (lane == 0) {
          const int Lc = p.Q + kConvWidth - 2;
          const int wb = p.conv_weight_fp32 ? 4 : 2;
          const int G = p.act_mode == 1 ? 4 : 3;
          const uint32_t total = KD * G * p.Q * 2 + (p.act_mode == 2 ? KD * p.Q * 2 : 0) + 3 * KD * Lc * 2 +
                                 3 * KD * kConvWidth * wb + KD * 4 + fold_bytes;
          uint64_t* bar = &bars.sm_full[slot];
          mbar_arrive_expect_tx(bar, total);
          if (fold_bytes) fold_copies<KD, QMAX, VAR>(p, sl, jh, jfm, jfr, bar);
          tma_load_3d(sl + Lay::kAct, &p.tm_act, jh * KD, 0, jbos, bar);
          if (p.act_mode == 2) tma_load_2d(sl + Lay::kGate, &p.tm_gate, jh * KD, jbos, bar);
          if (DF)
            tma_load_4d(sl + Lay::kConv, &p.tm_conv, 0, jh * KD * Lc / 128, 0, static_cast<int>(js), bar);
          else
            tma_load_4d(sl + Lay::kConv, &p.tm_conv, jh * KD, 0, 0, static_cast<int>(js), bar);
          tma_load_3d(sl + Lay::kW, &p.tm_w, 0, jh * KD * kConvWidth / 128, 0, bar);
          bulk_g2s(sl + Lay::kDt, p.dt_bias + static_cast<long long>(jh) * KD, KD * 4, bar);
        }
        __syncwarp();
      } else if (jflags & kLive) {
        // at most 7 QMAX + 10 copies, three per lane; the barrier expects every
        // byte before the first copy can land
        const void* src[3];
        void* dst[3];
        uint32_t bytes[3] = {0, 0, 0};
        uint32_t mine = 0;
        if (DF && 4 * QMAX + 7 <= 32) {  // one copy per lane, computed without branches
          if (!small_copy_lane<KD, QMAX, VAR>(p, lane, jn, jbos, js, jh, sl, &src[0], &dst[0], &bytes[0]))
            bytes[0] = 0;
          mine = bytes[0];
        } else {
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            if (!small_copy<KD, QMAX, DF, VAR>(p, lane + 32 * c, jn, jbos, js, jh, sl, &src[c], &dst[c], &bytes[c]))
              bytes[c] = 0;
            mine += bytes[c];
          }
        }
        mine = __reduce_add_sync(0xffffffffu, mine) + fold_bytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars.sm_full[slot], mine);
          if (fold_bytes) fold_copies<KD, QMAX, VAR>(p, sl, jh, jfm, jfr, &bars.sm_full[slot]);
        }
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

template <int KD, int QMAX, int VAR>
__device__ void produce_state(const VerifyParams& p, unsigned char* smem, int lane, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX, VAR>;
  Bars<KD, QMAX, VAR> bars(smem);
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

// ---------------------------------------------------------------- prep team

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

// Conv + SiLU of one channel (group g of q | k | v, key index k) over the
// window, in three steps so that a thread's channels run interleaved:
// conv_load reads the weights, the W - 1 stored taps and the window inputs
// (zero past n); conv_pairs evaluates NP token pairs on the packed fp32x2 unit
// without branches; conv_roll stores the rolled taps to the slot in global
// memory (taps 0 .. W-3+n <- seq[1 .. W-2+n]; later taps are left as they are).
template <int QMAX>
struct ConvIn {
  float w[kConvWidth];
  uint16_t seq[kConvWidth - 1 + QMAX + 1];
};

template <int KD, int QMAX, bool DF, int VAR>
__device__ __forceinline__ void conv_load(const VerifyParams& p, const unsigned char* sl, int g, int k, int n, int a,
                                          int Lc, uint32_t act_lo, ConvIn<QMAX>& in) {
  using Lay = Layout<KD, QMAX, VAR>;
  const uint16_t* conv = reinterpret_cast<const uint16_t*>(sl + Lay::kConv);
  if (p.conv_weight_fp32) {
    const float4 wv = reinterpret_cast<const float4*>(sl + Lay::kW)[g * KD + k];
    in.w[0] = wv.x; in.w[1] = wv.y; in.w[2] = wv.z; in.w[3] = wv.w;
  } else {
    const uint2 wv = reinterpret_cast<const uint2*>(sl + Lay::kW)[g * KD + k];
    in.w[0] = bf16_to_f32(wv.x & 0xffff); in.w[1] = bf16_to_f32(wv.x >> 16);
    in.w[2] = bf16_to_f32(wv.y & 0xffff); in.w[3] = bf16_to_f32(wv.y >> 16);
  }
  in.seq[kConvWidth - 1 + QMAX] = 0;
#pragma unroll
  for (int j = 0; j < kConvWidth - 1; ++j)
    in.seq[j] = DF ? conv[(g * KD + k) * Lc + a - 1 + j] : conv[((a - 1 + j) * 3 + g) * KD + k];
#pragma unroll
  for (int t = 0; t < QMAX; ++t) {
    uint16_t x;
    if (p.act_mode == 0) {
      // the activation hull of (token t, group g) starts act_lo + 16-byte
      // multiples before the segment: the segment's offset is its address mod 16
      const uint32_t off = (act_lo + static_cast<uint32_t>(t) * static_cast<uint32_t>(p.qkv_stride) * 2u +
                            static_cast<uint32_t>(g) * static_cast<uint32_t>(p.H) * KD * 2u) & 15u;
      x = *reinterpret_cast<const uint16_t*>(sl + Lay::kAct + (t * 3 + g) * Lay::kSeg + off + 2 * k);
    } else {  // tensor tile [t][q | k | v (| gate)][K]
      const int G = p.act_mode == 1 ? 4 : 3;
      x = *reinterpret_cast<const uint16_t*>(sl + Lay::kAct + ((t * G + g) * KD + k) * 2);
    }
    in.seq[kConvWidth - 1 + t] = t < n ? x : static_cast<uint16_t>(0);  // slots past n hold no token
  }
}

template <int NP, int QMAX>
__device__ __forceinline__ void conv_pairs(const ConvIn<QMAX>& in, uint16_t (&y)[QMAX]) {
#pragma unroll
  for (int t = 0; t < QMAX; ++t) y[t] = 0;
#pragma unroll
  for (int pr = 0; pr < NP; ++pr) {
    const int t = 2 * pr;
    const float xa[kConvWidth] = {bf16_to_f32(in.seq[t]), bf16_to_f32(in.seq[t + 1]), bf16_to_f32(in.seq[t + 2]),
                                  bf16_to_f32(in.seq[t + 3])};
    const float xb[kConvWidth] = {bf16_to_f32(in.seq[t + 1]), bf16_to_f32(in.seq[t + 2]),
                                  bf16_to_f32(in.seq[t + 3]), bf16_to_f32(in.seq[t + 4])};
    const uint32_t yy = conv_silu_bf16x2(in.w, xa, xb);
    y[t] = static_cast<uint16_t>(yy & 0xffffu);
    y[t + 1] = static_cast<uint16_t>(yy >> 16);
  }
}

template <int KD, int QMAX, bool DF, int VAR>
__device__ __forceinline__ void conv_roll(const VerifyParams& p, const ConvIn<QMAX>& in, int g, int k, int n, int Lc,
                                          uint16_t* gconv, long long hk) {
  const long long HK = static_cast<long long>(p.H) * KD;
  const long long c = g * HK + hk + k;
#pragma unroll
  for (int j = 0; j < kConvWidth - 2 + QMAX; ++j) {
    if (j < kConvWidth - 2 + n) {
      if (DF)
        gconv[c * Lc + j] = in.seq[j + 1];
      else
        gconv[j * 3 * HK + c] = in.seq[j + 1];
    }
  }
}

// Both channels of a prep thread, their pairs interleaved: np = ceil(n / 2)
// pairs each, the codes of tokens past n zeroed.
template <int QMAX>
__device__ __forceinline__ void conv_two(const ConvIn<QMAX>& in0, const ConvIn<QMAX>& in1, int n,
                                         uint16_t (&y0)[QMAX], uint16_t (&y1)[QMAX]) {
  const int np = (n + 1) >> 1;
  if (QMAX <= 4) {
    if (np <= 1) {
      conv_pairs<1, QMAX>(in0, y0);
      conv_pairs<1, QMAX>(in1, y1);
    } else {
      conv_pairs<(QMAX + 1) / 2, QMAX>(in0, y0);
      conv_pairs<(QMAX + 1) / 2, QMAX>(in1, y1);
    }
  } else {
    switch (np) {
      case 1: conv_pairs<1, QMAX>(in0, y0); conv_pairs<1, QMAX>(in1, y1); break;
      case 2: conv_pairs<2, QMAX>(in0, y0); conv_pairs<2, QMAX>(in1, y1); break;
      case 3: conv_pairs<3, QMAX>(in0, y0); conv_pairs<3, QMAX>(in1, y1); break;
      default: conv_pairs<(QMAX + 1) / 2, QMAX>(in0, y0); conv_pairs<(QMAX + 1) / 2, QMAX>(in1, y1); break;
    }
  }
#pragma unroll
  for (int t = 0; t < QMAX; ++t) {
    y0[t] = t < n ? y0[t] : static_cast<uint16_t>(0);
    y1[t] = t < n ? y1[t] : static_cast<uint16_t>(0);
  }
}

template <int KD, int QMAX, bool DF, int VAR>
__device__ void prep(const VerifyParams& p, unsigned char* smem, int pt, volatile int* misc) {
  using Lay = Layout<KD, QMAX, VAR>;
  constexpr int NREDP = Lay::kPart;  // |q_t|^2, |k_t|^2, raw M / N grid, padded to 32
  constexpr int PER = NREDP / 32;
  Bars<KD, QMAX, VAR> bars(smem);
  volatile int* abort_flag = misc + kMiscAbort;
  float* part = reinterpret_cast<float*>(smem + Lay::oPart);
  float* xs = reinterpret_cast<float*>(smem + Lay::oXs);  // [2][QMAX][KD] q | k
  const int warp = pt >> 5;
  const int lane = pt & 31;
  const int nloc = local_items(p.B * p.H);
  const int Lc = p.Q + kConvWidth - 2;
  const uint32_t qkv_lo = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.mixed_qkv));
  const uint32_t gate_lo = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.raw_gate));
  for (int i = 0; i < nloc; ++i) {
    const int it = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int h = it - (it / p.H) * p.H;
    const int slot = i % Lay::kNumSmall;
    const int oslot = i % Lay::kNumOp;
    unsigned char* sl = smem + Lay::oSmall + slot * Lay::kSmall;
    unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
    const bool ok = warp_wait(&bars.sm_full[slot], (i / Lay::kNumSmall) & 1, lane, abort_flag) &&
                    warp_wait(&bars.op_empty[oslot], ((i / Lay::kNumOp) & 1) ^ 1, lane, abort_flag);
    if (!ok && lane == 0) misc[kMiscPrepFail] = 1;
    const SmallMeta<QMAX> m = *reinterpret_cast<const SmallMeta<QMAX>*>(sl);
    const bool live = ok && (m.flags & kLive);
    const int n = m.n;
    const uint32_t hoff = static_cast<uint32_t>(h) * KD * 2u;
    uint16_t* kg = p.key_gate + m.r * p.kg_stride + static_cast<long long>(h) * p.Q * 2 * KD;

    // ---- conv: channels pt and pt + 192 of the head's 3K (q | k | v) ----
    if (ok && (m.flags & kNull)) {  // null slot: zero outputs, nothing else
      for (int e = pt; e < n * KD; e += kPrepConvThreads) {
        const int t = e / KD;
        p.out[static_cast<long long>(m.bos + t) * p.out_stride + static_cast<long long>(h) * KD + (e - t * KD)] = 0;
      }
    }
    if (live && n > 0) {  // (a fold-only item of the fold variant has no window)
      const uint32_t act_lo = qkv_lo + static_cast<uint32_t>(m.bos) * static_cast<uint32_t>(p.qkv_stride) * 2u + hoff;
      uint16_t* gconv = p.conv_state + m.s * p.conv_slot_stride;
      const long long hk = static_cast<long long>(h) * KD;
      // channels c0 = pt and c1 = pt + 192 of the head's 3K (q | k | v)
      const int c0 = pt, c1 = pt + kPrepConvThreads;
      const bool has1 = c1 < 3 * KD;
      const int g0 = c0 / KD, k0 = c0 - g0 * KD;
      const int g1 = c1 / KD, k1 = c1 - g1 * KD;
      ConvIn<QMAX> in0, in1;
      conv_load<KD, QMAX, DF, VAR>(p, sl, g0, k0, n, m.a, Lc, act_lo, in0);
      if (has1) {
        conv_load<KD, QMAX, DF, VAR>(p, sl, g1, k1, n, m.a, Lc, act_lo, in1);
      } else {
#pragma unroll
        for (int j = 0; j < kConvWidth; ++j) in1.w[j] = 0.0f;
#pragma unroll
        for (int j = 0; j < kConvWidth + QMAX; ++j) in1.seq[j] = 0;
      }
      uint16_t y0[QMAX], y1[QMAX];
      conv_two<QMAX>(in0, in1, n, y0, y1);
      conv_roll<KD, QMAX, DF, VAR>(p, in0, g0, k0, n, Lc, gconv, hk);
      if (has1) conv_roll<KD, QMAX, DF, VAR>(p, in1, g1, k1, n, Lc, gconv, hk);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        if (cc == 1 && !has1) break;
        const int g = cc == 0 ? g0 : g1;
        const int k = cc == 0 ? k0 : k1;
        const uint16_t(&y)[QMAX] = cc == 0 ? y0 : y1;
        if (g < 2) {
#pragma unroll
          for (int t = 0; t < QMAX; ++t) xs[(g * QMAX + t) * KD + k] = bf16_to_f32(y[t]);
          if (g == 1) {
#pragma unroll
            for (int t = 0; t < QMAX; ++t)
              if (t < n) kg[t * 2 * KD + k] = y[t];  // key record: the bf16 conv output
          }
        } else {
          float* opv = reinterpret_cast<float*>(op + Lay::kOpV);
#pragma unroll
          for (int t = 0; t < QMAX; ++t)
            if (t < n) opv[t * KD + k] = bf16_to_f32(y[t]);
        }
      }
    }
    named_barrier(kBarPrep, kPrepConvThreads);
    if (misc[kMiscPrepFail]) break;  // every prep thread sees the same flag here

    // ---- gates, gate record and the per-channel partial sums: key channel k = pt ----
    float qv[QMAX], kv[QMAX], eg[QMAX];
    if (live && pt < KD) {
      const int k = pt;
      const float dtb = reinterpret_cast<const float*>(sl + Lay::kDt)[k];
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        qv[t] = xs[t * KD + k];  // zero past n
        kv[t] = xs[(QMAX + t) * KD + k];
        // every slot of the window is read (rows past n hold other tokens,
        // zeros or stale bytes) and the gate of a missing token is discarded,
        // so the QMAX gates evaluate side by side without branches
        uint16_t rg;
        if (p.act_mode == 0) {
          const uint32_t goff =
              (gate_lo + static_cast<uint32_t>(m.bos + t) * static_cast<uint32_t>(p.gate_stride) * 2u + hoff) & 15u;
          rg = *reinterpret_cast<const uint16_t*>(sl + Lay::kGate + t * Lay::kSeg + goff + 2 * k);
        } else if (p.act_mode == 1) {  // gate rows follow v in the q | k | v | gate tile
          rg = *reinterpret_cast<const uint16_t*>(sl + Lay::kAct + ((t * 4 + 3) * KD + k) * 2);
        } else {
          rg = *reinterpret_cast<const uint16_t*>(sl + Lay::kGate + (t * KD + k) * 2);
        }
        const float e = kda_decay_fast(bf16_to_f32(rg), dtb, m.A, p.lower_bound_gate, p.lower_bound);
        eg[t] = t < n ? e : 0.0f;
        if (t < n) kg[t * 2 * KD + KD + k] = rg;  // gate record: bit copy
      }
      // vals: [t] |q_t|^2, [QMAX + t] |k_t|^2, [2QMAX + t QMAX + u] k_u D_{u+1..t} k_t (u < t),
      //       [2QMAX + u QMAX + t] k_u D_{u+1..t} q_t (u <= t); zero past n (qv = kv = 0 there).
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
      if constexpr (Lay::kFold) {
        // the pending records of the previous step: key k_u and decay e^{g_u}
        // (this layer's gate), the unnormalised k_u prod_{w>u} e^{g_w}, the
        // product of all the decays, |k_u|^2 into the reduction, and the
        // corrections c_u of row v = k handed on to the gemv team
        static_assert(Lay::kFoldIdx + QMAX <= NREDP, "room for the pending keys' norms");
        const int mf = m.fold_m;
        if (mf > 0) {
          const uint16_t* fkg = reinterpret_cast<const uint16_t*>(sl + Lay::kFoldKg);
          const float* fc = reinterpret_cast<const float*>(sl + Lay::kFoldC);
          float* dall = reinterpret_cast<float*>(op + Lay::kOpDall);
          float* kd = reinterpret_cast<float*>(op + Lay::kOpKd);
          float* oc = reinterpret_cast<float*>(op + Lay::kOpFc);
          float kf[QMAX], ef[QMAX];
#pragma unroll
          for (int u = 0; u < QMAX; ++u) {
            kf[u] = u < mf ? bf16_to_f32(fkg[u * 2 * KD + k]) : 0.0f;
            ef[u] = u < mf ? kda_decay_fast(bf16_to_f32(fkg[u * 2 * KD + KD + k]), dtb, m.A, p.lower_bound_gate,
                                            p.lower_bound)
                           : 1.0f;
            vals[Lay::kFoldIdx + u] = kf[u] * kf[u];
            if (u < mf) oc[u * KD + k] = fc[u * KD + k];
          }
          float suffix = 1.0f;
#pragma unroll
          for (int u = QMAX - 1; u >= 0; --u) {
            if (u < mf) kd[u * KD + k] = kf[u] * suffix;
            suffix *= ef[u];
          }
          dall[k] = suffix;
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
    named_barrier(kBarPrep, kPrepConvThreads);
    if (pt == 0) mbar_arrive(&bars.sm_empty[slot]);  // the small inputs are consumed

    // ---- norms, the operands X_t = D_t k^_t, Y_t = D_t q^_t, M and N ----
    if (live && pt < KD) {
      float* vec = reinterpret_cast<float*>(op + Lay::kOpVec);
      float* mn = reinterpret_cast<float*>(op + Lay::kOpMN);
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
      if constexpr (Lay::kTC) {
        // the MMA's B operand: vector c (X_0..X_{n-1}, Y_0..Y_{n-1}, then
        // zeros) split as hi = the value with its low 13 mantissa bits cleared
        // (exact in tf32) in row c and lo = value - hi in row 2 QMAX + c
        unsigned char* bt = op + (pt >> 5) * Lay::kBSlice;
        const int kk = pt & 31;
        auto put = [&](int c, float v) {
          const float hi = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
          *reinterpret_cast<float*>(bt + sw128_offset(c, kk)) = hi;
          *reinterpret_cast<float*>(bt + sw128_offset(2 * QMAX + c, kk)) = v - hi;
        };
        float D = 1.0f;
#pragma unroll
        for (int t = 0; t < QMAX; ++t) {
          if (t < n) {
            D *= eg[t];
            put(t, D * (kv[t] * rk[t]));      // X_t
            put(n + t, D * (qv[t] * rq[t]));  // Y_t
          }
        }
#pragma unroll
        for (int c = 0; c < 2 * QMAX; ++c)
          if (c >= 2 * n) put(c, 0.0f);
      } else {
        float D = 1.0f;
#pragma unroll
        for (int t = 0; t < QMAX; ++t) {
          if (t < n) {
            D *= eg[t];
            vec[t * KD + pt] = D * (kv[t] * rk[t]);        // X_t
            vec[(n + t) * KD + pt] = D * (qv[t] * rq[t]);  // Y_t
          }
        }
      }
      if (pt < QMAX * QMAX) {
        const int i2 = pt / QMAX, j2 = pt - (pt / QMAX) * QMAX;
        float raw = 0.0f;
#pragma unroll
        for (int w = 0; w < KD / 32; ++w) raw += part[w * NREDP + 2 * QMAX + pt];
        // i2 > j2: M = raw rk_j rk_i (t = i2, u = j2); i2 <= j2: N = raw rk_i rq_j (u = i2, t = j2)
        float ri = 0.0f, rj = 0.0f;
#pragma unroll
        for (int t = 0; t < QMAX; ++t) {
          if (t == i2) ri = rk[t];
          if (t == j2) rj = (i2 > j2) ? rk[t] : rq[t];
        }
        mn[pt] = raw * ri * rj;
      }
    }
    if (pt == 0) {
      OpMeta<QMAX>* om = reinterpret_cast<OpMeta<QMAX>*>(op + Lay::kOpMeta);
      om->flags = live ? kLive : 0;
      om->bos = m.bos;
      om->n = n;
      om->pad = 0;
      om->r = m.r;
#pragma unroll
      for (int t = 0; t < QMAX; ++t) om->beta[t] = m.beta[t];
      om->fold_m = 0;
      om->pad2 = 0;
      om->s = m.s;
      if constexpr (Lay::kFold) {
        om->fold_m = live ? m.fold_m : 0;
#pragma unroll
        for (int u = 0; u < QMAX; ++u) {
          float kk = 0.0f;
#pragma unroll
          for (int w = 0; w < KD / 32; ++w) kk += part[w * NREDP + Lay::kFoldIdx + u];
          om->rkf[u] = rsqrtf(kk + 1e-6f);  // k^_u = k_u rsqrt(|k_u|^2 + eps)
        }
      }
    }
    if constexpr (Lay::kTC) fence_async_shared();  // the B operand is read by the tensor cores
    named_barrier(kBarPrep, kPrepConvThreads);
    if (pt == 0) mbar_arrive(&bars.op_full[oslot]);
  }
  if (misc[kMiscPrepFail] && pt == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

// ---------------------------------------------------------------- gemv team

// Dot products of a warp's RW state rows with NCG operand vectors.  Lane =
// 4 rs + kq: four lanes share a row and split its K; a lane covers rows
// rs + 8i (i < RW/8) and, at step j, the float4 key chunk 4 (j ^ (rs & 1)) + kq.
// The xor sends rows of odd rs to the other 64-byte half of the 128-byte bank
// window, so a warp-wide LDS.128 of 8 rows x 64 bytes is conflict-free, and
// the operand loads stay at 8 distinct float4 (one wavefront).  Each dot
// product runs as two interleaved halves in one packed fp32x2 FMA chain
// (elements x, y and z, w of each float4); the halves are added, and the 4
// partial sums of a row meet in a two-stage reduce-scatter.
template <int KD, int NCG, bool kToRed>
__device__ __forceinline__ void gemv_chunk(const float* __restrict__ st, const float* __restrict__ vec,
                                           float* __restrict__ red, int lane, float (&mine)[8]) {
  constexpr int RW = KD / kGemvWarps;
  constexpr int R = RW / 8;   // rows per lane
  constexpr int J = KD / 16;  // float4 chunks per lane and row
  constexpr int NV = R * NCG;
  constexpr int NVP = (NV + 3) / 4 * 4;
  const int kq = lane & 3;
  const int rs = lane >> 2;
  const int flip = rs & 1;
  float2 acc2[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc2[i] = make_float2(0.0f, 0.0f);
  // not unrolled: one step already holds NV independent FMA chains, and the
  // kernel's hot code competes for the instruction cache with four roles
#pragma unroll 1
  for (int j = 0; j < J; ++j) {
    const int kk = 4 * (4 * (j ^ flip) + kq);
    float4 vv[NCG];
#pragma unroll
    for (int c = 0; c < NCG; ++c) vv[c] = *reinterpret_cast<const float4*>(vec + c * KD + kk);
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const float4 sv = *reinterpret_cast<const float4*>(st + (rs + 8 * i) * KD + kk);
#pragma unroll
      for (int c = 0; c < NCG; ++c) {
        acc2[i * NCG + c] = __ffma2_rn(make_float2(sv.x, sv.y), make_float2(vv[c].x, vv[c].y), acc2[i * NCG + c]);
        acc2[i * NCG + c] = __ffma2_rn(make_float2(sv.z, sv.w), make_float2(vv[c].z, vv[c].w), acc2[i * NCG + c]);
      }
    }
  }
  float acc[NVP];
#pragma unroll
  for (int i = 0; i < NVP; ++i) acc[i] = i < NV ? acc2[i].x + acc2[i].y : 0.0f;
  reduce_scatter_stage<NVP>(acc, 2, (kq & 2) != 0);
  reduce_scatter_stage<NVP / 2>(acc, 1, (kq & 1) != 0);
  // lane kq now holds values v = (NVP/4) kq + i: row v / NCG, vector v % NCG
  if constexpr (kToRed) {
#pragma unroll
    for (int i = 0; i < NVP / 4; ++i) {
      const int v = (NVP / 4) * kq + i;
      if (v < NV) {
        const int row = v / NCG;
        const int c = v - row * NCG;
        red[c * RW + rs + 8 * row] = acc[i];
      }
    }
  } else {
    static_assert(NVP / 4 <= 8, "at most eight values per lane stay in registers");
#pragma unroll
    for (int i = 0; i < NVP / 4; ++i) mine[i] = acc[i];
  }
}

// The row-local solve with P | R in registers (K = 128, 16 rows per warp,
// 2N <= 8 vectors in one group): after gemv_chunk<128, 2N, false> lane
// (rs, kq) holds, for row rs + 8 (kq >> 1) of its chunk, P_0..P_{N-1} if kq is
// even and R_0..R_{N-1} if kq is odd.  The two lanes of a row swap their
// halves and both run the recurrence; the even lane stores the corrections,
// the odd lane the outputs.
template <int KD, int QMAX, int N, int VAR>
__device__ __forceinline__ void solve_regs(const VerifyParams& p, const OpMeta<QMAX>& m, const unsigned char* op,
                                           int h, int gw, int lane, const float (&mine)[8]) {
  using Lay = Layout<KD, QMAX, VAR>;
  static_assert(Lay::RW == 16, "two lanes per row: 16 rows per gemv warp");
  const int kq = lane & 3;
  const int row = gw * Lay::RW + (lane >> 2) + 8 * (kq >> 1);
  const bool xlane = (kq & 1) == 0;
  const float* mn = reinterpret_cast<const float*>(op + Lay::kOpMN);
  const float* xv = reinterpret_cast<const float*>(op + Lay::kOpV);
  float P[N], R[N];
#pragma unroll
  for (int t = 0; t < N; ++t) {
    const float other = __shfl_xor_sync(0xffffffffu, mine[t], 1);
    P[t] = xlane ? mine[t] : other;
    R[t] = xlane ? other : mine[t];
  }
  float* corr = p.corr + m.r * p.corr_stride + static_cast<long long>(h) * p.Q * KD + row;
  uint16_t* out = p.out + static_cast<long long>(m.bos) * p.out_stride + static_cast<long long>(h) * KD + row;
  float cv[N];
#pragma unroll
  for (int t = 0; t < N; ++t) {
    float x = xv[t * KD + row] - P[t];
#pragma unroll
    for (int u = 0; u < t; ++u) x = fmaf(-mn[t * QMAX + u], cv[u], x);
    const float c = x * m.beta[t];
    cv[t] = c;
    float o = R[t];
#pragma unroll
    for (int u = 0; u <= t; ++u) o = fmaf(mn[u * QMAX + t], cv[u], o);
    if (xlane)
      corr[t * KD] = c;
    else
      out[static_cast<long long>(t) * p.out_stride] = f32_to_bf16(o);
  }
}

// Fold variant: the gemv warp's chunk (rows gw RW .. gw RW + RW - 1 of the
// item's state, [RW][K] fp32 in shared memory) folded in place with the
// previous step's pending records,
//   S[v, k] <- S[v, k] prod_u e^{g_u}[k] + sum_u (c_u[v] / |k_u|) k_u[k] prod_{w>u} e^{g_w}[k],
// which is the commit's fold; then one lane stores the folded rows back to
// the checkpoint with a bulk copy (its smem read is awaited before the chunk
// slot is released).
template <int KD, int QMAX, int VAR>
__device__ __forceinline__ void fold_chunk(const VerifyParams& p, const OpMeta<QMAX>& m, const unsigned char* op,
                                           int h, int gw, int lane, float* st) {
  using Lay = Layout<KD, QMAX, VAR>;
  constexpr int RW = Lay::RW;
  constexpr int C4 = KD / 4;  // float4 per row
  static_assert(32 % C4 == 0, "a lane keeps one float4 column of the chunk");
  const int kc = lane % C4;
  const float4 d4 = reinterpret_cast<const float4*>(op + Lay::kOpDall)[kc];
  const float* kd = reinterpret_cast<const float*>(op + Lay::kOpKd);
  const float* oc = reinterpret_cast<const float*>(op + Lay::kOpFc);
  const int mf = m.fold_m;
  float4 k4[QMAX];
#pragma unroll
  for (int u = 0; u < QMAX; ++u)
    k4[u] = u < mf ? reinterpret_cast<const float4*>(kd + u * KD)[kc] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float4* s4 = reinterpret_cast<float4*>(st);
#pragma unroll 4
  for (int e = lane; e < RW * C4; e += 32) {
    const int row = e / C4;  // row of the chunk
    float4 v = s4[e];
    v.x *= d4.x;
    v.y *= d4.y;
    v.z *= d4.z;
    v.w *= d4.w;
#pragma unroll
    for (int u = 0; u < QMAX; ++u) {
      if (u < mf) {
        const float c = oc[u * KD + gw * RW + row] * m.rkf[u];
        v.x = fmaf(c, k4[u].x, v.x);
        v.y = fmaf(c, k4[u].y, v.y);
        v.z = fmaf(c, k4[u].z, v.z);
        v.w = fmaf(c, k4[u].w, v.w);
      }
    }
    s4[e] = v;
  }
  fence_async_shared();  // the folded rows are read by the bulk store
  __syncwarp();
  if (lane == 0) {
    float* g = const_cast<float*>(p.state) + m.s * p.state_slot_stride + (static_cast<long long>(h) * KD + gw * RW) * KD;
    bulk_s2g(g, st, RW * KD * 4);
    bulk_commit();
  }
}

template <int KD, int QMAX, int VAR>
__device__ void gemv_team(const VerifyParams& p, unsigned char* smem, int gw, int lane, volatile int* misc) {
  using Lay = Layout<KD, QMAX, VAR>;
  constexpr int RW = Lay::RW;
  Bars<KD, QMAX, VAR> bars(smem);
  volatile int* abort_flag = misc + kMiscAbort;
  float* red = reinterpret_cast<float*>(smem + Lay::oRed) + gw * Lay::kRedPerWarp;
  const int nloc = local_items(p.B * p.H);
  uint32_t live = 0;
  bool ok = true;
  for (int i = 0; i < nloc && ok; ++i) {
    const int it = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int h = it - (it / p.H) * p.H;
    const int oslot = i % Lay::kNumOp;
    ok = warp_wait(&bars.op_full[oslot], (i / Lay::kNumOp) & 1, lane, abort_flag);
    if (!ok) break;
    const unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
    const OpMeta<QMAX> m = *reinterpret_cast<const OpMeta<QMAX>*>(op + Lay::kOpMeta);
    if (m.flags & kLive) {
      const int n = m.n;
      const uint32_t pc = live * kGemvWarps + gw;
      const int pos = pc % Lay::kNumChunk;
      ok = warp_wait(&bars.ch_full[pos], (pc / Lay::kNumChunk) & 1, lane, abort_flag);
      if (!ok) break;
      float* st = reinterpret_cast<float*>(smem + Lay::oChunks + pos * Lay::kChunk);
      const float* vec = reinterpret_cast<const float*>(op + Lay::kOpVec);
      bool stored = false;  // the folded chunk is on its way back to the checkpoint
      if constexpr (Lay::kFold) {
        if (m.fold_m > 0) {
          fold_chunk<KD, QMAX, VAR>(p, m, op, h, gw, lane, st);
          stored = true;
        }
      }
      // the chunk slot goes back to the state warp once the products (and the
      // bulk store of a folded chunk) have read it
      auto release = [&] {
        __syncwarp();
        if (lane == 0) {
          if (stored) bulk_wait_read();
          mbar_arrive(&bars.ch_empty[pos]);
        }
      };
      if (n == 0) {  // fold only: no window to verify
        release();
        ++live;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.op_empty[oslot]);
        continue;
      }
      float mine[8];
      if (KD == 128 && n <= 4) {  // one vector group: P | R stay in registers
        if constexpr (KD == 128) {
          switch (n) {
            case 1:
              gemv_chunk<KD, 2, false>(st, vec, red, lane, mine);
              release();
              solve_regs<KD, QMAX, 1, VAR>(p, m, op, h, gw, lane, mine);
              break;
            case 2:
              gemv_chunk<KD, 4, false>(st, vec, red, lane, mine);
              release();
              solve_regs<KD, QMAX, 2, VAR>(p, m, op, h, gw, lane, mine);
              break;
            case 3:
              gemv_chunk<KD, 6, false>(st, vec, red, lane, mine);
              release();
              solve_regs<KD, QMAX, 3, VAR>(p, m, op, h, gw, lane, mine);
              break;
            default:
              gemv_chunk<KD, 8, false>(st, vec, red, lane, mine);
              release();
              solve_regs<KD, QMAX, 4, VAR>(p, m, op, h, gw, lane, mine);
              break;
          }
        }
        ++live;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.op_empty[oslot]);
        continue;
      }
      for (int cg = 0; cg < 2 * n; cg += 8) {
        switch (min(8, 2 * n - cg)) {
          case 2: gemv_chunk<KD, 2, true>(st, vec + cg * KD, red + cg * RW, lane, mine); break;
          case 4: gemv_chunk<KD, 4, true>(st, vec + cg * KD, red + cg * RW, lane, mine); break;
          case 6: gemv_chunk<KD, 6, true>(st, vec + cg * KD, red + cg * RW, lane, mine); break;
          default: gemv_chunk<KD, 8, true>(st, vec + cg * KD, red + cg * RW, lane, mine); break;
        }
      }
      release();
      if (lane < RW) {
        const int row = gw * RW + lane;
        const float* mn = reinterpret_cast<const float*>(op + Lay::kOpMN);
        const float* xv = reinterpret_cast<const float*>(op + Lay::kOpV);
        float* corr = p.corr + m.r * p.corr_stride + static_cast<long long>(h) * p.Q * KD;
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
            p.out[static_cast<long long>(m.bos + t) * p.out_stride + static_cast<long long>(h) * KD + row] =
                f32_to_bf16(o);
          }
        }
      }
      ++live;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.op_empty[oslot]);
  }
  if (Lay::kFold && lane == 0) bulk_wait_all();  // the folded chunks have reached the checkpoint
  if (!ok && lane == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

// ---------------------------------------------------------------- tensor-core path (K = 128, Q = 4 or 8)
//
// The products P | R = S0 [X_0..X_{n-1} | Y_0..Y_{n-1}] of an item come from
// tcgen05 MMAs: D[128 x 4Q] in tensor memory = S0 [128 x 128] times B^T, B =
// [hi rows 0..2Q-1 | lo rows 2Q..4Q-1] of the 2n <= 2Q operand vectors.  fp32
// accuracy from tf32 inputs: S0 = S_hi + S_lo with S_hi the value with its
// low 13 mantissa bits cleared (exact in tf32) and S_lo = S0 - S_hi (exact in
// fp32, at most 11 significant bits, rounded to tf32 within 2^-21 of S0);
// likewise for B.  Two MMAs per K step, S_hi B^T + S_lo B^T, accumulate
// column c < 2Q = S0 v_c,hi and column 2Q + c = S0 v_c,lo, whose sum is S0 v_c.

// State producer: each live item's state as four K-slices (TMA tiles of 128
// rows x 32 fp32 with the 128-byte swizzle) into the ring of slice slots.
template <int KD, int QMAX, int VAR>
__device__ void tc_produce_state(const VerifyParams& p, unsigned char* smem, int lane, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX, VAR>;
  Bars<KD, QMAX, VAR> bars(smem);
  const int nloc = local_items(p.B * p.H);
  uint32_t g = 0;  // slices issued
  bool ok = true;
  for (int i0 = 0; i0 < nloc && ok; i0 += 32) {
    const int it = static_cast<int>(blockIdx.x) + (i0 + lane) * static_cast<int>(gridDim.x);
    const ItemMeta<QMAX> im = decode_item<QMAX>(p, it, i0 + lane < nloc, false);
    const int count = min(32, nloc - i0);
    for (int j = 0; j < count && ok; ++j) {
      if (!(__shfl_sync(0xffffffffu, im.flags, j) & kLive)) continue;
      const int jh = __shfl_sync(0xffffffffu, im.h, j);
      const int js = static_cast<int>(shfl_ll(im.s, j));
      for (int kb = 0; kb < 4 && ok; ++kb, ++g) {
        const int pos = static_cast<int>(g % Lay::kNumChunk);
        if (lane == 0) {
          ok = mbar_wait_or_abort(&bars.ch_empty[pos], ((g / Lay::kNumChunk) & 1) ^ 1, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(&bars.ch_full[pos], Lay::kChunk);
            tma_load_3d(smem + Lay::oChunks + pos * Lay::kChunk, &p.tm_state, kb * 32, jh * KD, js, &bars.ch_full[pos]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
  }
  if (!ok && lane == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
  // the slots are released by MMA completion: see every release land before
  // the CTA (and its shared memory) goes away
  if (lane == 0) {
    for (uint32_t e = 0; e < static_cast<uint32_t>(Lay::kNumChunk); ++e, ++g)
      (void)mbar_wait_bounded(&bars.ch_empty[g % Lay::kNumChunk], ((g / Lay::kNumChunk) & 1) ^ 1);
  }
}

// MMA issuer (one thread).  Per K-slice of a live item: the 4 K-steps of
// S_hi B^T as soon as the slice has landed (committed to hi_done, after which
// the split team overwrites the slice with its low part), then, one slice
// later, the 4 K-steps of S_lo B^T once the low part is complete (committed
// to the slot's release and, after an item's last slice, to its D buffer).
// Issuing the next slice's S_hi before the previous slice's S_lo keeps the
// split team fed while the tensor cores work.
struct LoPending {
  bool valid, last;
  int pos, oslot;
  uint32_t g, db;
  uint64_t bk;
};

template <int KD, int QMAX, int VAR>
__device__ __forceinline__ bool tc_issue_lo(unsigned char* smem, uint32_t taddr, LoPending& lp,
                                            const volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX, VAR>;
  constexpr uint32_t kIdesc = umma_idesc_tf32(128, Layout<KD, QMAX, VAR>::kMmaN);
  Bars<KD, QMAX, VAR> bars(smem);
  if (!lp.valid) return true;
  lp.valid = false;
  if (!mbar_wait_or_abort(&bars.lo_full[lp.pos], (lp.g / Lay::kNumChunk) & 1, abort_flag)) return false;
  tmem_fence_after();
  const uint64_t a = umma_desc_sw128(smem + Lay::oChunks + lp.pos * Lay::kChunk);
  const uint32_t d = taddr + lp.db * Lay::kDCols;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) umma_tf32(d, a + 2 * ks, lp.bk + 2 * ks, kIdesc, true);
  umma_commit(&bars.ch_empty[lp.pos]);
  if (lp.last) {
    umma_commit(&bars.d_full[lp.db]);
    mbar_arrive(&bars.op_empty[lp.oslot]);
  }
  return true;
}

template <int KD, int QMAX, int VAR>
__device__ void tc_mma(const VerifyParams& p, unsigned char* smem, volatile int* misc) {
  using Lay = Layout<KD, QMAX, VAR>;
  constexpr uint32_t kIdesc = umma_idesc_tf32(128, Layout<KD, QMAX, VAR>::kMmaN);
  Bars<KD, QMAX, VAR> bars(smem);
  volatile int* abort_flag = misc + kMiscAbort;
  const int nloc = local_items(p.B * p.H);
  const uint32_t taddr = static_cast<uint32_t>(misc[kMiscTaddr]);
  uint32_t g = 0, live = 0;
  LoPending lp{false, false, 0, 0, 0, 0, 0};
  bool ok = true;
  for (int i = 0; i < nloc && ok; ++i) {
    const int oslot = i % Lay::kNumOp;
    const unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
    ok = mbar_wait_or_abort(&bars.op_full[oslot], (i / Lay::kNumOp) & 1, abort_flag);
    if (!ok) break;
    if (!(reinterpret_cast<const OpMeta<QMAX>*>(op + Lay::kOpMeta)->flags & kLive)) {
      // finish the previous item first: its operand slot may be the next one
      // the prep team needs
      ok = tc_issue_lo<KD, QMAX, VAR>(smem, taddr, lp, abort_flag);
      mbar_arrive(&bars.op_empty[oslot]);
      continue;
    }
    const uint32_t db = live & 1;
    ok = mbar_wait_or_abort(&bars.d_empty[db], ((live >> 1) & 1) ^ 1, abort_flag);
    const uint64_t b = umma_desc_sw128(op);
    const uint32_t d = taddr + db * Lay::kDCols;
    for (int kb = 0; kb < 4 && ok; ++kb, ++g) {
      const int pos = static_cast<int>(g % Lay::kNumChunk);
      ok = mbar_wait_or_abort(&bars.ch_full[pos], (g / Lay::kNumChunk) & 1, abort_flag);
      if (!ok) break;
      tmem_fence_after();
      const uint64_t a = umma_desc_sw128(smem + Lay::oChunks + pos * Lay::kChunk);
      const uint64_t bk = b + static_cast<uint64_t>(kb) * (Lay::kBSlice >> 4);  // B slice kb
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) umma_tf32(d, a + 2 * ks, bk + 2 * ks, kIdesc, kb > 0 || ks > 0);
      umma_commit(&bars.hi_done[pos]);
      ok = tc_issue_lo<KD, QMAX, VAR>(smem, taddr, lp, abort_flag);
      lp = LoPending{true, kb == 3, pos, oslot, g, db, bk};
    }
    ++live;
  }
  if (ok) ok = tc_issue_lo<KD, QMAX, VAR>(smem, taddr, lp, abort_flag);
  if (!ok) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

// Readout team (4 warps, warp q of the CTA's last warpgroup reads tensor-memory
// lanes 32 q .. 32 q + 31): each lane owns one state row; it sums the hi and
// lo columns into P_t | R_t and runs the row's solve.
template <int KD, int QMAX, int N, int VAR>
__device__ __forceinline__ void tc_solve(const VerifyParams& p, const OpMeta<QMAX>& m, const unsigned char* op, int h,
                                         int row, const float* d) {
  using Lay = Layout<KD, QMAX, VAR>;
  const float* mn = reinterpret_cast<const float*>(op + Lay::kOpMN);
  const float* xv = reinterpret_cast<const float*>(op + Lay::kOpV);
  float* corr = p.corr + m.r * p.corr_stride + static_cast<long long>(h) * p.Q * KD + row;
  uint16_t* out = p.out + static_cast<long long>(m.bos) * p.out_stride + static_cast<long long>(h) * KD + row;
  float cv[N];
#pragma unroll
  for (int t = 0; t < N; ++t) {
    float x = xv[t * KD + row] - (d[t] + d[2 * QMAX + t]);
#pragma unroll
    for (int u = 0; u < t; ++u) x = fmaf(-mn[t * QMAX + u], cv[u], x);
    const float c = x * m.beta[t];
    cv[t] = c;
    float o = d[N + t] + d[2 * QMAX + N + t];
#pragma unroll
    for (int u = 0; u <= t; ++u) o = fmaf(mn[u * QMAX + t], cv[u], o);
    corr[t * KD] = c;
    out[static_cast<long long>(t) * p.out_stride] = f32_to_bf16(o);
  }
}

// Readout of a live item's products, in the split warp that owns tensor-memory
// lanes 32 wq .. 32 wq + 31 (one state row per lane): P_t | R_t = hi column +
// lo column, then the row's solve.  Releases the D buffer and the operand slot.
template <int KD, int QMAX, int VAR>
__device__ __forceinline__ bool tc_readout(const VerifyParams& p, unsigned char* smem, int i, uint32_t live, int wq,
                                           int lane, uint32_t taddr, const volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX, VAR>;
  Bars<KD, QMAX, VAR> bars(smem);
  const int it = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
  const int h = it - (it / p.H) * p.H;
  const int oslot = i % Lay::kNumOp;
  const unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
  const uint32_t db = live & 1;
  if (!warp_wait(&bars.d_full[db], (live >> 1) & 1, lane, abort_flag)) return false;
  tmem_fence_after();
  float d[Lay::kDCols];
  const uint32_t ta = taddr + db * Lay::kDCols + (static_cast<uint32_t>(wq * 32) << 16);
#pragma unroll
  for (int c = 0; c < Lay::kDCols; c += 16) tmem_ld16(ta + c, *reinterpret_cast<float(*)[16]>(d + c));
  tmem_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars.d_empty[db]);
  const OpMeta<QMAX> m = *reinterpret_cast<const OpMeta<QMAX>*>(op + Lay::kOpMeta);
  const int row = wq * 32 + lane;
  if constexpr (QMAX <= 4) {
    switch (m.n) {
      case 1: tc_solve<KD, QMAX, 1, VAR>(p, m, op, h, row, d); break;
      case 2: tc_solve<KD, QMAX, 2, VAR>(p, m, op, h, row, d); break;
      case 3: tc_solve<KD, QMAX, 3, VAR>(p, m, op, h, row, d); break;
      default: tc_solve<KD, QMAX, 4, VAR>(p, m, op, h, row, d); break;
    }
  } else {
    switch (m.n) {
      case 1: tc_solve<KD, QMAX, 1, VAR>(p, m, op, h, row, d); break;
      case 2: tc_solve<KD, QMAX, 2, VAR>(p, m, op, h, row, d); break;
      case 3: tc_solve<KD, QMAX, 3, VAR>(p, m, op, h, row, d); break;
      case 4: tc_solve<KD, QMAX, 4, VAR>(p, m, op, h, row, d); break;
      case 5: tc_solve<KD, QMAX, 5, VAR>(p, m, op, h, row, d); break;
      case 6: tc_solve<KD, QMAX, 6, VAR>(p, m, op, h, row, d); break;
      case 7: tc_solve<KD, QMAX, 7, VAR>(p, m, op, h, row, d); break;
      default: tc_solve<KD, QMAX, 8, VAR>(p, m, op, h, row, d); break;
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars.op_empty[oslot]);
  return true;
}

// Split team (4 warps, each on its own).  A tf32 MMA reads an fp32 operand
// with its low 13 mantissa bits ignored, so a K-slice as loaded is S_hi to the
// tensor cores.  Once its S_hi products are done, the warps overwrite the
// slice in place with its low part S - S_hi for the S_lo products.
// Two slices into an item, the warp reads out the previous live item, whose
// MMAs have completed by then.
template <int KD, int QMAX, int VAR>
__device__ void tc_split(const VerifyParams& p, unsigned char* smem, int st, volatile int* misc) {
  using Lay = Layout<KD, QMAX, VAR>;
  Bars<KD, QMAX, VAR> bars(smem);
  volatile int* abort_flag = misc + kMiscAbort;
  const int lane = st & 31;
  const int wq = st >> 5;
  const int nloc = local_items(p.B * p.H);
  const uint32_t taddr = static_cast<uint32_t>(misc[kMiscTaddr]);
  uint32_t g = 0, live = 0;
  int pending = -1;  // live item awaiting readout
  bool ok = true;
  for (int i = 0; i < nloc && ok; ++i) {
    const int oslot = i % Lay::kNumOp;
    const unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
    ok = warp_wait(&bars.op_full[oslot], (i / Lay::kNumOp) & 1, lane, abort_flag);
    if (!ok) break;
    if (!(reinterpret_cast<const OpMeta<QMAX>*>(op + Lay::kOpMeta)->flags & kLive)) {
      // read the pending item out now: with no live item to follow soon, its
      // operand slot would be missing when the prep team comes round to it
      if (pending >= 0) ok = tc_readout<KD, QMAX, VAR>(p, smem, pending, live - 1, wq, lane, taddr, abort_flag);
      pending = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.op_empty[oslot]);
      continue;
    }
    for (int kb = 0; kb < 4 && ok; ++kb, ++g) {
      const int pos = static_cast<int>(g % Lay::kNumChunk);
      ok = warp_wait(&bars.ch_full[pos], (g / Lay::kNumChunk) & 1, lane, abort_flag) &&
           warp_wait(&bars.hi_done[pos], (g / Lay::kNumChunk) & 1, lane, abort_flag);
      if (!ok) break;
      float4* s4 = reinterpret_cast<float4*>(smem + Lay::oChunks + pos * Lay::kChunk);
#pragma unroll 4
      for (int e = st; e < Lay::kChunk / 16; e += 32 * kSplitWarps) {
        const float4 x = s4[e];
        float4 l;
        l.x = x.x - __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u);
        l.y = x.y - __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u);
        l.z = x.z - __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u);
        l.w = x.w - __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u);
        s4[e] = l;
      }
      fence_async_shared();  // the low parts are read by the tensor cores
      mbar_arrive(&bars.lo_full[pos]);
      if (kb == 1 && pending >= 0) {  // the pending item's MMAs are done by now
        ok = tc_readout<KD, QMAX, VAR>(p, smem, pending, live - 1, wq, lane, taddr, abort_flag);
        pending = -1;
      }
    }
    if (!ok) break;
    pending = i;
    ++live;
  }
  if (ok && pending >= 0) ok = tc_readout<KD, QMAX, VAR>(p, smem, pending, live - 1, wq, lane, taddr, abort_flag);
  if (!ok && lane == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

template <int KD, int QMAX, bool DF, int VAR>
__global__ void __launch_bounds__(Layout<KD, QMAX, VAR>::kThreads, 1) verify_kernel(const __grid_constant__ VerifyParams p) {
  using Lay = Layout<KD, QMAX, VAR>;
  extern __shared__ __align__(1024) unsigned char smem[];
  volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::oMisc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  if (tid == 0) {
    Bars<KD, QMAX, VAR> bars(smem);
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
      // released by the gemv warps, or by the readout warps and the MMA issuer
      mbar_init(&bars.op_empty[i], Lay::kTC ? kSplitWarps + 1 : kGemvWarps);
    }
    if constexpr (Lay::kTC) {
      for (int i = 0; i < Lay::kNumChunk; ++i) {
        mbar_init(&bars.hi_done[i], 1);
        mbar_init(&bars.lo_full[i], 32 * kSplitWarps);
      }
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.d_full[i], 1);
      mbar_init(&bars.d_empty[i], kSplitWarps);
    }
    for (int i = 0; i < 8; ++i)
      if (i != kMiscTaddr) misc[i] = 0;  // the tensor-memory base is written by the allocating warp
    fence_barrier_init();
  }
  if constexpr (Lay::kTC) {
    // the 128-byte swizzle of the MMA operands is anchored at 1024-byte boundaries
    if (smem_u32(smem) & 1023u) {
      if (tid == 0) report(p.workspace, KDA_DEVERR_MISALIGNED, blockIdx.x);
      return;
    }
    // tensor memory for two D buffers of 4 QMAX fp32 columns, owned by the MMA warp
    if (warp == kMmaWarp)
      tmem_alloc(reinterpret_cast<uint32_t*>(const_cast<int*>(misc) + kMiscTaddr), Lay::kTmemCols);
    tmem_fence_before();
  }
  __syncthreads();
  if constexpr (Lay::kTC) tmem_fence_after();
  if (warp == 0) {
    produce_inputs<KD, QMAX, DF, VAR>(p, smem, tid & 31, misc + kMiscAbort);
  } else if (warp == 1) {
    if constexpr (Lay::kTC)
      tc_produce_state<KD, QMAX, VAR>(p, smem, tid & 31, misc + kMiscAbort);
    else
      produce_state<KD, QMAX, VAR>(p, smem, tid & 31, misc + kMiscAbort);
  } else if (warp < 2 + kPrepWarps) {
    prep<KD, QMAX, DF, VAR>(p, smem, tid - 64, misc);
  } else if constexpr (Lay::kTC) {
    if (warp < kMmaWarp)
      tc_split<KD, QMAX, VAR>(p, smem, tid - 32 * (2 + kPrepWarps), misc);
    else if ((tid & 31) == 0)
      tc_mma<KD, QMAX, VAR>(p, smem, misc);
  } else {
    gemv_team<KD, QMAX, VAR>(p, smem, warp - 2 - kPrepWarps, tid & 31, misc);
  }
  if constexpr (Lay::kTC) {
    // every role is done and the MMA issuer has seen its last MMAs complete:
    // release the tensor memory
    tmem_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
      tmem_fence_after();
      tmem_dealloc(static_cast<uint32_t>(misc[kMiscTaddr]), Lay::kTmemCols);
    }
  }
}

// ---------------------------------------------------------------- tensor maps (host)

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once (no link to libcuda).
EncodeTiledFn tensor_map_encoder() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool encode_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  const EncodeTiledFn fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint32_t unit[5] = {1, 1, 1, 1, 1};
  return fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, unit,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps for the small inputs when every start and stride they need is
// 16-byte aligned; otherwise act_mode stays 0 (per-segment hull copies).
//   q | k | v (| gate): dims {HK, 3 or 4 groups, T}, box {K, groups, Q}, at
//     {h K, 0, bos}; rows past T arrive as zeros;
//   gate (separate): dims {HK, T}, box {K, Q}, at {h K, bos};
//   conv taps, dim-first [slots][3HK][Lc]: dims {128, HK Lc / 128, 3, slots},
//     box {128, K Lc / 128, 3, 1}, at {0, h K Lc / 128, 0, s};
//     seq-first [slots][Lc][3HK]: dims {HK, 3, Lc, slots}, box {K, 3, Lc, 1},
//     at {h K, 0, 0, s};
//   conv weights [3HK][W]: dims {128, HK W / 128, 3}, box {128, K W / 128, 3},
//     at {0, h K W / 128, 0}.
// Every box lands in the layout the hull copies would give, except q | k | v
// (| gate), which lands as [t][group][K].
// The fp32 state pool for the tensor-core path, [slots][H K][K] with the slot
// stride given: dims {K, H K, slots}, box {32, 128, 1} with the 128-byte
// swizzle, at {32 kb, h K, s}: K-slice kb of head h's state.
bool build_state_map(VerifyParams& p, int KD) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(KD), static_cast<cuuint64_t>(p.H) * KD,
                              static_cast<cuuint64_t>(p.num_slots)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(KD) * 4, static_cast<cuuint64_t>(p.state_slot_stride) * 4};
  const cuuint32_t box[3] = {32, 128, 1};
  return encode_map(&p.tm_state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.state, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

void build_tensor_maps(VerifyParams& p, int KD) {
  p.act_mode = 0;
  const cuuint64_t H = static_cast<cuuint64_t>(p.H), K = static_cast<cuuint64_t>(KD), HK = H * K;
  const cuuint64_t T = static_cast<cuuint64_t>(p.T), Q = static_cast<cuuint64_t>(p.Q);
  const cuuint64_t Lc = Q + kConvWidth - 2, W = kConvWidth;
  const cuuint64_t wb = p.conv_weight_fp32 ? 4 : 2;
  auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  if (!al16(p.mixed_qkv) || (p.qkv_stride * 2) % 16 != 0) return;
  int mode;
  if (p.raw_gate == p.mixed_qkv + 3 * HK && p.gate_stride == p.qkv_stride &&
      static_cast<cuuint64_t>(p.qkv_stride) >= 4 * HK)
    mode = 1;
  else if (al16(p.raw_gate) && (p.gate_stride * 2) % 16 == 0)
    mode = 2;
  else
    return;
  if (p.conv_dim_first && (K * Lc) % 128 != 0) return;
  if ((K * W) % 128 != 0 || !al16(p.conv_state) || (p.conv_slot_stride * 2) % 16 != 0 || !al16(p.conv_weight)) return;
  const cuuint64_t groups = mode == 1 ? 4 : 3;
  {
    const cuuint64_t dims[3] = {HK, groups, T};
    const cuuint64_t strides[2] = {HK * 2, static_cast<cuuint64_t>(p.qkv_stride) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(K), static_cast<cuuint32_t>(groups), static_cast<cuuint32_t>(Q)};
    if (!encode_map(&p.tm_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.mixed_qkv, dims, strides, box)) return;
  }
  if (mode == 2) {
    const cuuint64_t dims[2] = {HK, T};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.gate_stride) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(K), static_cast<cuuint32_t>(Q)};
    if (!encode_map(&p.tm_gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.raw_gate, dims, strides, box)) return;
  }
  const cuuint64_t slots = static_cast<cuuint64_t>(p.num_slots);
  if (p.conv_dim_first) {
    const cuuint64_t dims[4] = {128, HK * Lc / 128, 3, slots};
    const cuuint64_t strides[3] = {256, HK * Lc * 2, static_cast<cuuint64_t>(p.conv_slot_stride) * 2};
    const cuuint32_t box[4] = {128, static_cast<cuuint32_t>(K * Lc / 128), 3, 1};
    if (!encode_map(&p.tm_conv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.conv_state, dims, strides, box)) return;
  } else {
    const cuuint64_t dims[4] = {HK, 3, Lc, slots};
    const cuuint64_t strides[3] = {HK * 2, 3 * HK * 2, static_cast<cuuint64_t>(p.conv_slot_stride) * 2};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(K), 3, static_cast<cuuint32_t>(Lc), 1};
    if (!encode_map(&p.tm_conv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.conv_state, dims, strides, box)) return;
  }
  {
    const cuuint64_t dims[3] = {128, HK * W / 128, 3};
    const cuuint64_t strides[2] = {128 * wb, HK * W * wb};
    const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(K * W / 128), 3};
    const CUtensorMapDataType dt = p.conv_weight_fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!encode_map(&p.tm_w, dt, 3, p.conv_weight, dims, strides, box)) return;
  }
  p.act_mode = mode;
}

// Which verify runs the products at K = 128.  An M = 128 tf32 MMA costs about
// the same whatever N is, and fp32 accuracy takes a second (low-part) pass,
// so the tensor cores win only when the window brings many operand vectors:
// measured on GB300, the tcgen05 verify is faster for windows of 8 (C3) and
// slower for windows of 4 (C2), so that is the default split.
// KDA_VERIFY_TCGEN05=1 forces the tensor cores, =0 the CUDA-core gemv.
bool use_tcgen05(bool window_up_to_4) {
  const char* v = std::getenv("KDA_VERIFY_TCGEN05");
  if (v != nullptr && v[0] == '1' && v[1] == '\0') return true;
  if (v != nullptr && v[0] == '0' && v[1] == '\0') return false;
  return !window_up_to_4;
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

template <int KD, int QMAX, bool DF, int VAR>
cudaError_t launch(const VerifyParams& p, cudaStream_t stream) {
  constexpr int bytes = Layout<KD, QMAX, VAR>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<KD, QMAX, DF, VAR>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const int items = p.B * p.H;
  const int grid = items < sm_count() ? items : sm_count();
  verify_kernel<KD, QMAX, DF, VAR><<<grid, Layout<KD, QMAX, VAR>::kThreads, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& params, int K, cudaStream_t stream) {
  VerifyParams p = params;
  build_tensor_maps(p, K);
  // the conv-state layout is a template parameter: straight-line tap addressing
  const bool q4 = p.Q <= 4;
  if (p.fold_qsl != nullptr) {  // the host accepts the fold for windows up to 4 only
    if (!q4) return cudaErrorInvalidValue;
    if (K == 128) return p.conv_dim_first ? launch<128, 4, true, kVarFold>(p, stream) : launch<128, 4, false, kVarFold>(p, stream);
    return p.conv_dim_first ? launch<64, 4, true, kVarFold>(p, stream) : launch<64, 4, false, kVarFold>(p, stream);
  }
  if (K == 128 && use_tcgen05(q4) && build_state_map(p, K)) {
    if (q4) return p.conv_dim_first ? launch<128, 4, true, kVarTcgen05>(p, stream) : launch<128, 4, false, kVarTcgen05>(p, stream);
    return p.conv_dim_first ? launch<128, 8, true, kVarTcgen05>(p, stream) : launch<128, 8, false, kVarTcgen05>(p, stream);
  }
  if (p.conv_dim_first) {
    if (K == 128) return q4 ? launch<128, 4, true, kVarPlain>(p, stream) : launch<128, 8, true, kVarPlain>(p, stream);
    return q4 ? launch<64, 4, true, kVarPlain>(p, stream) : launch<64, 8, true, kVarPlain>(p, stream);
  }
  if (K == 128) return q4 ? launch<128, 4, false, kVarPlain>(p, stream) : launch<128, 8, false, kVarPlain>(p, stream);
  return q4 ? launch<64, 4, false, kVarPlain>(p, stream) : launch<64, 8, false, kVarPlain>(p, stream);
}

}  // namespace kda
