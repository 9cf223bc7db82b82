// kda_verify.cu -- the KDA RecoverSSM speculative verify for sm_103a.
//
// Computes what "vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py"
// (_kda_recoverssm_verify_kernel with _kda_recurrent_step and _kda_gate)
// computes, with the short causal conv of
// "vllm.models.kimi_k3.nvidia.recoverssm.kernels" (CuteRecoverSSMVerify:
// rolled conv state of Q + W - 2 taps) in front.  Two launches per layer:
//   conv_kernel    one CTA per (request, head): the conv + SiLU codes of the
//                  head's q, k and v channels, correctly rounded to bf16, and
//                  the rolled conv state; the codes go, with the raw gate
//                  rows, the beta gates and the key channels' decays e^g,
//                  into the item's block of the caller's scratch;
//   verify_kernel  the verify proper, below, launched as the conv pass's
//                  programmatic dependent: its CTAs set up and stream state
//                  while the conv pass drains, and wait for it before the
//                  first read of the scratch.
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
// Schedule of the verify kernel.  One persistent CTA per SM takes
// (request, head) items from a ticket counter until none are left (the
// schedule, at the inputs warp) and works them with four roles that meet
// only at mbarrier rings in shared memory, so the stages of consecutive items
// overlap:
//   inputs (1 warp)  draws the tickets, decodes each item's request metadata
//                    a few items ahead (a ring of headers, which the state
//                    warp follows) and copies each item's rows of the conv
//                    pass's block (q | v, k | gate, the beta gates and the
//                    decays; the fold variant adds the head's dt_bias and
//                    the pending records) into a ring of small slots (bulk
//                    copies);
//   state (1 warp)   streams each live item's 64 KB fp32 state as eight row
//                    chunks into a ring of chunk slots, running ahead of the
//                    arithmetic by two to three items, and records the lap it
//                    arms in each slot;
//   prep (4 warps)   one key channel per thread: the key / gate record (one
//                    bulk store of the block's k | gate rows), the norms and
//                    the closed-form operands X_t, Y_t, M, N, handed on
//                    through a ring of operand slots;
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

#include <atomic>
#include <mutex>

#include "kda_device.cuh"

namespace kda {

namespace {

constexpr int kConvWidth = 4;
constexpr int kPrepWarps = 4;  // one key channel per thread
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
// default for windows of 8; kda_verify_args.variant chooses), and the
// CUDA-core verify that first folds each request's pending records of the
// previous step into its checkpoint.
enum : int { kVarPlain = 0, kVarTcgen05 = 1, kVarFold = 2 };

// Item flags.  kEnd marks the end of a CTA's item sequence: the tickets ran out.
enum : int { kLive = 1, kNull = 2, kEnd = 4 };

// Inputs warp -> state warp (ticket ring) and -> prep (small slot header),
// per item: the decoded request metadata of item `item` = b H + h.
template <int QMAX>
struct SmallMeta {
  int flags, item, bos, n, a;
  int fold_m;  // fold variant: pending records to fold, and their row
  long long s, r, fold_r;
  float A;
  int h;  // the item's head
};

// Prep -> gemv, per item (head of an operand slot).
template <int QMAX>
struct OpMeta {
  int flags, bos, n, h;
  long long r;
  float beta[QMAX];
  int fold_m, pad2;   // fold variant: pending records folded into the chunk,
  long long s;        // the slot the folded state goes back to,
  float rkf[QMAX];    // and 1 / |k_u| (with the eps) of each pending key
};

template <int KD, int QMAX, int VAR>
struct Layout {
  // Tensor-core instantiation (K = 128, windows of 4 or 8 tokens): the state
  // streams as K-slices of 32 (128 rows x 128 bytes, 128-byte swizzle) and the
  // products S0 [X | Y] come from tcgen05 MMAs; otherwise CUDA-core gemv warps.
  static_assert(VAR != kVarTcgen05 || (KD == 128 && (QMAX == 4 || QMAX == 8)), "the tensor-core path covers K = 128");
  static_assert(QMAX * 4 <= kScratchBetaBytes, "the block's beta area holds a window");
  static constexpr bool kTC = VAR == kVarTcgen05;
  static constexpr bool kFold = VAR == kVarFold;
  static constexpr int kThreads = 32 * (kTC ? kMmaWarp + 1 : 2 + kPrepWarps + kGemvWarps);
  static constexpr int RW = KD / kGemvWarps;  // state rows per gemv warp (one chunk)
  static constexpr int kChunk = kTC ? 128 * 32 * 4 : RW * KD * 4;  // bytes per state unit (chunk or K-slice)
  static constexpr int kNumSmall = QMAX <= 4 ? 3 : 2;  // small-input ring
  // ticket ring (inputs warp -> state warp): the inputs warp keeps kLead
  // items drawn and decoded ahead of its copies, in batches of up to
  // kMaxBatch; an entry is free again once both producer warps have read it
  static constexpr int kLead = 3;
  static constexpr int kMaxBatch = 8;
  static constexpr int kTick = 16;
  static constexpr int kTickBytes = ru(int(sizeof(SmallMeta<QMAX>)), 16);
  // small slot: the item's rows of the conv pass's block (q | v rows, then
  // k | gate rows, [QMAX][2K] bf16 each) and its head's dt_bias
  static constexpr int kQV = ru(int(sizeof(SmallMeta<QMAX>)), 128);
  static constexpr int kKG = kQV + QMAX * 2 * KD * 2;
  static constexpr int kDt = kKG + QMAX * 2 * KD * 2;                  // [KD] dt_bias
  static constexpr int kBeta = kDt + KD * 4;  // [8] fp32 sigmoid(raw beta), from the conv pass's block
  static constexpr int kBetaBytes = kScratchBetaBytes;
  static constexpr int kEg = kBeta + kBetaBytes;  // [QMAX][KD] fp32 decays e^g, from the conv pass's block
  // fold variant: the pending records of the item, [QMAX][2K] bf16 key/gate
  // and [QMAX][V] fp32 corrections (V == K)
  static constexpr int kFoldKg = ru(kEg + QMAX * KD * 4, 128);
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
  // prep runs up to three items ahead of the gemv team (windows up to 4:
  // measured on C2, 4 slots 0.171 ms per call against 0.180 with 3, no gain
  // from 5 or 6); on the tensor-core path an item's slot is also held until
  // its readout, one item later
  static constexpr int kNumOp = kTC ? (QMAX <= 4 ? 4 : 3) : QMAX <= 4 ? 4 : 2;
  // per-warp scratch
  static constexpr int kRedPerWarp = kTC ? 0 : 2 * QMAX * RW;         // floats
  static constexpr int kFoldIdx = 2 * QMAX + QMAX * QMAX;  // fold variant: |k_u|^2 of the pending keys
  static constexpr int kPart = ru(kFoldIdx + (kFold ? QMAX : 0), 32);         // reduced values per prep warp
  static constexpr int kFixed = kNumSmall * kSmall + kNumOp * kOp + kGemvWarps * kRedPerWarp * 4 +
                                kPrepWarps * kPart * 4 + 32 + 64 + 64 + kTick * kTickBytes +
                                (2 * kNumSmall + 2 * kNumOp + 4 + 2 * kTick) * 8 + (kTC ? 1024 : 0);
  static constexpr int kBarsPerChunk = kTC ? 4 : 2;
  static constexpr int kChunkFit = (kSmemLimit - kFixed - 64 * kBarsPerChunk * 8) / kChunk;
  static constexpr int kNumChunk = kChunkFit > 64 ? 64 : kChunkFit;
  // CTA layout
  static constexpr int oChunks = 0;
  static constexpr int oSmall = oChunks + kNumChunk * kChunk;
  static constexpr int oOp = ru(oSmall + kNumSmall * kSmall, kTC ? 1024 : 128);
  static constexpr int oRed = oOp + kNumOp * kOp;
  static constexpr int oPart = oRed + kGemvWarps * kRedPerWarp * 4;
  static constexpr int oMisc = oPart + kPrepWarps * kPart * 4;  // int[8]
  static constexpr int oArm = oMisc + 32;                      // uint8[64]: last armed phase per chunk slot
  static constexpr int oLap = oArm + 64;                        // uint8[64]: lap last armed per chunk slot
  static constexpr int oTick = ru(oLap + 64, 16);               // SmallMeta[kTick]: the ticket ring
  static constexpr int oBars = ru(oTick + kTick * kTickBytes, 8);
  static constexpr int kNumBars = kBarsPerChunk * kNumChunk + 2 * kNumSmall + 2 * kNumOp + 4 + 2 * kTick;
  static constexpr int kBytes = oBars + kNumBars * 8;
  static_assert(kBytes <= kSmemLimit, "shared memory budget");
  // at least six K-slices (tensor cores), 1.5 items of chunks (fold variant,
  // whose slots carry the pending records) or two items of chunks in flight
  static_assert(kNumChunk >= (kTC ? 6 : kFold ? 3 * kGemvWarps / 2 : 2 * kGemvWarps), "state in flight");
  static_assert(kNumChunk <= 64, "one record of the last armed phase per chunk slot");
  static_assert(kTick >= kLead + kMaxBatch + 1, "the ticket ring holds the drawer's lead and a batch");
  static_assert(kMaxBatch <= 32, "one lane per item of a batch");
};

template <int KD, int QMAX, int VAR>
struct Bars {
  uint64_t *ch_full, *ch_empty, *sm_full, *sm_empty, *op_full, *op_empty, *d_full, *d_empty, *hi_done, *lo_full;
  uint64_t *tk_full, *tk_empty;
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
    tk_full = d_empty + 2;             // [kTick]
    tk_empty = tk_full + Lay::kTick;   // [kTick]
    hi_done = tk_empty + Lay::kTick;   // [kNumChunk] tensor-core path
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
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane, const volatile int* abort_flag,
                                          uint64_t limit_ns) {
  bool ok = true;
  if (lane == 0) ok = mbar_wait_or_abort(bar, parity, abort_flag, limit_ns);
  ok = __all_sync(0xffffffffu, ok);
  if (ok && lane != 0) mbar_acquire_seen(bar, parity);
  return ok;
}

// warp_wait for a chunk of the state ring, seen by a gemv warp.  A gemv
// warp takes every eighth chunk and may run up to three items (24 chunks)
// ahead of another, so it can come to a chunk slot one lap ahead of a copy
// still in flight there; the parity alone would then match the slot's
// previous, completed phase.  The state warp records in `lap` the lap it
// arms in each slot, only once the slot's previous lap has been consumed:
// lane 0 first waits (bounded, with a short sleep per poll) for the slot to
// show this warp's lap, after which the parity names a single phase.
__device__ __forceinline__ bool warp_wait_chunk(uint64_t* bar, const unsigned char* lap_base, int pos, uint32_t lap_no,
                                                int lane, const volatile int* abort_flag, uint64_t limit_ns) {
  const uint32_t parity = lap_no & 1;
  bool ok = true;
  if (lane == 0) {
    const volatile uint8_t* lap = reinterpret_cast<const volatile uint8_t*>(lap_base);
    const uint8_t want = static_cast<uint8_t>(lap_no);
    // (an iteration bound: each poll sleeps at most about 128 ns, so the
    // bound is a couple of seconds at most)
    for (uint32_t it = 0; ok && lap[pos] != want; ++it) {
      if (*abort_flag || it >= (1u << 24)) ok = false;
      else __nanosleep(64);
    }
    if (ok) ok = mbar_wait_or_abort(bar, parity, abort_flag, limit_ns);
  }
  ok = __all_sync(0xffffffffu, ok);
  if (ok && lane != 0) mbar_acquire_seen(bar, parity);
  return ok;
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

// The raw request values an item's metadata is made of: one round of
// independent loads (it < 0: none).
struct ItemLoads {
  int it, q0, q1, si, ri, nap, fq0, fq1, fna, fri;
  float alog;
};

__device__ __forceinline__ ItemLoads load_item(const VerifyParams& p, int it) {
  ItemLoads l{it, 0, 0, 0, 0, 1, 0, 0, 0, 0, 0.0f};
  if (it < 0) return l;
  const int b = it / p.H;
  l.q0 = p.qsl[b];
  l.q1 = p.qsl[b + 1];
  l.si = p.state_indices[b];
  l.ri = p.record_indices ? p.record_indices[b] : l.si;
  l.nap = p.num_accepted_prev ? p.num_accepted_prev[b] : 1;
  if (p.fold_qsl != nullptr) {
    l.fq0 = p.fold_qsl[b];
    l.fq1 = p.fold_qsl[b + 1];
    l.fna = p.fold_num_accepted[b];
    l.fri = p.fold_record_indices ? p.fold_record_indices[b] : l.si;
  }
  l.alog = p.A_log[it - b * p.H];
  return l;
}

template <int QMAX>
__device__ __forceinline__ ItemMeta<QMAX> item_meta(const VerifyParams& p, const ItemLoads& l, bool report_errors) {
  ItemMeta<QMAX> m{0, 0, 0, 0, 1, 0, 0, 0, 0};
  if (l.it < 0) return m;
  const int it = l.it;
  const int b = it / p.H;
  m.h = it - b * p.H;
  m.bos = l.q0;
  const int len = l.q1 - m.bos;
  m.s = l.si;
  m.r = l.ri;
  m.a = min(max(l.nap, 1), p.Q);
  m.n = min(max(len, 0), p.Q);
  if (p.fold_qsl != nullptr) {  // the previous step's pending records, folded first
    const int plen = l.fq1 - l.fq0;
    m.fold_m = min(max(l.fna, 0), min(max(plen, 0), p.Q));
    m.fold_r = l.fri;
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

// ---------------------------------------------------------------- conv pass
//
// The short causal conv in front of the verify, as its own launch: one CTA
// per (request, head) item, 3K/2 threads, each on two adjacent channels of
// one of the head's q, k and v groups.  Per channel it reads the W - 1 stored
// taps from tap a - 1 and the window's inputs, evaluates the bf16 codes of
// SiLU(conv) (tier 1 of kda_device.cuh, both channels of the pair at once;
// the rare codes it leaves in doubt go to the exact tiers, out of line), and
// rolls the conv state in place (taps 0 .. W-3+n <- seq[1 .. W-2+n], later
// taps untouched).  The codes go, with the raw gate rows, into the item's
// block of the caller's scratch: [Q][2K] bf16 rows q | v, then [Q][2K] rows
// k | raw gate, rows t < n written, then the window's beta gates
// sigmoid(raw beta) and the key channels' decays e^g, in fp32.  The k | gate
// rows are the item's key / gate record verbatim.  Null items, empty windows and items with bad metadata are
// skipped here; the verify kernel reports the latter.
//
// A pair's values travel as 32-bit words, channel c in the low half and
// c + 1 in the high half: that is the layout of the activations, the seq-first
// conv state and the scratch rows, so a pair costs one access where the rows
// allow it (an even stride from a 4-byte aligned start, checked once per
// launch; two 16-bit accesses otherwise).

__device__ __forceinline__ float lo_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two adjacent bf16 values from a row; w32: the pair sits on 4 bytes.
__device__ __forceinline__ uint32_t load_pair(const uint16_t* ptr, bool w32) {
  if (w32) return __ldg(reinterpret_cast<const unsigned int*>(ptr));
  return static_cast<uint32_t>(__ldg(ptr)) | (static_cast<uint32_t>(__ldg(ptr + 1)) << 16);
}

__device__ __forceinline__ void store_pair(uint16_t* ptr, uint32_t v, bool w32) {
  if (w32) {
    *reinterpret_cast<uint32_t*>(ptr) = v;
  } else {
    ptr[0] = static_cast<uint16_t>(v & 0xffffu);
    ptr[1] = static_cast<uint16_t>(v >> 16);
  }
}

// The codes of one channel pair: sq[j] holds both channels' sequence value j
// (the W - 1 taps, then the window); y[t] the two codes of token t.
template <int QMAX, bool W32>
__device__ __forceinline__ void pair_codes(const float (&wa)[kConvWidth], const float (&wb)[kConvWidth],
                                           const uint32_t (&sq)[kConvWidth - 1 + QMAX], int n, uint32_t (&y)[QMAX]) {
  uint32_t doubt = 0;
#pragma unroll
  for (int t = 0; t < QMAX; ++t) {
    y[t] = 0;
    if (t < n) {
      const float xa[kConvWidth] = {lo_f32(sq[t]), lo_f32(sq[t + 1]), lo_f32(sq[t + 2]), lo_f32(sq[t + 3])};
      const float xb[kConvWidth] = {hi_f32(sq[t]), hi_f32(sq[t + 1]), hi_f32(sq[t + 2]), hi_f32(sq[t + 3])};
      uint32_t d;
      y[t] = conv_silu_bf16x2<W32>(wa, wb, xa, xb, &d);
      doubt |= d << (2 * t);
    }
  }
  if (doubt) {  // a few codes in 10^4
#pragma unroll
    for (int t = 0; t < QMAX; ++t) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if ((doubt >> (2 * t + half)) & 1u) {
          const int sh = 16 * half;
          const float* w = half ? wb : wa;
          const uint32_t code = static_cast<uint32_t>(exact_conv::conv_code_exact(
              w[0], w[1], w[2], w[3], bf16_to_f32((sq[t] >> sh) & 0xffffu), bf16_to_f32((sq[t + 1] >> sh) & 0xffffu),
              bf16_to_f32((sq[t + 2] >> sh) & 0xffffu), bf16_to_f32((sq[t + 3] >> sh) & 0xffffu)));
          y[t] = (y[t] & (0xffff0000u >> sh)) | (code << sh);
        }
      }
    }
  }
}

// Seven CTAs per SM (42 warps, eleven on some scheduler: 40 registers, a few
// spilled): the pass is latency-bound, and more CTAs in flight measured
// faster than five without spills (eight also get 40 and measured slower).
// DF: dim-first conv state; W32: fp32 conv weights (else bf16).
template <int KD, int QMAX, bool DF, bool W32>
__global__ void __launch_bounds__(3 * KD / 2, 7) conv_kernel(const __grid_constant__ VerifyParams p) {
  // The verify kernel may start now: it waits for this grid before it reads
  // the scratch, and its other work (state streaming) does not depend on it.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Two dependent memory round trips: the item's metadata with the pair's
  // weights, then every tap, input and gate value of the window; then the
  // codes and the stores.  Groups (q, k, v) are K/2 threads: whole warps.
  const int it = static_cast<int>(blockIdx.x);
  const int g = (2 * static_cast<int>(threadIdx.x)) / KD;  // 0: q, 1: k, 2: v
  const int k = 2 * static_cast<int>(threadIdx.x) - g * KD;
  const int h = it - (it / p.H) * p.H;
  const long long HK = static_cast<long long>(p.H) * KD;
  const long long c = g * HK + static_cast<long long>(h) * KD + k;  // the pair's first channel (even)
  // the item's metadata, decoded once by the first warp and shared
  __shared__ int s_meta[6];
  if (threadIdx.x < 32) {
    const ItemMeta<QMAX> m0 = item_meta<QMAX>(p, load_item(p, it), false);
    if (threadIdx.x == 0) {
      s_meta[0] = (m0.flags & kLive) ? m0.n : 0;
      s_meta[1] = m0.a;
      s_meta[2] = m0.bos;
      s_meta[3] = static_cast<int>(m0.s);
      s_meta[4] = static_cast<int>(m0.s >> 32);
    }
  }
  float wa[kConvWidth], wb[kConvWidth];
  if (W32) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p.conv_weight) + c);
    const float4 b = __ldg(reinterpret_cast<const float4*>(p.conv_weight) + c + 1);
    wa[0] = a.x; wa[1] = a.y; wa[2] = a.z; wa[3] = a.w;
    wb[0] = b.x; wb[1] = b.y; wb[2] = b.z; wb[3] = b.w;
  } else {
    const uint4 wv = __ldg(reinterpret_cast<const uint4*>(p.conv_weight) + c / 2);
    wa[0] = lo_f32(wv.x); wa[1] = hi_f32(wv.x); wa[2] = lo_f32(wv.y); wa[3] = hi_f32(wv.y);
    wb[0] = lo_f32(wv.z); wb[1] = hi_f32(wv.z); wb[2] = lo_f32(wv.w); wb[3] = hi_f32(wv.w);
  }
  __syncthreads();
  const int n = s_meta[0];  // 0: nothing to convolve (a null, empty or bad item)
  if (n <= 0) return;
  struct {
    int a, bos;
    long long s;
  } im;
  im.a = s_meta[1];
  im.bos = s_meta[2];
  im.s = static_cast<long long>(static_cast<uint32_t>(s_meta[3])) | (static_cast<long long>(s_meta[4]) << 32);
  const int Lc = p.Q + kConvWidth - 2;
  const bool x32 = (p.qkv_stride & 1) == 0 && (reinterpret_cast<uintptr_t>(p.mixed_qkv) & 3u) == 0;
  const bool g32 = (p.gate_stride & 1) == 0 && (reinterpret_cast<uintptr_t>(p.raw_gate) & 3u) == 0;
  uint16_t* cs = p.conv_state + im.s * p.conv_slot_stride;
  const uint16_t* x = p.mixed_qkv + static_cast<long long>(im.bos) * p.qkv_stride + c;
  // sq[j]: the W - 1 stored taps from tap a - 1, then the window (zero past n)
  uint32_t sq[kConvWidth - 1 + QMAX];
  uint32_t gate[QMAX];
#pragma unroll
  for (int j = 0; j < kConvWidth - 1; ++j) {
    if (DF) {  // rows of Lc taps per channel: the pair's taps are Lc apart
      const uint16_t* r = cs + c * Lc + im.a - 1 + j;
      sq[j] = static_cast<uint32_t>(r[0]) | (static_cast<uint32_t>(r[Lc]) << 16);
    } else {  // the slot is 16-byte aligned and rows are 3HK (even) wide
      sq[j] = *reinterpret_cast<const uint32_t*>(cs + static_cast<long long>(im.a - 1 + j) * 3 * HK + c);
    }
  }
#pragma unroll
  for (int t = 0; t < QMAX; ++t) sq[kConvWidth - 1 + t] = t < n ? load_pair(x + t * p.qkv_stride, x32) : 0u;
  if (g == 1) {
    const uint16_t* gr = p.raw_gate + static_cast<long long>(im.bos) * p.gate_stride + h * KD + k;
#pragma unroll
    for (int t = 0; t < QMAX; ++t) gate[t] = t < n ? load_pair(gr + t * p.gate_stride, g32) : 0u;
  }
  // the key group: both channels' dt_bias and the head's A = e^A_log, for the decays
  float2 dtb = make_float2(0.0f, 0.0f);
  float A = 0.0f;
  if (g == 1) {
    dtb = __ldg(reinterpret_cast<const float2*>(p.dt_bias + static_cast<long long>(h) * KD + k));
    A = expf(p.A_log[h]);
  }
  // thread t < n of the q group: the gate sigmoid(raw beta) of token t
  const int tb = static_cast<int>(threadIdx.x);
  const uint16_t rbeta = tb < n ? p.raw_beta[static_cast<long long>(im.bos + tb) * p.beta_stride + h] : uint16_t(0);
  // the codes: a bf16 weight times a bf16 input is exact in fp32; an fp32 weight's product rounds
  uint32_t y[QMAX];
  pair_codes<QMAX, W32>(wa, wb, sq, n, y);
  // the item's block: q at [t][k], v at [t][K + k], k at [Q + t][k], gate at [Q + t][K + k]
  uint16_t* blk = p.scratch + static_cast<long long>(it) * scratch_item_elems(p.Q, KD) + k;
  uint16_t* dst = g == 0 ? blk : g == 2 ? blk + KD : blk + 2LL * p.Q * KD;
#pragma unroll
  for (int t = 0; t < QMAX; ++t)
    if (t < n) *reinterpret_cast<uint32_t*>(dst + t * 2 * KD) = y[t];
  if (g == 1) {
    // the gate record, and the decays e^g of both channels for the verify
    float* egb = reinterpret_cast<float*>(p.scratch + static_cast<long long>(it) * scratch_item_elems(p.Q, KD) +
                                          scratch_eg_elem(p.Q, KD)) + k;
#pragma unroll
    for (int t = 0; t < QMAX; ++t) {
      if (t < n) {
        *reinterpret_cast<uint32_t*>(dst + t * 2 * KD + KD) = gate[t];
        const float ea = kda_decay_fast(lo_f32(gate[t]), dtb.x, A, p.lower_bound_gate, p.lower_bound);
        const float eb = kda_decay_fast(hi_f32(gate[t]), dtb.y, A, p.lower_bound_gate, p.lower_bound);
        *reinterpret_cast<float2*>(egb + t * KD) = make_float2(ea, eb);
      }
    }
  }
  if (tb < n)
    reinterpret_cast<float*>(p.scratch + static_cast<long long>(it) * scratch_item_elems(p.Q, KD) + 4LL * p.Q * KD)[tb] =
        sigmoid_fast(bf16_to_f32(rbeta));
  // the rolled taps: 0 .. W-3+n <- seq[1 .. W-2+n], later taps untouched
  if (DF) {
    // rows c and c + 1 start Lc apart; c Lc is even, so row c takes 32-bit
    // stores of tap pairs, and row c + 1 too when Lc is even
    uint16_t* r0 = cs + c * Lc;
    uint16_t* r1 = r0 + Lc;
    const bool l32 = (Lc & 1) == 0;
#pragma unroll
    for (int j = 0; j < kConvWidth - 2 + QMAX; j += 2) {
      if (j + 1 < kConvWidth - 2 + n) {
        store_pair(r0 + j, __byte_perm(sq[j + 1], sq[j + 2], 0x5410), true);
        store_pair(r1 + j, __byte_perm(sq[j + 1], sq[j + 2], 0x7632), l32);
      } else if (j < kConvWidth - 2 + n) {
        r0[j] = static_cast<uint16_t>(sq[j + 1] & 0xffffu);
        r1[j] = static_cast<uint16_t>(sq[j + 1] >> 16);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kConvWidth - 2 + QMAX; ++j)
      if (j < kConvWidth - 2 + n) *reinterpret_cast<uint32_t*>(cs + static_cast<long long>(j) * 3 * HK + c) = sq[j + 1];
  }
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

// The schedule.  Items are dealt out at run time from a ticket counter in the
// workspace: the inputs warp of each CTA takes the next item number with one
// atomic, until the numbers run out, so a CTA that starts late (behind the
// conv pass) or runs slow takes fewer items and the CTAs finish within about
// an item of each other.  The last CTA to finish zeroes the counter for the
// next launch (end of verify_kernel).
//
// The inputs warp draws and decodes kLead items ahead of its copies and puts
// each item's header into the ticket ring, from which the state warp takes
// its items (no metadata loads of its own) and from which the header later
// goes into the item's small slot for the prep team.  After the last item,
// an entry with item -1 ends the state warp's sequence and a header flagged
// kEnd ends the prep team's, which forwards it to the gemv team.

// The header of an item from its loads (item -1: none, the end mark); the
// lane that decodes an item reports its metadata errors.
template <int QMAX>
__device__ __forceinline__ SmallMeta<QMAX> item_header(const VerifyParams& p, const ItemLoads& l) {
  SmallMeta<QMAX> m;
  const ItemMeta<QMAX> im = item_meta<QMAX>(p, l, l.it >= 0);
  m.flags = l.it >= 0 ? im.flags : kEnd;
  m.item = l.it;
  m.bos = im.bos;
  m.n = im.n;
  m.a = im.a;
  m.fold_m = im.fold_m;
  m.s = im.s;
  m.r = im.r;
  m.fold_r = im.fold_r;
  m.A = l.it >= 0 ? expf(l.alog) : 0.0f;
  m.h = im.h;
  return m;
}

template <int KD, int QMAX, int VAR>
__device__ void produce_inputs(const VerifyParams& p, unsigned char* smem, int lane, volatile int* misc) {
  using Lay = Layout<KD, QMAX, VAR>;
  using Meta = SmallMeta<QMAX>;
  Bars<KD, QMAX, VAR> bars(smem);
  volatile int* abort_flag = misc + kMiscAbort;
  unsigned char* ring = smem + Lay::oTick;
  const int items = p.B * p.H;
  const int grid = static_cast<int>(gridDim.x);
  int* counter = p.workspace + kWsTicket;
  bool ok = true;
  int drawn = 0;       // ring entries written
  bool ended = false;  // the entry with item -1 is written
  int seen = 0;        // the counter's value at this CTA's last draw
  // One draw: a batch of consecutive tickets sized from what is left (about
  // a half of this CTA's fair share of the rest, at least one and at most
  // kMaxBatch), decoded one item per lane in one round of loads, and its
  // entries published; an empty draw publishes the end mark.  Large batches
  // early keep the decode's code and round trips rare; single tickets at
  // the end even out the CTAs' finish.
  auto draw = [&]() {
    int t0 = 0, k = 1;
    if (lane == 0) {
      k = min(max((items - seen) / (2 * grid), 1), Lay::kMaxBatch);
      t0 = atomicAdd(counter, k);
    }
    t0 = __shfl_sync(0xffffffffu, t0, 0);
    k = __shfl_sync(0xffffffffu, k, 0);
    seen = t0 + k;
    const int nb = t0 < items ? min(k, items - t0) : 0;
    const int count = nb > 0 ? nb : 1;
    // the entries' slots are free once the last of them is (readers go in order)
    const int last = drawn + count - 1;
    ok = warp_wait(&bars.tk_empty[last % Lay::kTick], ((last / Lay::kTick) & 1) ^ 1, lane, abort_flag,
                   p.wait_limit_ns);
    if (!ok) return;
    const int it = lane < nb ? t0 + lane : -1;
    const Meta m = item_header<QMAX>(p, load_item(p, it));
    if (lane < count) {
      const int e = (drawn + lane) % Lay::kTick;
      *reinterpret_cast<Meta*>(ring + e * Lay::kTickBytes) = m;
      mbar_arrive(&bars.tk_full[e]);
    }
    __syncwarp();
    drawn += count;
    ended = nb == 0;
  };
  // per small slot: whether this warp has armed a phase of its full barrier,
  // and that phase's parity (the copies behind it are waited for at exit)
  uint32_t armed = 0, armed_parity = 0;
  for (int i = 0; ok; ++i) {
    // at least kLead entries past this one are published (the first pass
    // fills the lead); drawn before the wait for the slot, which it overlaps
    // when the prep team is the slower side
    while (ok && !ended && drawn <= i + Lay::kLead) draw();
    // the conv pass's rows are read from here on (the headers so far come
    // from the caller's metadata, not from it); every CTA waits, so this
    // grid cannot complete before the conv pass has
    if (i == 0) wait_prior_grid();
    if (!ok) break;
    const int e = i % Lay::kTick;
    const Meta m = *reinterpret_cast<const Meta*>(reinterpret_cast<const unsigned char*>(ring) + e * Lay::kTickBytes);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.tk_empty[e]);
    const int slot = i % Lay::kNumSmall;
    ok = warp_wait(&bars.sm_empty[slot], ((i / Lay::kNumSmall) & 1) ^ 1, lane, abort_flag, p.wait_limit_ns);
    if (!ok) break;
    unsigned char* sl = smem + Lay::oSmall + slot * Lay::kSmall;
    // a phase armed here is the slot's last so far (the exit drain waits for
    // the last one; a later phase of the slot would alias its parity)
    auto arm = [&] {
      armed |= 1u << slot;
      armed_parity = (armed_parity & ~(1u << slot)) | (static_cast<uint32_t>((i / Lay::kNumSmall) & 1) << slot);
    };
    if (m.item < 0) {  // no items left: the prep team's end mark
      arm();
      if (lane == 0) {
        reinterpret_cast<Meta*>(sl)->flags = kEnd;
        mbar_arrive(&bars.sm_full[slot]);
      }
      break;
    }
    // kda_verify_debug: this item's inputs are withheld (no copy, no
    // arrival), so the prep team's bounded wait on them runs out
    if (m.item != p.withhold_item) {
      arm();
      if (lane == 0) {
        *reinterpret_cast<Meta*>(sl) = m;
        uint64_t* bar = &bars.sm_full[slot];
        if (m.flags & kLive) {
          // the item's rows of the conv pass's block (q | v, then k | gate),
          // its head's dt_bias and, in the fold variant, its pending records:
          // a few bulk copies
          const int h = m.h;
          const uint32_t rows = static_cast<uint32_t>(m.n) * 2 * KD * 2;
          const uint32_t fold_bytes = static_cast<uint32_t>(m.fold_m) * (2 * KD * 2 + KD * 4);
          const uint32_t egs = static_cast<uint32_t>(m.n) * KD * 4;
          const uint32_t dts = Lay::kFold ? KD * 4 : 0u;
          mbar_arrive_expect_tx(bar, (rows ? 2 * rows + Lay::kBetaBytes + egs : 0u) + dts + fold_bytes);
          if (fold_bytes) fold_copies<KD, QMAX, VAR>(p, sl, h, m.fold_m, m.fold_r, bar);
          if (rows) {  // (a fold-only item has no window)
            const uint16_t* blk = p.scratch + static_cast<long long>(m.item) * scratch_item_elems(p.Q, KD);
            bulk_g2s(sl + Lay::kQV, blk, rows, bar);
            bulk_g2s(sl + Lay::kKG, blk + 2LL * p.Q * KD, rows, bar);
            bulk_g2s(sl + Lay::kBeta, blk + 4LL * p.Q * KD, Lay::kBetaBytes, bar);
            bulk_g2s(sl + Lay::kEg, blk + scratch_eg_elem(p.Q, KD), egs, bar);
          }
          // the fold variant decodes the pending keys' decays with this layer's gate
          if (Lay::kFold) bulk_g2s(sl + Lay::kDt, p.dt_bias + static_cast<long long>(h) * KD, KD * 4, bar);
        } else {
          mbar_arrive(bar);
        }
      }
      __syncwarp();
    }
  }
  if (!ok && lane == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
  // no copy may land after the CTA is gone: wait (bounded) for the last armed
  // phase of every slot (a phase the prep team already consumed is complete)
  if (lane == 0) {
    for (int sl_i = 0; sl_i < Lay::kNumSmall; ++sl_i)
      if ((armed >> sl_i) & 1u) (void)mbar_wait_bounded(&bars.sm_full[sl_i], (armed_parity >> sl_i) & 1u, p.wait_limit_ns);
  }
}

// ---------------------------------------------------------------- state warp

// The next item of the state warp from the ticket ring: its header's flags,
// item number and state slot; false once the wait gave up.
template <int KD, int QMAX, int VAR>
__device__ __forceinline__ bool next_ticket(const VerifyParams& p, unsigned char* smem, int i, int lane,
                                            const volatile int* abort_flag, int& flags, int& item, long long& slot) {
  using Lay = Layout<KD, QMAX, VAR>;
  Bars<KD, QMAX, VAR> bars(smem);
  const int e = i % Lay::kTick;
  if (!warp_wait(&bars.tk_full[e], (i / Lay::kTick) & 1, lane, abort_flag, p.wait_limit_ns)) return false;
  const SmallMeta<QMAX>* m = reinterpret_cast<const SmallMeta<QMAX>*>(smem + Lay::oTick + e * Lay::kTickBytes);
  flags = m->flags;
  item = m->item;
  slot = m->s;
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars.tk_empty[e]);
  return true;
}

template <int KD, int QMAX, int VAR>
__device__ void produce_state(const VerifyParams& p, unsigned char* smem, int lane, volatile int* abort_flag) {
  using Lay = Layout<KD, QMAX, VAR>;
  Bars<KD, QMAX, VAR> bars(smem);
  uint32_t ch_cnt = 0;
  bool ok = true;
  // per chunk slot, the last armed phase: 0 never, 1 + its parity (shared
  // memory, written by the arming lane; waited for at exit)
  volatile uint8_t* arm = reinterpret_cast<volatile uint8_t*>(smem + Lay::oArm);
  volatile uint8_t* lap = reinterpret_cast<volatile uint8_t*>(smem + Lay::oLap);
  if (lane < Lay::kNumChunk) arm[lane] = 0;
  if (lane + 32 < Lay::kNumChunk) arm[lane + 32] = 0;
  __syncwarp();
  for (int i = 0; ok; ++i) {
    int flags, item;
    long long js;
    ok = next_ticket<KD, QMAX, VAR>(p, smem, i, lane, abort_flag, flags, item, js);
    if (!ok || item < 0) break;
    if (!(flags & kLive)) continue;
    const int jh = item - (item / p.H) * p.H;
    // lane c streams row chunk c into the next free chunk slot
    if (lane < kGemvWarps) {
      const uint32_t cc = ch_cnt + lane;
      const int pos = cc % Lay::kNumChunk;
      ok = mbar_wait_or_abort(&bars.ch_empty[pos], ((cc / Lay::kNumChunk) & 1) ^ 1, abort_flag, p.wait_limit_ns);
      if (ok) {
        arm[pos] = static_cast<uint8_t>(1 + ((cc / Lay::kNumChunk) & 1));
        lap[pos] = static_cast<uint8_t>(cc / Lay::kNumChunk);  // before the phase is armed
        const float* src = p.state + js * p.state_slot_stride + static_cast<long long>(jh) * KD * KD;
        mbar_arrive_expect_tx(&bars.ch_full[pos], Lay::kChunk);
        bulk_g2s(smem + Lay::oChunks + pos * Lay::kChunk, src + lane * Lay::RW * KD, Lay::kChunk,
                 &bars.ch_full[pos]);
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    ch_cnt += kGemvWarps;
  }
  if (!ok && lane == 0) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
  // no copy may land after the CTA is gone: wait (bounded) for the last
  // armed phase of every chunk slot (complete once its copy has landed)
  __syncwarp();
  if (lane == 0) {
    for (int pos = 0; pos < Lay::kNumChunk; ++pos)
      if (arm[pos]) (void)mbar_wait_bounded(&bars.ch_full[pos], arm[pos] - 1u, p.wait_limit_ns);
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

// Plan of a warp sum of N values per lane: H reduce-scatter stages over lane
// bits 16, 8, ... (each halves the count and costs 2 x the count in
// instructions: two selects, a shuffle and an add per pair), then an
// all-reduce of the C = N / 2^H values left over the 5 - H low lane bits
// (2 instructions per value and bit).  N is first padded to P (a multiple of
// 2^H); the cheapest (P, H) is taken.  Afterwards lane l holds the totals of
// values [C (l >> (5 - H)), + C).
template <int N>
struct WarpSumPlan {
  static constexpr int cost(int p, int h) {
    int c = 0, w = p;
    for (int i = 0; i < h; ++i) { c += 2 * w; w /= 2; }
    return c + 2 * w * (5 - h);
  }
  static constexpr int best_h() {
    int bh = 5, bc = cost(ru(N, 32), 5);
    for (int h = 0; h <= 5; ++h) {
      const int c = cost(ru(N, 1 << h), h);
      if (c < bc) { bc = c; bh = h; }
    }
    return bh;
  }
  static constexpr int H = best_h();
  static constexpr int P = ru(N, 1 << H);
  static constexpr int C = P >> H;
};

template <int P, int H, int C>
__device__ __forceinline__ void warp_sum_values(float* vals, int lane) {
  if constexpr (H > 0) reduce_scatter_stage<P>(vals, 16, (lane & 16) != 0);
  if constexpr (H > 1) reduce_scatter_stage<P / 2>(vals, 8, (lane & 8) != 0);
  if constexpr (H > 2) reduce_scatter_stage<P / 4>(vals, 4, (lane & 4) != 0);
  if constexpr (H > 3) reduce_scatter_stage<P / 8>(vals, 2, (lane & 2) != 0);
  if constexpr (H > 4) reduce_scatter_stage<P / 16>(vals, 1, (lane & 1) != 0);
#pragma unroll
  for (int b = 0; b < 5 - H; ++b) {
#pragma unroll
    for (int i = 0; i < C; ++i) vals[i] += __shfl_xor_sync(0xffffffffu, vals[i], 1 << b);
  }
}

template <int KD, int QMAX, int VAR>
__device__ void prep(const VerifyParams& p, unsigned char* smem, int pt, volatile int* misc) {
  using Lay = Layout<KD, QMAX, VAR>;
  constexpr int NREDP = Lay::kPart;  // |q_t|^2, |k_t|^2, raw M / N grid (and the fold's norms), padded to 32
  // the warp sum over the key channels: only the values in use, by the
  // cheapest mix of reduce-scatter and all-reduce stages
  using Plan = WarpSumPlan<Lay::kFoldIdx + (Lay::kFold ? QMAX : 0)>;
  static_assert(Plan::P <= NREDP, "the summed values fit the per-warp parts");
  Bars<KD, QMAX, VAR> bars(smem);
  volatile int* abort_flag = misc + kMiscAbort;
  float* part = reinterpret_cast<float*>(smem + Lay::oPart);
  const int warp = pt >> 5;
  const int lane = pt & 31;
  for (int i = 0;; ++i) {
    const int slot = i % Lay::kNumSmall;
    const int oslot = i % Lay::kNumOp;
    unsigned char* sl = smem + Lay::oSmall + slot * Lay::kSmall;
    unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
    const bool ok = warp_wait(&bars.sm_full[slot], (i / Lay::kNumSmall) & 1, lane, abort_flag, p.wait_limit_ns) &&
                    warp_wait(&bars.op_empty[oslot], ((i / Lay::kNumOp) & 1) ^ 1, lane, abort_flag, p.wait_limit_ns);
    if (!ok && lane == 0) misc[kMiscPrepFail] = 1;
    const SmallMeta<QMAX> m = *reinterpret_cast<const SmallMeta<QMAX>*>(sl);
    if (ok && (m.flags & kEnd)) {  // every prep thread reads the same mark: hand it on, stop
      if (pt == 0) {
        reinterpret_cast<OpMeta<QMAX>*>(op + Lay::kOpMeta)->flags = kEnd;
        mbar_arrive(&bars.op_full[oslot]);
      }
      break;
    }
    const int h = m.h;
    const bool live = ok && (m.flags & kLive);
    const int n = m.n;
    // the window's beta gates, for the operand header (read before the slot
    // is released)
    float beta[QMAX];
#pragma unroll
    for (int t = 0; t < QMAX; ++t)
      beta[t] = (pt == 0 && live && t < n) ? reinterpret_cast<const float*>(sl + Lay::kBeta)[t] : 0.0f;
    const uint16_t* qv_rows = reinterpret_cast<const uint16_t*>(sl + Lay::kQV);  // [QMAX][2K] q | v
    const uint16_t* kg_rows = reinterpret_cast<const uint16_t*>(sl + Lay::kKG);  // [QMAX][2K] k | gate

    if (ok && (m.flags & kNull)) {  // null slot: zero outputs, nothing else
      for (int e = pt; e < n * KD; e += kPrepConvThreads) {
        const int t = e / KD;
        p.out[static_cast<long long>(m.bos + t) * p.out_stride + static_cast<long long>(h) * KD + (e - t * KD)] = 0;
      }
    }
    if (live && n > 0) {  // (a fold-only item of the fold variant has no window)
      // the key / gate record of the window is the block's k | gate rows as
      // they are: one bulk store (its read of the slot is awaited before the
      // slot is released)
      if (pt == 0) {
        bulk_s2g(p.key_gate + m.r * p.kg_stride + static_cast<long long>(h) * p.Q * 2 * KD, kg_rows,
                 static_cast<uint32_t>(n) * 2 * KD * 2);
        bulk_commit();
      }
      // v_t for the gemv team's solve
      if (pt < KD) {
        float* opv = reinterpret_cast<float*>(op + Lay::kOpV);
#pragma unroll
        for (int t = 0; t < QMAX; ++t)
          if (t < n) opv[t * KD + pt] = bf16_to_f32(qv_rows[t * 2 * KD + KD + pt]);
      }
    }

    // ---- gates and the per-channel partial sums: key channel k = pt ----
    float qv[QMAX], kv[QMAX], eg[QMAX];
    if (live && pt < KD) {
      const int k = pt;
      const float* egr = reinterpret_cast<const float*>(sl + Lay::kEg);  // [QMAX][KD] from the conv pass
#pragma unroll
      for (int t = 0; t < QMAX; ++t) {
        qv[t] = t < n ? bf16_to_f32(qv_rows[t * 2 * KD + k]) : 0.0f;
        kv[t] = t < n ? bf16_to_f32(kg_rows[t * 2 * KD + k]) : 0.0f;
        eg[t] = t < n ? egr[t * KD + k] : 0.0f;
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
          const float dtb = reinterpret_cast<const float*>(sl + Lay::kDt)[k];
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
      warp_sum_values<Plan::P, Plan::H, Plan::C>(vals, lane);
      if ((lane & ((1 << (5 - Plan::H)) - 1)) == 0) {
#pragma unroll
        for (int v = 0; v < Plan::C; ++v) part[warp * NREDP + (lane >> (5 - Plan::H)) * Plan::C + v] = vals[v];
      }
    }
    named_barrier(kBarPrep, kPrepConvThreads);
    if (misc[kMiscPrepFail]) break;  // every prep thread sees the same flag here
    if (pt == 0) {  // the small inputs are consumed (and read by the record store)
      bulk_wait_read();
      mbar_arrive(&bars.sm_empty[slot]);
    }

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
      om->h = h;
      om->r = m.r;
#pragma unroll
      for (int t = 0; t < QMAX; ++t) om->beta[t] = beta[t];
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
  if (pt == 0) bulk_wait_all();  // the record stores have completed
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
  // unrolled by two only: one step already holds NV independent FMA chains,
  // and the kernel's hot code competes for the instruction cache with the
  // other roles (C2 verify call: 0.1655 ms against 0.1667 rolled)
#pragma unroll 2
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
  uint32_t live = 0;
  bool ok = true;
  for (int i = 0; ok; ++i) {
    const int oslot = i % Lay::kNumOp;
    ok = warp_wait(&bars.op_full[oslot], (i / Lay::kNumOp) & 1, lane, abort_flag, p.wait_limit_ns);
    if (!ok) break;
    const unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
    const OpMeta<QMAX> m = *reinterpret_cast<const OpMeta<QMAX>*>(op + Lay::kOpMeta);
    if (m.flags & kEnd) break;
    const int h = m.h;
    if (m.flags & kLive) {
      const int n = m.n;
      const uint32_t pc = live * kGemvWarps + gw;
      const int pos = pc % Lay::kNumChunk;
      ok = warp_wait_chunk(&bars.ch_full[pos], smem + Lay::oLap, pos, pc / Lay::kNumChunk, lane, abort_flag,
                           p.wait_limit_ns);
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
  uint32_t g = 0;  // slices issued
  bool ok = true;
  for (int i = 0; ok; ++i) {
    int flags, item;
    long long js;
    ok = next_ticket<KD, QMAX, VAR>(p, smem, i, lane, abort_flag, flags, item, js);
    if (!ok || item < 0) break;
    if (!(flags & kLive)) continue;
    const int jh = item - (item / p.H) * p.H;
    for (int kb = 0; kb < 4 && ok; ++kb, ++g) {
      const int pos = static_cast<int>(g % Lay::kNumChunk);
      if (lane == 0) {
        ok = mbar_wait_or_abort(&bars.ch_empty[pos], ((g / Lay::kNumChunk) & 1) ^ 1, abort_flag, p.wait_limit_ns);
        if (ok) {
          mbar_arrive_expect_tx(&bars.ch_full[pos], Lay::kChunk);
          tma_load_3d(smem + Lay::oChunks + pos * Lay::kChunk, &p.tm_state, kb * 32, jh * KD, static_cast<int>(js),
                      &bars.ch_full[pos]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
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
      (void)mbar_wait_bounded(&bars.ch_empty[g % Lay::kNumChunk], ((g / Lay::kNumChunk) & 1) ^ 1, p.wait_limit_ns);
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
                                            const volatile int* abort_flag, uint64_t limit_ns) {
  using Lay = Layout<KD, QMAX, VAR>;
  constexpr uint32_t kIdesc = umma_idesc_tf32(128, Layout<KD, QMAX, VAR>::kMmaN);
  Bars<KD, QMAX, VAR> bars(smem);
  if (!lp.valid) return true;
  lp.valid = false;
  if (!mbar_wait_or_abort(&bars.lo_full[lp.pos], (lp.g / Lay::kNumChunk) & 1, abort_flag, limit_ns)) return false;
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
  const uint32_t taddr = static_cast<uint32_t>(misc[kMiscTaddr]);
  uint32_t g = 0, live = 0;
  LoPending lp{false, false, 0, 0, 0, 0, 0};
  bool ok = true;
  for (int i = 0; ok; ++i) {
    const int oslot = i % Lay::kNumOp;
    const unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
    ok = mbar_wait_or_abort(&bars.op_full[oslot], (i / Lay::kNumOp) & 1, abort_flag, p.wait_limit_ns);
    if (!ok) break;
    const int flags = reinterpret_cast<const OpMeta<QMAX>*>(op + Lay::kOpMeta)->flags;
    if (flags & kEnd) break;
    if (!(flags & kLive)) {
      // finish the previous item first: its operand slot may be the next one
      // the prep team needs
      ok = tc_issue_lo<KD, QMAX, VAR>(smem, taddr, lp, abort_flag, p.wait_limit_ns);
      mbar_arrive(&bars.op_empty[oslot]);
      continue;
    }
    const uint32_t db = live & 1;
    ok = mbar_wait_or_abort(&bars.d_empty[db], ((live >> 1) & 1) ^ 1, abort_flag, p.wait_limit_ns);
    const uint64_t b = umma_desc_sw128(op);
    const uint32_t d = taddr + db * Lay::kDCols;
    for (int kb = 0; kb < 4 && ok; ++kb, ++g) {
      const int pos = static_cast<int>(g % Lay::kNumChunk);
      ok = mbar_wait_or_abort(&bars.ch_full[pos], (g / Lay::kNumChunk) & 1, abort_flag, p.wait_limit_ns);
      if (!ok) break;
      tmem_fence_after();
      const uint64_t a = umma_desc_sw128(smem + Lay::oChunks + pos * Lay::kChunk);
      const uint64_t bk = b + static_cast<uint64_t>(kb) * (Lay::kBSlice >> 4);  // B slice kb
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) umma_tf32(d, a + 2 * ks, bk + 2 * ks, kIdesc, kb > 0 || ks > 0);
      umma_commit(&bars.hi_done[pos]);
      ok = tc_issue_lo<KD, QMAX, VAR>(smem, taddr, lp, abort_flag, p.wait_limit_ns);
      lp = LoPending{true, kb == 3, pos, oslot, g, db, bk};
    }
    ++live;
  }
  if (ok) ok = tc_issue_lo<KD, QMAX, VAR>(smem, taddr, lp, abort_flag, p.wait_limit_ns);
  if (!ok) {
    report(p.workspace, KDA_DEVERR_TIMEOUT, blockIdx.x);
    *abort_flag = 1;
  }
}

// Readout team (4 warps; warp w of the CTA reads tensor-memory lanes
// 32 (w mod 4) .. 32 (w mod 4) + 31): each lane owns one state row; it sums
// the hi and lo columns into P_t | R_t and runs the row's solve.
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
  const int oslot = i % Lay::kNumOp;
  const unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
  const uint32_t db = live & 1;
  if (!warp_wait(&bars.d_full[db], (live >> 1) & 1, lane, abort_flag, p.wait_limit_ns)) return false;
  tmem_fence_after();
  float d[Lay::kDCols];
  const uint32_t ta = taddr + db * Lay::kDCols + (static_cast<uint32_t>(wq * 32) << 16);
#pragma unroll
  for (int c = 0; c < Lay::kDCols; c += 16) tmem_ld16(ta + c, *reinterpret_cast<float(*)[16]>(d + c));
  tmem_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars.d_empty[db]);
  const OpMeta<QMAX> m = *reinterpret_cast<const OpMeta<QMAX>*>(op + Lay::kOpMeta);
  const int h = m.h;
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
  // tcgen05.ld reaches the tensor-memory lanes of the warp's quadrant of the
  // CTA (warp index mod 4): this warp reads out rows 32 wq .. 32 wq + 31
  const int wq = static_cast<int>(threadIdx.x >> 5) & 3;
  const uint32_t taddr = static_cast<uint32_t>(misc[kMiscTaddr]);
  uint32_t g = 0, live = 0;
  int pending = -1;  // live item awaiting readout
  bool ok = true;
  for (int i = 0; ok; ++i) {
    const int oslot = i % Lay::kNumOp;
    const unsigned char* op = smem + Lay::oOp + oslot * Lay::kOp;
    ok = warp_wait(&bars.op_full[oslot], (i / Lay::kNumOp) & 1, lane, abort_flag, p.wait_limit_ns);
    if (!ok) break;
    const int flags = reinterpret_cast<const OpMeta<QMAX>*>(op + Lay::kOpMeta)->flags;
    if (flags & kEnd) break;
    if (!(flags & kLive)) {
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
      ok = warp_wait(&bars.ch_full[pos], (g / Lay::kNumChunk) & 1, lane, abort_flag, p.wait_limit_ns) &&
           warp_wait(&bars.hi_done[pos], (g / Lay::kNumChunk) & 1, lane, abort_flag, p.wait_limit_ns);
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

// A CTA's last act (one thread, after every role): the finish time for
// kda_verify_debug, and the count of finished CTAs, whose last zeroes the
// ticket counter for the next launch (every CTA has drawn its last ticket
// before it counts itself done).
__device__ __forceinline__ void finish_cta(const VerifyParams& p) {
  if (p.cta_times != nullptr) p.cta_times[2 * blockIdx.x + 1] = global_timer_ns();
  __threadfence();
  if (atomicAdd(p.workspace + kWsDone, 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(p.workspace + kWsTicket, 0);
    atomicExch(p.workspace + kWsDone, 0);
  }
}

template <int KD, int QMAX, int VAR>
__global__ void __launch_bounds__(Layout<KD, QMAX, VAR>::kThreads, 1) verify_kernel(const __grid_constant__ VerifyParams p) {
  using Lay = Layout<KD, QMAX, VAR>;
  extern __shared__ __align__(1024) unsigned char smem[];
  volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::oMisc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  if (p.cta_times != nullptr && tid == 0) p.cta_times[2 * blockIdx.x] = global_timer_ns();
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
    for (int i = 0; i < Lay::kTick; ++i) {
      mbar_init(&bars.tk_full[i], 1);
      mbar_init(&bars.tk_empty[i], 2);  // read by both producer warps
    }
    for (int i = 0; i < 8; ++i)
      if (i != kMiscTaddr) misc[i] = 0;  // the tensor-memory base is written by the allocating warp
    for (int i = 0; i < 64; ++i) (smem + Lay::oLap)[i] = 0xff;  // no lap armed yet
    fence_barrier_init();
  }
  if constexpr (Lay::kTC) {
    // the 128-byte swizzle of the MMA operands is anchored at 1024-byte boundaries
    if (smem_u32(smem) & 1023u) {
      if (tid == 0) {
        report(p.workspace, KDA_DEVERR_MISALIGNED, blockIdx.x);
        wait_prior_grid();
        finish_cta(p);
      }
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
    produce_inputs<KD, QMAX, VAR>(p, smem, tid & 31, misc);
  } else if (warp == 1) {
    if constexpr (Lay::kTC)
      tc_produce_state<KD, QMAX, VAR>(p, smem, tid & 31, misc + kMiscAbort);
    else
      produce_state<KD, QMAX, VAR>(p, smem, tid & 31, misc + kMiscAbort);
  } else if (warp < 2 + kPrepWarps) {
    prep<KD, QMAX, VAR>(p, smem, tid - 64, misc);
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
  // every role is done (and the inputs warp has its last ticket back)
  __syncthreads();
  if (tid == 0) finish_cta(p);
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

// Which verify runs the products at K = 128.  An M = 128 tf32 MMA costs about
// the same whatever N is, and fp32 accuracy takes a second (low-part) pass,
// so the tensor cores win only when the window brings many operand vectors:
// measured on GB300, the tcgen05 verify is faster for windows of 8 (C3) and
// slower for windows of 4 (C2), so that is the automatic choice.
bool use_tcgen05(int variant, bool window_up_to_4) {
  if (variant == KDA_VERIFY_TCGEN05) return true;
  if (variant == KDA_VERIFY_CUDA_CORE) return false;
  return !window_up_to_4;
}

int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices];  // zero-initialised: static storage
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int KD, int QMAX, int VAR>
cudaError_t launch(const VerifyParams& p, bool after_conv, cudaStream_t stream) {
  constexpr int bytes = Layout<KD, QMAX, VAR>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<KD, QMAX, VAR>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const int items = p.B * p.H;
  // After the conv pass, the launch is programmatic: the CTAs may start
  // (barrier set-up, state streaming) while the conv pass drains; the inputs
  // warp waits for it before its first copy from the scratch.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(items < sm_count() ? items : sm_count()));
  cfg.blockDim = dim3(Layout<KD, QMAX, VAR>::kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_conv ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, verify_kernel<KD, QMAX, VAR>, p);
}

template <int KD, int QMAX, bool DF>
cudaError_t launch_conv(const VerifyParams& p, cudaStream_t stream) {
  if (p.conv_weight_fp32)
    conv_kernel<KD, QMAX, DF, true><<<p.B * p.H, 3 * KD / 2, 0, stream>>>(p);
  else
    conv_kernel<KD, QMAX, DF, false><<<p.B * p.H, 3 * KD / 2, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& params, int K, int variant, cudaStream_t stream) {
  VerifyParams p = params;
  const bool q4 = p.Q <= 4;
  // the conv pass (nothing to convolve when every window is empty)
  if (p.T > 0) {
    cudaError_t e;
    if (K == 128)
      e = q4 ? (p.conv_dim_first ? launch_conv<128, 4, true>(p, stream) : launch_conv<128, 4, false>(p, stream))
             : (p.conv_dim_first ? launch_conv<128, 8, true>(p, stream) : launch_conv<128, 8, false>(p, stream));
    else
      e = q4 ? (p.conv_dim_first ? launch_conv<64, 4, true>(p, stream) : launch_conv<64, 4, false>(p, stream))
             : (p.conv_dim_first ? launch_conv<64, 8, true>(p, stream) : launch_conv<64, 8, false>(p, stream));
    if (e != cudaSuccess) return e;
  }
  const bool pdl = p.T > 0;
  if (p.fold_qsl != nullptr) {
    if (K == 128) return q4 ? launch<128, 4, kVarFold>(p, pdl, stream) : launch<128, 8, kVarFold>(p, pdl, stream);
    return q4 ? launch<64, 4, kVarFold>(p, pdl, stream) : launch<64, 8, kVarFold>(p, pdl, stream);
  }
  if (K == 128 && use_tcgen05(variant, q4) && build_state_map(p, K))
    return q4 ? launch<128, 4, kVarTcgen05>(p, pdl, stream) : launch<128, 8, kVarTcgen05>(p, pdl, stream);
  if (K == 128) return q4 ? launch<128, 4, kVarPlain>(p, pdl, stream) : launch<128, 8, kVarPlain>(p, pdl, stream);
  return q4 ? launch<64, 4, kVarPlain>(p, pdl, stream) : launch<64, 8, kVarPlain>(p, pdl, stream);
}

}  // namespace kda
