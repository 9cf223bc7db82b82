// kda_api.cpp -- the C ABI of libkda: host-side validation of every argument
// the host can check, launch-parameter marshalling, dispatch to the sm_103a
// kernels, and the error report.  The checks mirror the ValueErrors of
// "vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py" (kda_recoverssm_verify,
// KDARecoverSSMCommitContext.create / .commit) and the layout / support rules
// of "vllm.models.kimi_k3.nvidia.recoverssm.kernels" (_check_layouts,
// can_use_cute_recoverssm), as status codes instead of exceptions.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "kda.h"
#include "kda_params.h"

namespace kda {
cudaError_t launch_verify(const VerifyParams& p, int K, int variant, cudaStream_t stream);
cudaError_t launch_commit(const CommitParams& p, int K, cudaStream_t stream);
cudaError_t noalloc_tables(long long** out);
cudaError_t noalloc_fill(const int64_t* const src[6], int L, cudaStream_t stream);
}  // namespace kda

namespace {

thread_local char g_error[512] = "no error";

kda_status fail(kda_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_error, sizeof g_error, fmt, ap);
  va_end(ap);
  return st;
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

constexpr int kMaxWindow = 8;
constexpr int kConvWidth = 4;

kda_status check_dims(int H, int K, int V, int Q) {
  if (H <= 0 || K <= 0 || V <= 0 || Q <= 0)
    return fail(KDA_ERR_INVALID_ARG, "H, K, V and Q must be positive (H=%d K=%d V=%d Q=%d)", H, K, V, Q);
  if (K != V) return fail(KDA_ERR_UNSUPPORTED, "K (%d) must equal V (%d)", K, V);
  if (K != 64 && K != 128) return fail(KDA_ERR_UNSUPPORTED, "head dim %d: supported 64 and 128", K);
  if (Q > kMaxWindow) return fail(KDA_ERR_UNSUPPORTED, "window %d: supported 1 to %d tokens", Q, kMaxWindow);
  return KDA_OK;
}

}  // namespace

extern "C" {

int32_t kda_abi_version(void) { return KDA_ABI_VERSION; }

size_t kda_workspace_bytes(void) { return kda::kWsWords * sizeof(int32_t); }

size_t kda_verify_scratch_bytes(int32_t B, int32_t H, int32_t K, int32_t Q) {
  if (B <= 0 || H <= 0 || K <= 0 || Q <= 0) return 0;
  return static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(kda::scratch_item_elems(Q, K)) * 2u;
}


const char* kda_last_error(void) { return g_error; }

}  // extern "C"

namespace {

// Checks the verify arguments and fills the launch parameters; *noop is set
// when there is nothing to launch.
kda_status verify_params(const kda_verify_args* a, bool fold, kda::VerifyParams& p, bool* noop) {
  *noop = false;
  if (a == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_verify: args is NULL");
  if (a->B < 0 || a->T < 0) return fail(KDA_ERR_INVALID_ARG, "kda_verify: negative B (%d) or T (%d)", a->B, a->T);
  kda_status st = check_dims(a->H, a->K, a->V, a->Q);
  if (st != KDA_OK) return st;
  if (a->W != kConvWidth) return fail(KDA_ERR_UNSUPPORTED, "kda_verify: conv width %d, supported %d", a->W, kConvWidth);
  if ((long long)a->T > (long long)a->B * a->Q)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: %d token rows exceed B*Q = %lld", a->T, (long long)a->B * a->Q);
  // the ticket counter of the verify's schedule lives in the workspace
  if (a->workspace == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_verify: workspace is NULL (required)");
  if (!aligned(a->workspace, 4)) return fail(KDA_ERR_MISALIGNED, "kda_verify: workspace must be 4-byte aligned");
  // the fold still has work when no token row is left
  if (a->B == 0 || (a->T == 0 && !fold)) {
    *noop = true;
    return KDA_OK;
  }
  const void* required[] = {a->A_log,    a->dt_bias, a->conv_weight,     a->conv_state,   a->state,
                            a->corr,     a->key_gate, a->query_start_loc, a->state_indices};
  for (const void* ptr : required)
    if (ptr == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_verify: a required pointer is NULL");
  // the activations are read only for token rows: a fold-only step (T == 0)
  // may pass NULL for them
  const void* activations[] = {a->mixed_qkv, a->raw_gate, a->raw_beta, a->out};
  for (const void* ptr : activations)
    if (ptr == nullptr && a->T > 0) return fail(KDA_ERR_INVALID_ARG, "kda_verify: an activation pointer is NULL");
  if (a->gate_mode != KDA_GATE_SOFTPLUS && a->gate_mode != KDA_GATE_LOWER_BOUND)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: gate_mode %d", a->gate_mode);
  if (a->gate_mode == KDA_GATE_LOWER_BOUND && !std::isfinite(a->lower_bound))
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: lower_bound is not finite");
  if (a->conv_layout != KDA_CONV_DIM_FIRST && a->conv_layout != KDA_CONV_SEQ_FIRST)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: conv_layout %d", a->conv_layout);
  if (a->conv_weight_dtype != KDA_DTYPE_BF16 && a->conv_weight_dtype != KDA_DTYPE_FP32)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: conv_weight_dtype %d", a->conv_weight_dtype);
  if (a->num_slots <= 0 || a->num_record_rows <= 0)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: num_slots and num_record_rows must be positive");
  const long long H = a->H, K = a->K, V = a->V, Q = a->Q;
  const long long conv_len = Q + kConvWidth - 2;
  // with no token row (a fold-only step) the activations are never read:
  // their pointers may be NULL and their strides anything
  if (a->T > 0 && (a->qkv_row_stride < 3 * H * K || a->gate_row_stride < H * K || a->beta_row_stride < H ||
                   a->out_row_stride < H * V))
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: an activation row stride is shorter than its row");
  if (a->variant != KDA_VERIFY_AUTO && a->variant != KDA_VERIFY_CUDA_CORE && a->variant != KDA_VERIFY_TCGEN05)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: variant %d", a->variant);
  if (a->variant == KDA_VERIFY_TCGEN05 && K != 128)
    return fail(KDA_ERR_UNSUPPORTED, "kda_verify: the tensor-core variant needs K == 128 (K = %lld)", K);
  if (a->T > 0) {
    const size_t need = kda_verify_scratch_bytes(a->B, a->H, a->K, a->Q);
    if (a->scratch == nullptr || a->scratch_bytes < 0 || static_cast<size_t>(a->scratch_bytes) < need)
      return fail(KDA_ERR_INVALID_ARG, "kda_verify: scratch of %zu bytes required (got %lld)", need,
                  static_cast<long long>(a->scratch_bytes));
    if (!aligned(a->scratch, 16)) return fail(KDA_ERR_MISALIGNED, "kda_verify: scratch must start on 16 bytes");
  }
  if (a->conv_slot_stride < 3 * H * K * conv_len)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: conv_slot_stride %lld < 3HK*(Q+W-2) = %lld",
                (long long)a->conv_slot_stride, 3 * H * K * conv_len);
  if (a->state_slot_stride < H * V * K)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: state_slot_stride %lld < H*V*K", (long long)a->state_slot_stride);
  if (a->corr_row_stride < H * Q * V || a->kg_row_stride < H * Q * 2 * K)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify: a record row stride is shorter than its row");
  // static tensors: 16-byte aligned starts and slot / row strides
  if (!aligned(a->state, 16) || (a->state_slot_stride * 4) % 16 || !aligned(a->corr, 16) ||
      (a->corr_row_stride * 4) % 16 || !aligned(a->key_gate, 16) || (a->kg_row_stride * 2) % 16 ||
      !aligned(a->conv_state, 16) || (a->conv_slot_stride * 2) % 16 || !aligned(a->conv_weight, 16) ||
      !aligned(a->A_log, 16) || !aligned(a->dt_bias, 16))
    return fail(KDA_ERR_MISALIGNED,
                "kda_verify: state, records, conv state, conv weight and gate parameters must start on "
                "16-byte boundaries with 16-byte multiple slot / row strides");
  if (!aligned(a->mixed_qkv, 2) || !aligned(a->raw_gate, 2) || !aligned(a->raw_beta, 2) || !aligned(a->out, 2))
    return fail(KDA_ERR_MISALIGNED, "kda_verify: bf16 activations must be 2-byte aligned");

  p = kda::VerifyParams{};
  p.B = a->B; p.H = a->H; p.Q = a->Q; p.T = a->T; p.null_block_id = a->null_block_id;
  p.num_slots = a->num_slots; p.num_record_rows = a->num_record_rows;
  p.mixed_qkv = static_cast<const uint16_t*>(a->mixed_qkv); p.qkv_stride = a->qkv_row_stride;
  p.raw_gate = static_cast<const uint16_t*>(a->raw_gate); p.gate_stride = a->gate_row_stride;
  p.raw_beta = static_cast<const uint16_t*>(a->raw_beta); p.beta_stride = a->beta_row_stride;
  p.out = static_cast<uint16_t*>(a->out); p.out_stride = a->out_row_stride;
  p.A_log = a->A_log; p.dt_bias = a->dt_bias;
  p.lower_bound_gate = a->gate_mode == KDA_GATE_LOWER_BOUND; p.lower_bound = a->lower_bound;
  p.conv_weight = a->conv_weight; p.conv_weight_fp32 = a->conv_weight_dtype == KDA_DTYPE_FP32;
  p.conv_state = static_cast<uint16_t*>(a->conv_state); p.conv_dim_first = a->conv_layout == KDA_CONV_DIM_FIRST;
  p.conv_slot_stride = a->conv_slot_stride;
  p.state = a->state; p.state_slot_stride = a->state_slot_stride;
  p.corr = a->corr; p.corr_stride = a->corr_row_stride;
  p.key_gate = static_cast<uint16_t*>(a->key_gate); p.kg_stride = a->kg_row_stride;
  p.qsl = a->query_start_loc; p.state_indices = a->state_indices;
  p.record_indices = a->record_indices; p.num_accepted_prev = a->num_accepted_prev;
  p.workspace = a->workspace;
  p.k_scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(K)));
  p.scratch = static_cast<uint16_t*>(a->scratch);
  p.wait_limit_ns = 1000000000ull;  // every device wait gives up after about a second
  p.withhold_item = -1;
  p.cta_times = nullptr;
  // the ticket counter runs to B*H plus one ticket per CTA
  if ((long long)p.B * p.H > 0x7fff0000LL) return fail(KDA_ERR_UNSUPPORTED, "kda_verify: B*H too large");
  return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_verify(const kda_verify_args* a, kda_stream_t stream) {
  kda::VerifyParams p;
  bool noop = false;
  const kda_status st = verify_params(a, false, p, &noop);
  if (st != KDA_OK || noop) return st;
  cudaError_t e = kda::launch_verify(p, a->K, a->variant, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "kda_verify: launch failed: %s", cudaGetErrorString(e));
  return KDA_OK;
}

kda_status kda_verify_fold(const kda_verify_args* a, const kda_fold_args* f, kda_stream_t stream) {
  if (f == nullptr || f->query_start_loc == nullptr) return kda_verify(a, stream);
  if (f->num_accepted == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_verify_fold: num_accepted is NULL");
  kda::VerifyParams p;
  bool noop = false;
  const kda_status st = verify_params(a, true, p, &noop);
  if (st != KDA_OK || noop) return st;
  p.fold_qsl = f->query_start_loc;
  p.fold_num_accepted = f->num_accepted;
  p.fold_record_indices = f->record_indices;
  cudaError_t e = kda::launch_verify(p, a->K, a->variant, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "kda_verify_fold: launch failed: %s", cudaGetErrorString(e));
  return KDA_OK;
}

kda_status kda_verify_debug(const kda_verify_args* a, const kda_debug_args* d, kda_stream_t stream) {
  if (d == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_verify_debug: debug args are NULL");
  if (d->wait_limit_ns <= 0) return fail(KDA_ERR_INVALID_ARG, "kda_verify_debug: wait_limit_ns must be positive");
  kda::VerifyParams p;
  bool noop = false;
  const kda_status st = verify_params(a, false, p, &noop);
  if (st != KDA_OK || noop) return st;
  if (d->withhold_item < -1 || static_cast<long long>(d->withhold_item) >= static_cast<long long>(a->B) * a->H)
    return fail(KDA_ERR_INVALID_ARG, "kda_verify_debug: withhold_item %d is not -1 or an item", d->withhold_item);
  if (!aligned(d->cta_times, 8)) return fail(KDA_ERR_MISALIGNED, "kda_verify_debug: cta_times must be 8-byte aligned");
  p.wait_limit_ns = static_cast<unsigned long long>(d->wait_limit_ns);
  p.withhold_item = d->withhold_item;
  p.cta_times = reinterpret_cast<unsigned long long*>(d->cta_times);
  // withholding exercises the abort sequence of the CUDA-core verify
  const int variant = d->withhold_item >= 0 ? KDA_VERIFY_CUDA_CORE : a->variant;
  cudaError_t e = kda::launch_verify(p, a->K, variant, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "kda_verify_debug: launch failed: %s", cudaGetErrorString(e));
  return KDA_OK;
}

kda_status kda_commit(const kda_commit_args* a, kda_stream_t stream) { return kda_commit_align(a, nullptr, stream); }

kda_status kda_commit_align(const kda_commit_args* a, const kda_align_args* al, kda_stream_t stream) {
  if (a == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_commit: args is NULL");
  if (al != nullptr && al->boundary_state_indices != nullptr && al->boundary_recovery_lens == nullptr)
    return fail(KDA_ERR_INVALID_ARG, "kda_commit_align: boundary_recovery_lens is NULL with boundary slots");
  if (a->L <= 0) return fail(KDA_ERR_INVALID_ARG, "kda_commit: needs at least one layer (L=%d)", a->L);
  if (a->B < 0) return fail(KDA_ERR_INVALID_ARG, "kda_commit: negative B (%d)", a->B);
  kda_status st = check_dims(a->H, a->K, a->V, a->Q);
  if (st != KDA_OK) return st;
  if (a->B == 0) return KDA_OK;
  const void* required[] = {a->state_base, a->state_slot_stride, a->corr_base, a->corr_row_stride,
                            a->kg_base,    a->kg_row_stride,     a->A_log,     a->dt_bias,
                            a->query_start_loc, a->state_indices, a->num_accepted};
  for (const void* ptr : required)
    if (ptr == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_commit: a required pointer is NULL");
  if (a->gate_mode != KDA_GATE_SOFTPLUS && a->gate_mode != KDA_GATE_LOWER_BOUND)
    return fail(KDA_ERR_INVALID_ARG, "kda_commit: gate_mode %d", a->gate_mode);
  if (a->gate_mode == KDA_GATE_LOWER_BOUND && !std::isfinite(a->lower_bound))
    return fail(KDA_ERR_INVALID_ARG, "kda_commit: lower_bound is not finite");
  if (a->num_slots <= 0 || a->num_record_rows <= 0)
    return fail(KDA_ERR_INVALID_ARG, "kda_commit: num_slots and num_record_rows must be positive");
  if (!aligned(a->A_log, 4) || !aligned(a->dt_bias, 4))
    return fail(KDA_ERR_MISALIGNED, "kda_commit: gate parameters must be 4-byte aligned");
  if ((long long)a->L * a->B * a->H > 0x7fffffffLL) return fail(KDA_ERR_UNSUPPORTED, "kda_commit: L*B*H too large");

  kda::CommitParams p{};
  p.L = a->L; p.B = a->B; p.H = a->H; p.Q = a->Q; p.null_block_id = a->null_block_id;
  p.num_slots = a->num_slots; p.num_record_rows = a->num_record_rows;
  p.state_base = reinterpret_cast<const long long*>(a->state_base);
  p.state_stride = reinterpret_cast<const long long*>(a->state_slot_stride);
  p.corr_base = reinterpret_cast<const long long*>(a->corr_base);
  p.corr_stride = reinterpret_cast<const long long*>(a->corr_row_stride);
  p.kg_base = reinterpret_cast<const long long*>(a->kg_base);
  p.kg_stride = reinterpret_cast<const long long*>(a->kg_row_stride);
  p.A_log = a->A_log; p.dt_bias = a->dt_bias;
  p.lower_bound_gate = a->gate_mode == KDA_GATE_LOWER_BOUND; p.lower_bound = a->lower_bound;
  p.qsl = a->query_start_loc; p.state_indices = a->state_indices;
  p.record_indices = a->record_indices; p.num_accepted = a->num_accepted;
  p.workspace = a->workspace;
  if (al != nullptr) {
    p.final_state_indices = al->final_state_indices;
    p.boundary_state_indices = al->boundary_state_indices;
    p.boundary_recovery_lens = al->boundary_recovery_lens;
  }
  cudaError_t e = kda::launch_commit(p, a->K, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "kda_commit: launch failed: %s", cudaGetErrorString(e));
  return KDA_OK;
}

kda_status kda_commit_noalloc(const kda_commit_args* a, kda_stream_t stream) {
  constexpr int kMax = KDA_NOALLOC_MAX_LAYERS;
  if (a == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_commit_noalloc: args is NULL");
  if (a->L <= 0) return fail(KDA_ERR_INVALID_ARG, "kda_commit_noalloc: needs at least one layer (L=%d)", a->L);
  if (a->L > kMax)
    return fail(KDA_ERR_UNSUPPORTED, "kda_commit_noalloc: L=%d layers exceed its static scratch of %d layers",
                a->L, kMax);
  if (a->B < 0) return fail(KDA_ERR_INVALID_ARG, "kda_commit_noalloc: negative B (%d)", a->B);
  kda_status st = check_dims(a->H, a->K, a->V, a->Q);
  if (st != KDA_OK) return st;
  if (a->B == 0) return KDA_OK;
  const void* required[] = {a->state_base, a->state_slot_stride, a->corr_base, a->corr_row_stride,
                            a->kg_base,    a->kg_row_stride,     a->A_log,     a->dt_bias,
                            a->query_start_loc, a->state_indices, a->num_accepted};
  for (const void* ptr : required)
    if (ptr == nullptr) return fail(KDA_ERR_INVALID_ARG, "kda_commit_noalloc: a required pointer is NULL");
  if (a->gate_mode != KDA_GATE_SOFTPLUS && a->gate_mode != KDA_GATE_LOWER_BOUND)
    return fail(KDA_ERR_INVALID_ARG, "kda_commit_noalloc: gate_mode %d", a->gate_mode);
  if (a->gate_mode == KDA_GATE_LOWER_BOUND && !std::isfinite(a->lower_bound))
    return fail(KDA_ERR_INVALID_ARG, "kda_commit_noalloc: lower_bound is not finite");
  if (a->num_slots <= 0 || a->num_record_rows <= 0)
    return fail(KDA_ERR_INVALID_ARG, "kda_commit_noalloc: num_slots and num_record_rows must be positive");
  if (!aligned(a->A_log, 4) || !aligned(a->dt_bias, 4))
    return fail(KDA_ERR_MISALIGNED, "kda_commit_noalloc: gate parameters must be 4-byte aligned");
  if ((long long)a->L * a->B * a->H > 0x7fffffffLL)
    return fail(KDA_ERR_UNSUPPORTED, "kda_commit_noalloc: L*B*H too large");

  long long* tables = nullptr;
  cudaError_t e = kda::noalloc_tables(&tables);
  if (e != cudaSuccess)
    return fail(KDA_ERR_CUDA, "kda_commit_noalloc: scratch set-up failed: %s", cudaGetErrorString(e));
  // the host tables travel by value in the parameters of a small kernel that
  // writes them into the scratch, in stream order (table j of layer l at
  // [j * kMax + l])
  const int64_t* src[6] = {a->state_base, a->state_slot_stride, a->corr_base,
                           a->corr_row_stride, a->kg_base, a->kg_row_stride};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  e = kda::noalloc_fill(src, a->L, s);
  if (e != cudaSuccess)
    return fail(KDA_ERR_CUDA, "kda_commit_noalloc: table fill failed: %s", cudaGetErrorString(e));

  kda::CommitParams p{};
  p.L = a->L; p.B = a->B; p.H = a->H; p.Q = a->Q; p.null_block_id = a->null_block_id;
  p.num_slots = a->num_slots; p.num_record_rows = a->num_record_rows;
  p.state_base = tables + 0 * kMax;
  p.state_stride = tables + 1 * kMax;
  p.corr_base = tables + 2 * kMax;
  p.corr_stride = tables + 3 * kMax;
  p.kg_base = tables + 4 * kMax;
  p.kg_stride = tables + 5 * kMax;
  p.A_log = a->A_log; p.dt_bias = a->dt_bias;
  p.lower_bound_gate = a->gate_mode == KDA_GATE_LOWER_BOUND; p.lower_bound = a->lower_bound;
  p.qsl = a->query_start_loc; p.state_indices = a->state_indices;
  p.record_indices = a->record_indices; p.num_accepted = a->num_accepted;
  p.workspace = a->workspace;
  e = kda::launch_commit(p, a->K, s);
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "kda_commit_noalloc: launch failed: %s", cudaGetErrorString(e));
  return KDA_OK;
}

kda_status kda_read_device_error(const int32_t* workspace, kda_stream_t stream, int32_t* flags) {
  if (workspace == nullptr || flags == nullptr)
    return fail(KDA_ERR_INVALID_ARG, "kda_read_device_error: NULL workspace or flags");
  int32_t host = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&host, workspace, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "kda_read_device_error: %s", cudaGetErrorString(e));
  *flags = host;
  if (host != 0) return fail(KDA_ERR_DEVICE, "device reported error bits 0x%x", host);
  return KDA_OK;
}

}  // extern "C"
