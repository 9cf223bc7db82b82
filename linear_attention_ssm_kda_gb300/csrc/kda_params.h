// kda_params.h -- launch parameters of the verify and commit kernels: plain
// structs of device pointers, built by the host API from the C-ABI arguments.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <stdint.h>

namespace kda {

// Workspace words (int32): [0] the error bits, [1] the item of the last
// report, [kWsTicket] the verify's next work item and [kWsDone] its finished
// CTAs (both zero between launches).
constexpr int kWsTicket = 8;
constexpr int kWsDone = 9;
constexpr int kWsWords = 16;

// The conv pass's block per (request, head) item in the scratch: [Q][2K] bf16
// rows q | v, [Q][2K] rows k | raw gate, 8 fp32 sigmoid(raw beta), then
// [Q][K] fp32 decays e^g of the key channels (rows t < n written).  In
// uint16 elements; scratch_eg_elem is where the decays start.
constexpr int kScratchBetaBytes = 32;
#if defined(__CUDACC__)
__host__ __device__
#endif
constexpr long long scratch_eg_elem(int Q, int K) {
  return 4LL * Q * K + kScratchBetaBytes / 2;
}
#if defined(__CUDACC__)
__host__ __device__
#endif
constexpr long long scratch_item_elems(int Q, int K) {
  return scratch_eg_elem(Q, K) + 2LL * Q * K;
}

struct VerifyParams {
  int B, H, Q, T, null_block_id;
  long long num_slots, num_record_rows;
  const uint16_t* mixed_qkv; long long qkv_stride;
  const uint16_t* raw_gate; long long gate_stride;
  const uint16_t* raw_beta; long long beta_stride;
  uint16_t* out; long long out_stride;
  const float* A_log;
  const float* dt_bias;
  int lower_bound_gate; float lower_bound;
  const void* conv_weight; int conv_weight_fp32;
  uint16_t* conv_state; int conv_dim_first; long long conv_slot_stride;
  const float* state; long long state_slot_stride;
  float* corr; long long corr_stride;
  uint16_t* key_gate; long long kg_stride;
  const int* qsl; const int* state_indices; const int* record_indices; const int* num_accepted_prev;
  int* workspace;
  float k_scale;  // K^-1/2
  // the conv pass's output: per (request, head) item a block of
  // scratch_item_elems(Q, K) uint16 (layout above)
  uint16_t* scratch;
  // fp32 state pool [slots][H V][K] in K-slices of 32 (128-byte swizzle), for
  // the tensor-core path of the verify
  CUtensorMap tm_state;
  // kda_verify_fold: each request's pending records of the previous step
  // (query_start_loc, accepted counts, record rows or NULL for the state slot)
  // folded into its checkpoint first; fold_qsl == nullptr: plain verify
  const int* fold_qsl; const int* fold_num_accepted; const int* fold_record_indices;
  // bounded waits: the limit (about a second; kda_verify_debug may shorten
  // it) and the item whose inputs the inputs warp withholds (kda_verify_debug;
  // -1: none)
  unsigned long long wait_limit_ns;
  int withhold_item;
  // kda_verify_debug: per CTA the global timer at its start and finish, or
  // nullptr
  unsigned long long* cta_times;
};

struct CommitParams {
  int L, B, H, Q, null_block_id;
  long long num_slots, num_record_rows;
  const long long* state_base; const long long* state_stride;
  const long long* corr_base; const long long* corr_stride;
  const long long* kg_base; const long long* kg_stride;
  const float* A_log; const float* dt_bias;
  int lower_bound_gate; float lower_bound;
  const int* qsl; const int* state_indices; const int* record_indices; const int* num_accepted;
  int* workspace;
  // align mode (kda_commit_align), each [B] or nullptr: the final slot (the
  // source slot when null), the boundary slot and its recovery length
  const int* final_state_indices; const int* boundary_state_indices; const int* boundary_recovery_lens;
};

}  // namespace kda
