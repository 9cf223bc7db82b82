// kda_commit.cu -- the KDA RecoverSSM accepted-state commit for sm_103a.
//
// Computes what "vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py"
// (_commit_kda_state_kernel, launched by KDARecoverSSMCommitContext.commit)
// computes for the non-align plan: every layer in one launch, each request
// folding its first m = min(max(num_accepted, 0), n) verify records into its
// fp32 state in place,
//   S <- S0 diag(prod_t e^{g_t}) + sum_t c_t (k^_t * prod_{u>t} e^{g_u})^T,
// with k^_t and g_t recomputed from the key/gate record and c_t the stored
// correction.  One CTA per (layer, request, head); the 64 KB state block
// arrives by one bulk copy (TMA) issued first, the records and gates are
// prepared while it is in flight, and the result leaves by 16-byte stores.
//
// Align mode (prefix caching, the kernel's ALIGN_MODE on the same page): the
// committed state goes to final_state_indices[b] (nothing is written when
// that slot is null), and a live boundary_state_indices[b] receives the state
// after the first R = boundary_recovery_lens[b] of the m tokens, from the
// same pass over the state.
#include <cuda_runtime.h>

#include "kda_device.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;

template <int KD, int QMAX, bool ALIGN>
struct CommitLayout {
  static constexpr int kState = 0;                       // float [KD][KD]
  static constexpr int kKd = kState + KD * KD * 4;       // float [QMAX][KD]  k^_t * prod_{u>t} e^g
  static constexpr int kDall = kKd + QMAX * KD * 4;      // float [KD]        prod_t e^g
  // align mode: the same over the tokens before the boundary
  static constexpr int kKdb = kDall + KD * 4;            // float [QMAX][KD]  k^_t * prod_{t<u<R} e^g
  static constexpr int kDallb = kKdb + (ALIGN ? QMAX * KD * 4 : 0);  // float [KD] prod_{t<R} e^g
  static constexpr int kC = kDallb + (ALIGN ? KD * 4 : 0);           // float [QMAX][KD]  c_t
  static constexpr int kNorm = kC + QMAX * KD * 4;       // float [QMAX][KD/32] per-warp parts of |k_t|^2
  static constexpr int kBar = (kNorm + QMAX * (KD / 32) * 4 + 7) / 8 * 8;
  static constexpr int kBytes = kBar + 8;
};

__device__ __forceinline__ bool aligned16(long long addr) { return (addr & 15) == 0; }

template <int KD, int QMAX, bool ALIGN>
__global__ void __launch_bounds__(kThreads, 3) commit_kernel(const CommitParams p) {
  using Lay = CommitLayout<KD, QMAX, ALIGN>;
  extern __shared__ __align__(128) unsigned char smem[];
  float* s_state = reinterpret_cast<float*>(smem + Lay::kState);
  float* s_kd = reinterpret_cast<float*>(smem + Lay::kKd);
  float* s_dall = reinterpret_cast<float*>(smem + Lay::kDall);
  float* s_c = reinterpret_cast<float*>(smem + Lay::kC);
  float* s_norm = reinterpret_cast<float*>(smem + Lay::kNorm);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Lay::kBar);

  const int tid = threadIdx.x;
  const int item = blockIdx.x;
  const int per_layer = p.B * p.H;
  const int l = item / per_layer;
  const int rem = item - l * per_layer;
  const int b = rem / p.H;
  const int h = rem - b * p.H;

  // the layer's tables, loaded with the request's metadata (one round trip)
  const long long state_base = p.state_base[l], state_stride = p.state_stride[l];
  const long long corr_base = p.corr_base[l], corr_stride = p.corr_stride[l];
  const long long kg_base = p.kg_base[l], kg_stride = p.kg_stride[l];
  // ---- plan: skip null slots and empty commits ----
  const long long s = p.state_indices[b];
  if (s <= p.null_block_id) return;
  const int len = p.qsl[b + 1] - p.qsl[b];
  const int n = min(max(len, 0), p.Q);
  const int m = min(max(p.num_accepted[b], 0), n);
  if (m == 0) return;
  if (s < 0 || s >= p.num_slots) {
    if (tid == 0) report(p.workspace, KDA_DEVERR_SLOT_RANGE, item);
    return;
  }
  const long long r = p.record_indices ? (long long)p.record_indices[b] : s;
  if (r < 0 || r >= p.num_record_rows) {
    if (tid == 0) report(p.workspace, KDA_DEVERR_ROW_RANGE, item);
    return;
  }
  long long fs = s, bs = p.null_block_id;  // final and boundary slots
  int rb = 0;                              // tokens before the boundary
  if constexpr (ALIGN) {
    fs = p.final_state_indices ? (long long)p.final_state_indices[b] : s;
    if (fs <= p.null_block_id) return;
    bs = p.boundary_state_indices ? (long long)p.boundary_state_indices[b] : p.null_block_id;
    if (fs >= p.num_slots || bs >= p.num_slots) {
      if (tid == 0) report(p.workspace, KDA_DEVERR_SLOT_RANGE, item);
      return;
    }
    rb = p.boundary_recovery_lens ? min(max(p.boundary_recovery_lens[b], 0), m) : 0;
  }
  if (!aligned16(state_base) || !aligned16(state_stride * 4) || !aligned16(corr_base) ||
      !aligned16(corr_stride * 4) || !aligned16(kg_base) || !aligned16(kg_stride * 2)) {
    if (tid == 0) report(p.workspace, KDA_DEVERR_MISALIGNED, item);
    return;
  }
  float* gS = reinterpret_cast<float*>(state_base) + s * state_stride + (long long)h * KD * KD;
  float* gF = reinterpret_cast<float*>(state_base) + fs * state_stride + (long long)h * KD * KD;
  float* gB = reinterpret_cast<float*>(state_base) + bs * state_stride + (long long)h * KD * KD;
  const float* gc = reinterpret_cast<const float*>(corr_base) + r * corr_stride + (long long)h * p.Q * KD;
  const uint16_t* gkg = reinterpret_cast<const uint16_t*>(kg_base) + r * kg_stride + (long long)h * p.Q * 2 * KD;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, KD * KD * 4);
#pragma unroll
    for (int c = 0; c < 4; ++c) bulk_g2s(s_state + c * (KD * KD / 4), gS + c * (KD * KD / 4), KD * KD, bar);
  }
  for (int i = tid; i < m * KD; i += kThreads) s_c[i] = gc[i];
  __syncthreads();

  // ---- gates and normalised keys from the key/gate records ----
  const int lane = tid & 31;
  float kv[QMAX], eg[QMAX];
  if (tid < KD) {
    const float A = expf(p.A_log[l * p.H + h]);
    const float dtb = p.dt_bias[((long long)l * p.H + h) * KD + tid];
#pragma unroll
    for (int t = 0; t < QMAX; ++t) {
      if (t < m) {
        kv[t] = bf16_to_f32(gkg[t * 2 * KD + tid]);
        eg[t] = expf(kda_gate(bf16_to_f32(gkg[t * 2 * KD + KD + tid]), dtb, A, p.lower_bound_gate, p.lower_bound));
        const float kk = warp_sum(kv[t] * kv[t]);
        if (lane == 0) s_norm[t * (KD / 32) + (tid >> 5)] = kk;  // summed in a fixed order below
      }
    }
  }
  __syncthreads();
  if (tid < KD) {
    float suffix = 1.0f;   // prod_{u>t} e^{g_u}
    float suffixb = 1.0f;  // align mode: prod_{t<u<R} e^{g_u}
#pragma unroll
    for (int t = QMAX - 1; t >= 0; --t) {
      if (t < m) {
        float kk = 0.0f;
#pragma unroll
        for (int w = 0; w < KD / 32; ++w) kk += s_norm[t * (KD / 32) + w];
        const float kn = kv[t] * rsqrtf(kk + 1e-6f);
        s_kd[t * KD + tid] = kn * suffix;
        suffix *= eg[t];
        if constexpr (ALIGN) {
          if (t < rb) {
            reinterpret_cast<float*>(smem + Lay::kKdb)[t * KD + tid] = kn * suffixb;
            suffixb *= eg[t];
          }
        }
      }
    }
    s_dall[tid] = suffix;
    if constexpr (ALIGN) reinterpret_cast<float*>(smem + Lay::kDallb)[tid] = suffixb;
  }
  __syncthreads();

  const bool ok = mbar_wait_bounded(bar, 0);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) {
      report(p.workspace, KDA_DEVERR_TIMEOUT, item);
      (void)mbar_wait_bounded(bar, 0);
    }
    return;
  }

  // ---- fold and store ----
  const float4* st4 = reinterpret_cast<const float4*>(s_state);
  const float4* dall4 = reinterpret_cast<const float4*>(s_dall);
  const float4* kd4 = reinterpret_cast<const float4*>(s_kd);
  float4* out4 = reinterpret_cast<float4*>(gF);
  constexpr int kChunksPerRow = KD / 4;
  if constexpr (ALIGN) {
    if (bs > p.null_block_id) {  // written first: a final slot equal to it wins
      const float4* dallb4 = reinterpret_cast<const float4*>(smem + Lay::kDallb);
      const float4* kdb4 = reinterpret_cast<const float4*>(smem + Lay::kKdb);
      float4* bnd4 = reinterpret_cast<float4*>(gB);
#pragma unroll 4
      for (int idx = tid; idx < KD * KD / 4; idx += kThreads) {
        const int row = idx / kChunksPerRow;
        const int kc = idx - row * kChunksPerRow;
        const float4 sv = st4[idx];
        const float4 d = dallb4[kc];
        float4 o = make_float4(sv.x * d.x, sv.y * d.y, sv.z * d.z, sv.w * d.w);
#pragma unroll
        for (int t = 0; t < QMAX; ++t) {
          if (t < rb) {
            const float c = s_c[t * KD + row];
            const float4 k = kdb4[t * kChunksPerRow + kc];
            o.x = fmaf(c, k.x, o.x);
            o.y = fmaf(c, k.y, o.y);
            o.z = fmaf(c, k.z, o.z);
            o.w = fmaf(c, k.w, o.w);
          }
        }
        bnd4[idx] = o;
      }
      if (bs == fs) __syncthreads();  // the final state overwrites it in order
    }
  }
#pragma unroll 4
  for (int idx = tid; idx < KD * KD / 4; idx += kThreads) {
    const int row = idx / kChunksPerRow;
    const int kc = idx - row * kChunksPerRow;
    const float4 sv = st4[idx];
    const float4 d = dall4[kc];
    float4 o = make_float4(sv.x * d.x, sv.y * d.y, sv.z * d.z, sv.w * d.w);
#pragma unroll
    for (int t = 0; t < QMAX; ++t) {
      if (t < m) {
        const float c = s_c[t * KD + row];
        const float4 k = kd4[t * kChunksPerRow + kc];
        o.x = fmaf(c, k.x, o.x);
        o.y = fmaf(c, k.y, o.y);
        o.z = fmaf(c, k.z, o.z);
        o.w = fmaf(c, k.w, o.w);
      }
    }
    out4[idx] = o;
  }
}

template <int KD, int QMAX, bool ALIGN>
cudaError_t launch(const CommitParams& p, cudaStream_t stream) {
  constexpr int bytes = CommitLayout<KD, QMAX, ALIGN>::kBytes;
  cudaError_t e =
      cudaFuncSetAttribute(commit_kernel<KD, QMAX, ALIGN>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  commit_kernel<KD, QMAX, ALIGN><<<p.L * p.B * p.H, kThreads, bytes, stream>>>(p);
  return cudaGetLastError();
}

template <bool ALIGN>
cudaError_t launch_k(const CommitParams& p, int K, cudaStream_t stream) {
  if (K == 128) return p.Q <= 4 ? launch<128, 4, ALIGN>(p, stream) : launch<128, 8, ALIGN>(p, stream);
  return p.Q <= 4 ? launch<64, 4, ALIGN>(p, stream) : launch<64, 8, ALIGN>(p, stream);
}

}  // namespace

cudaError_t launch_commit(const CommitParams& p, int K, cudaStream_t stream) {
  const bool align = p.final_state_indices != nullptr || p.boundary_state_indices != nullptr;
  return align ? launch_k<true>(p, K, stream) : launch_k<false>(p, K, stream);
}

}  // namespace kda
