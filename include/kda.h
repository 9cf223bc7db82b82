/*
 * kda.h -- C ABI of libkda: the Kimi Delta Attention (KDA) RecoverSSM
 * speculative verify and accepted-state commit on one GB300 (sm_103a).
 *
 * Operations (vLLM pages on the Kimi-K3 RecoverSSM path):
 *   kda_verify  "vllm.models.kimi_k3.nvidia.recoverssm.kernels",
 *               CuteRecoverSSMVerify.__call__: the short causal conv + SiLU
 *               fused in front of the verify of
 *               "vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py",
 *               kda_recoverssm_verify / _kda_recoverssm_verify_kernel
 *               (gate _kda_gate, step _kda_recurrent_step).
 *   kda_commit  same ops page, KDARecoverSSMCommitContext.commit /
 *               _commit_kda_state_kernel, and the kernels page,
 *               cute_recoverssm_commit: all layers folded in one launch.
 *
 * Conventions for every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller.  The
 *     library allocates nothing, keeps no pointer past the call, and never
 *     synchronises (kda_read_device_error is the one exception).
 *   - Kernels are enqueued on `stream` and run asynchronously, in stream order.
 *   - Strides are in ELEMENTS of the buffer's own type.  Innermost dimensions
 *     are contiguous (unit stride) as stated per field.
 *   - A non-zero status means nothing was enqueued; kda_last_error() then
 *     describes the cause (thread-local, valid until the next call).
 *   - Errors that only the device can see (a slot or record row out of range,
 *     a decreasing query_start_loc, a token range past T) skip the affected
 *     (request, head) work item and OR a KDA_DEVERR_* bit into workspace[0];
 *     kda_read_device_error() fetches it.  A commit's workspace may be NULL
 *     (no report); the verify entry points require one (below).
 *   - No device wait is unbounded: a wait that exceeds about one second sets
 *     KDA_DEVERR_TIMEOUT and the work item returns.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *kda_stream_t;

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* a null pointer, a bad size, stride or enum */
    KDA_ERR_UNSUPPORTED = 2,  /* a valid configuration this build does not serve */
    KDA_ERR_MISALIGNED = 3,   /* a static tensor off its required alignment */
    KDA_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
    KDA_ERR_DEVICE = 5        /* kda_read_device_error: the device reported errors */
} kda_status;

typedef enum kda_gate_mode {
    KDA_GATE_SOFTPLUS = 0,    /* g = -exp(A_log) * softplus(raw_g + dt_bias) */
    KDA_GATE_LOWER_BOUND = 1  /* g = lower_bound * sigmoid(exp(A_log) * (raw_g + dt_bias)) */
} kda_gate_mode;

typedef enum kda_conv_layout {
    KDA_CONV_DIM_FIRST = 0,   /* conv state [slots, 3HK, Q+W-2], taps contiguous     */
    KDA_CONV_SEQ_FIRST = 1    /* conv state [slots, Q+W-2, 3HK], channels contiguous */
} kda_conv_layout;

typedef enum kda_dtype { KDA_DTYPE_BF16 = 0, KDA_DTYPE_FP32 = 1 } kda_dtype;

/* Device error bits (workspace[0]). */
enum {
    KDA_DEVERR_SLOT_RANGE = 1,  /* state_indices[b] >= num_slots                     */
    KDA_DEVERR_ROW_RANGE = 2,   /* record row < 0 or >= num_record_rows              */
    KDA_DEVERR_TOKEN_RANGE = 4, /* query_start_loc decreasing, negative, or past T   */
    KDA_DEVERR_TIMEOUT = 8,     /* a bounded device wait gave up                     */
    KDA_DEVERR_MISALIGNED = 16  /* a per-layer table entry off 16-byte alignment     */
};

/*
 * kda_verify -- verify one KDA layer's speculative windows without touching
 * the checkpointed SSM state.
 *
 * For request b: tokens are rows [bos, bos + n) of the activation buffers,
 * bos = query_start_loc[b], n = min(query_start_loc[b+1] - bos, Q); slot
 * s = state_indices[b]; record row r = record_indices ? record_indices[b] : s.
 * If s <= null_block_id the request writes zeros to out[bos .. bos+n) (its
 * heads' columns) and nothing else.  Otherwise, per head h:
 *   1. conv: for each of the head's q, k and v channels c (channel blocks
 *      [0,HK) q, [HK,2HK) k, [2HK,3HK) v; head h owns c = blk*HK + h*K + i),
 *      history = the W-1 stored taps starting at tap a-1 of slot s, where
 *      a = clamp(num_accepted_prev[b], 1, Q) (a = 1 when the pointer is NULL);
 *      seq = history followed by mixed_qkv[bos..bos+n, c];
 *      y_t = bf16_rne(silu(sum_j w[c,j] * seq[t+j])), w[c,W-1] on the newest
 *      input, rounded once from the mathematical value (an fp32 evaluation
 *      with an error bound; the few codes within that bound of a rounding
 *      boundary are recomputed in float-float or double arithmetic);
 *      the slot then stores seq[1 .. W-2+n] at taps 0 .. W-3+n (in place;
 *      later taps are left as they were).
 *   2. q^ = q * rsqrt(|q|^2 + 1e-6) * K^-1/2, k^ = k * rsqrt(|k|^2 + 1e-6),
 *      beta = sigmoid(raw_beta), g per the gate mode (A = exp(A_log[h])).
 *   3. from S = state[s, h] (read only): per token t < n,
 *      S <- S diag(e^g); c = beta (v - S k^); S <- S + c k^T; o = S q^.
 *      out[bos+t, h*V .. h*V+V) = bf16_rne(o); corr[r, h, t, :] = c (fp32);
 *      key_gate[r, h, t, 0..K) = k (the bf16 conv output);
 *      key_gate[r, h, t, K..2K) = raw_gate[bos+t, h*K ..] (bit copy).
 *      Rows and records of tokens t >= n are not written.
 * T == 0 or B == 0 is a no-op returning KDA_OK.
 *
 * Two kernels run, in stream order: the conv pass (one CTA per (request,
 * head): the codes y_t, packed with the raw gate rows, the beta gates
 * sigmoid(raw_beta) and the decays e^g into `scratch`, and the rolled conv
 * state) and the
 * verify proper (persistent, one CTA per SM; it may start while the conv
 * pass drains and waits for it before reading `scratch`).
 * `scratch` is caller-owned device memory of at least
 * kda_verify_scratch_bytes(B, H, K, Q) bytes, 16-byte aligned; its contents
 * between calls are unspecified (calls that may overlap need distinct
 * scratch buffers).  It may be NULL when T == 0.
 *
 * Supported: K == V in {64, 128}, W == 4, 1 <= Q <= 8.  Alignment: state,
 * corr, key_gate, conv_state, conv_weight, A_log and dt_bias must start on
 * 16 bytes, and their slot / row strides must be multiples of 16 bytes
 * (KDA_ERR_MISALIGNED otherwise).  Activation buffers (mixed_qkv, raw_gate,
 * raw_beta, out) need only element alignment: rows at any offset are handled
 * in-kernel.  Distinct requests must use distinct slots and record rows.
 */
typedef struct kda_verify_args {
    int32_t B;                    /* requests                                       */
    int32_t H, K, V;              /* heads, key dim, value dim (K == V)            */
    int32_t Q;                    /* window (spec_query_len)                        */
    int32_t W;                    /* conv width                                     */
    int32_t T;                    /* token rows in the activation buffers, <= B*Q   */
    int32_t null_block_id;        /* slot s is null when s <= null_block_id         */
    int64_t num_slots;            /* slots of the state and conv-state pools        */
    int64_t num_record_rows;      /* rows of corr / key_gate                        */

    const void *mixed_qkv;  int64_t qkv_row_stride;  /* bf16 [T, 3HK], pre-conv       */
    const void *raw_gate;   int64_t gate_row_stride; /* bf16 [T, HK]                  */
    const void *raw_beta;   int64_t beta_row_stride; /* bf16 [T, H]                   */
    void *out;              int64_t out_row_stride;  /* bf16 [T, HV]                  */

    const float *A_log;           /* fp32 [H]                                       */
    const float *dt_bias;         /* fp32 [H*K]                                     */
    int32_t gate_mode;            /* kda_gate_mode                                  */
    float lower_bound;            /* used by KDA_GATE_LOWER_BOUND                   */

    const void *conv_weight;      /* [3HK, W] contiguous, no bias                   */
    int32_t conv_weight_dtype;    /* kda_dtype                                      */
    void *conv_state;             /* bf16, kda_conv_layout, updated in place        */
    int32_t conv_layout;          /* kda_conv_layout                                */
    int64_t conv_slot_stride;     /* elements between slots (>= 3HK*(Q+W-2))         */

    const float *state;           /* fp32 [slots, H, V, K], inner (V*K, K, 1); read only */
    int64_t state_slot_stride;    /* elements between slots (>= H*V*K)              */
    float *corr;                  /* fp32 [rows, H, Q, V], inner contiguous         */
    int64_t corr_row_stride;      /* elements between rows (>= H*Q*V)               */
    void *key_gate;               /* bf16 [rows, H, Q, 2K], inner contiguous        */
    int64_t kg_row_stride;        /* elements between rows (>= H*Q*2K)              */

    const int32_t *query_start_loc;   /* [B+1]                                      */
    const int32_t *state_indices;     /* [B]                                        */
    const int32_t *record_indices;    /* [B] or NULL (records at the state slot)    */
    const int32_t *num_accepted_prev; /* [B] conv read offset, or NULL (a = 1)      */
    int32_t *workspace;               /* kda_workspace_bytes() bytes, zeroed: required */
    void *scratch;                    /* device, >= kda_verify_scratch_bytes(), 16-byte aligned */
    int64_t scratch_bytes;            /* its size in bytes                          */
    int32_t variant;                  /* kda_verify_variant                         */
} kda_verify_args;

/* Which kernel computes the products S0 [X | Y] of the verify.  AUTO picks
 * the faster on GB300 for the window (tensor cores for Q > 4 at K == 128,
 * CUDA cores otherwise); the others force one (tensor cores need K == 128,
 * and the fold runs on the CUDA cores whatever is asked). */
typedef enum kda_verify_variant {
    KDA_VERIFY_AUTO = 0,
    KDA_VERIFY_CUDA_CORE = 1,
    KDA_VERIFY_TCGEN05 = 2
} kda_verify_variant;

/* Bytes of scratch the verify needs: B * H blocks of Q * 12K + 32 bytes (the
 * conv pass's output per (request, head): [Q][2K] bf16 rows q | v, [Q][2K]
 * rows k | gate, 8 fp32 beta gates, then [Q][K] fp32 decays e^g). */
size_t kda_verify_scratch_bytes(int32_t B, int32_t H, int32_t K, int32_t Q);


/*
 * kda_commit -- fold each request's first m accepted verify records into its
 * fp32 state, for all L layers in one launch (in place).
 *
 * m = min(max(num_accepted[b], 0), n), n = min(query_start_loc[b+1] -
 * query_start_loc[b], Q).  Requests with a null slot or m == 0 write nothing.
 * For layer l, head h, with k^_t and g_t recomputed from the key/gate record
 * of token t and c_t its correction record:
 *   S <- S diag(prod_t e^{g_t}) + sum_t c_t (k^_t * prod_{u>t} e^{g_u})^T,
 * which is the verify's running state after m tokens.
 *
 * Per-layer buffers are reached through device tables of L int64 entries:
 * base addresses and slot / row strides (elements).  Every layer shares the
 * inner layouts of kda_verify: state [slots, H, V, K] fp32, corr
 * [rows, H, Q, V] fp32, key_gate [rows, H, Q, 2K] bf16.  Entries must be
 * 16-byte aligned (checked on the device: KDA_DEVERR_MISALIGNED).
 * A_log is fp32 [L, H] and dt_bias fp32 [L, H*K], contiguous.
 * Supported: K == V in {64, 128}, 1 <= Q <= 8, L >= 1.
 */
typedef struct kda_commit_args {
    int32_t L, B, H, K, V, Q;
    int32_t null_block_id;
    int64_t num_slots, num_record_rows;
    const int64_t *state_base;        /* device [L]: fp32 state pool addresses     */
    const int64_t *state_slot_stride; /* device [L]                                */
    const int64_t *corr_base;         /* device [L]: fp32 correction records       */
    const int64_t *corr_row_stride;   /* device [L]                                */
    const int64_t *kg_base;           /* device [L]: bf16 key/gate records         */
    const int64_t *kg_row_stride;     /* device [L]                                */
    const float *A_log;               /* fp32 [L, H]                               */
    const float *dt_bias;             /* fp32 [L, H*K]                             */
    int32_t gate_mode;
    float lower_bound;
    const int32_t *query_start_loc;   /* [B+1] of the verified step                */
    const int32_t *state_indices;     /* [B]                                       */
    const int32_t *record_indices;    /* [B] or NULL (records at the state slot)   */
    const int32_t *num_accepted;      /* [B]                                       */
    int32_t *workspace;               /* zeroed kda_workspace_bytes(), or NULL     */
} kda_commit_args;

/*
 * kda_verify_fold -- the pending commit of the previous step fused into this
 * step's verify of one layer.  This is the deferred form of the hot path
 * ("vllm.models.kimi_k3.nvidia.specialized_decode.recoverssm.state",
 * deferred_recoverssm_verify: the last step's accepted tokens are folded into
 * the checkpoints before the verify; the pages run that fold as a separate
 * commit of all layers).  For each request b with a live slot
 * s = state_indices[b]:
 *   m = min(max(fold->num_accepted[b], 0), n'),
 *   n' = min(fold->query_start_loc[b+1] - fold->query_start_loc[b], Q),
 * and the records of row r' = fold->record_indices ? fold->record_indices[b]
 * : s, tokens t < m, are folded exactly as kda_commit folds them (this
 * layer's A_log, dt_bias and gate mode), the folded state is written back to
 * state[s] (so args->state is WRITTEN by this call), and the verify of this
 * step then runs on it as kda_verify does.  The pending records are read
 * before this step's records are written, so r' may equal this step's record
 * row.  It must not be another request's record row of this step: the
 * requests are verified concurrently, and that request's new records could
 * overwrite row r' before it is read.  A request with n = 0 and m > 0 is
 * folded only.  The result equals kda_commit with the fold arguments
 * followed by kda_verify, up to fp32
 * rounding.  The fold pointers are device arrays ([B+1], [B], [B] or NULL);
 * fold == NULL or fold->query_start_loc == NULL runs the plain verify.  With
 * T == 0 (every window empty) only the folds run, and the activation
 * pointers may be NULL.
 * The fold runs on the CUDA cores whatever args->variant says.  The other
 * arguments and errors are those of kda_verify; a pending record row out of
 * range is a device error (KDA_DEVERR_ROW_RANGE) that skips the item.
 */
typedef struct kda_fold_args {
    const int32_t *query_start_loc;  /* [B+1] of the step whose records are pending */
    const int32_t *num_accepted;     /* [B] its accepted tokens                      */
    const int32_t *record_indices;   /* [B] its record rows, or NULL (the state slot) */
} kda_fold_args;

kda_status kda_verify_fold(const kda_verify_args *args, const kda_fold_args *fold, kda_stream_t stream);

/*
 * kda_commit_align -- kda_commit in the align mode of prefix caching
 * ("vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py",
 * _commit_kda_state_kernel with ALIGN_MODE; the mode is chosen per step in
 * "vllm.models.kimi_k3.nvidia.specialized_decode.recoverssm.state",
 * _build_deferred).  Per (layer, request, head) with a live source slot s and
 * m > 0 as in kda_commit (records read at row r from S = state[s]):
 *   - fs = final_state_indices ? final_state_indices[b] : s; fs at or below
 *     null_block_id writes nothing; otherwise state[fs] = the committed state;
 *   - bs = boundary_state_indices ? boundary_state_indices[b] : null; when
 *     bs is live, state[bs] = the state after the first
 *     R = min(max(boundary_recovery_lens[b], 0), m) tokens (S itself for
 *     R = 0), written before the final state (so fs == bs keeps the final).
 * Slots written must not be read as a source by another request of the same
 * launch.  All three arrays are device [B]; align == NULL or all three NULL
 * is kda_commit.  A final or boundary slot >= num_slots is a device error
 * (KDA_DEVERR_SLOT_RANGE) that skips the item.
 */
typedef struct kda_align_args {
    const int32_t *final_state_indices;     /* [B] or NULL (the source slot)           */
    const int32_t *boundary_state_indices;  /* [B] or NULL (no boundary state)          */
    const int32_t *boundary_recovery_lens;  /* [B], required with boundary slots        */
} kda_align_args;

kda_status kda_commit_align(const kda_commit_args *args, const kda_align_args *align, kda_stream_t stream);

/* Enqueue the verify of one layer (the conv pass, then the verify kernel).
 * Returns before the kernels run.  args->variant selects the products'
 * kernel (kda_verify_variant): at K == 128 the tcgen05 tensor cores (tf32
 * with a hi/lo split of the state, same tolerances) or the CUDA cores.
 * The verify kernel deals its (request, head) items to its CTAs at run time
 * from a ticket counter in args->workspace, which every launch leaves at
 * zero: verify launches that may run at the same time (different streams)
 * need different workspaces. */
kda_status kda_verify(const kda_verify_args *args, kda_stream_t stream);

/*
 * kda_verify_debug -- kda_verify with two test hooks: the failure handling
 * exercised, and the schedule's balance timed.  The pages have no
 * counterpart.
 *   - wait_limit_ns (> 0) replaces the one-second limit of every device wait
 *     of the verify kernel for this call;
 *   - withhold_item (-1: none; else an item b * H + h) is an item whose
 *     inputs the verify kernel's inputs warp never delivers: no copy is
 *     issued and its slot never fills.  The kernel's wait for it gives up
 *     after wait_limit_ns, KDA_DEVERR_TIMEOUT is set in the workspace, the
 *     CTA that owns the item stops (its later items are left unwritten) and
 *     the kernel returns; the other CTAs' items are verified as by kda_verify.
 *     Withholding runs the CUDA-core verify whatever args->variant says;
 *   - cta_times (NULL: none) is a device array of at least 2 * B * H
 *     entries: verify-kernel CTA i writes the global timer (ns) at its start
 *     to entry 2 i and at its finish (after all its roles) to 2 i + 1.  The
 *     kernel has min(B * H, the device's SM count) CTAs; later entries are
 *     left as they were.
 * Everything else is as for kda_verify (the conv pass runs for every item).
 */
typedef struct kda_debug_args {
    int64_t wait_limit_ns;   /* > 0                                      */
    int32_t withhold_item;   /* -1, or an item in [0, B * H)            */
    uint64_t *cta_times;     /* NULL, or device [>= 2 * B * H], 8-aligned */
} kda_debug_args;

kda_status kda_verify_debug(const kda_verify_args *args, const kda_debug_args *debug, kda_stream_t stream);

/* Enqueue the commit of all layers (one kernel launch). */
kda_status kda_commit(const kda_commit_args *args, kda_stream_t stream);

/* Allocation-free commit.  The pages have no counterpart to this entry point:
 * their commit context keeps the per-layer tables in device memory it
 * allocates once (KDARecoverSSMCommitContext.create).  It serves callers that
 * cannot allocate device memory: code running where a device allocator is
 * not available or not allowed (inside an allocator callback, a memory pool
 * that must not grow, or an embedding runtime that owns all device memory).
 *
 * args is read as for kda_commit, except that the six per-layer tables
 * (state_base, state_slot_stride, corr_base, corr_row_stride, kg_base,
 * kg_row_stride) are HOST arrays of L entries, read during the call into the
 * launch parameters of a small kernel that writes them, in stream order, into
 * a library-owned static device scratch of KDA_NOALLOC_MAX_LAYERS layers
 * (6 x 64 int64 = 3 KB); then the kda_commit kernel runs on it.  Two kernel
 * launches, no copy from host memory: the call allocates nothing, on the host
 * or the device, keeps no pointer to the host tables and does not wait for
 * the stream.
 *   - L > KDA_NOALLOC_MAX_LAYERS: KDA_ERR_UNSUPPORTED, nothing enqueued.
 *   - The first call on a device does the set-up: it resolves the scratch's
 *     device address (cudaGetSymbolAddress), which may load the module.
 *     Recording this call in a CUDA graph is not tested.
 *   - Nothing in the scratch has to start at zero: each call writes every
 *     table entry its kernel reads, before the kernel, in stream order.  The
 *     optional workspace is the caller's and is used as for kda_commit.
 *   - There is one scratch per device and process: calls whose kernels can
 *     overlap (different streams, or threads without a common stream order)
 *     race on it.  Serialise them. */
#define KDA_NOALLOC_MAX_LAYERS 64
kda_status kda_commit_noalloc(const kda_commit_args *args, kda_stream_t stream);

/* Bytes of device workspace (int32-aligned, zeroed by the caller before
 * first use): the error report, into which the kernels OR bits, and the
 * verify's ticket counter, which each verify launch returns to zero. */
size_t kda_workspace_bytes(void);

/* Synchronise `stream`, copy workspace[0] into *flags, and return KDA_OK if
 * it is zero, KDA_ERR_DEVICE if not (KDA_ERR_CUDA if the copy failed). */
kda_status kda_read_device_error(const int32_t *workspace, kda_stream_t stream, int32_t *flags);

/* Description of the last non-OK status returned on this thread. */
const char *kda_last_error(void);

/* ABI version of this header (bumped on any layout change). */
int32_t kda_abi_version(void);

#define KDA_ABI_VERSION 3

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
