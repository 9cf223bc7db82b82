/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU restatement of the Kimi Delta Attention
 * (KDA) RecoverSSM speculative verify and of its accepted-state commit.  It is
 * the oracle that the CUDA path is checked against.  Only the test-suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * library never does, and the two share no code, header or helper.
 *
 * Sources restated here (vLLM pages on the Kimi-K3 RecoverSSM path):
 *   [ops]     "vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py":
 *             _kda_gate, _kda_recurrent_step, _kda_recoverssm_verify_kernel,
 *             _commit_kda_state_kernel, kda_recoverssm_verify,
 *             KDARecoverSSMCommitContext.create / .commit.
 *   [kernels] "vllm.models.kimi_k3.nvidia.recoverssm.kernels":
 *             CuteRecoverSSMVerify.__call__ (conv fused into the verify,
 *             conv_state [slots, 3HK, Q+2] or [slots, Q+2, 3HK]),
 *             CuteRecoverSSMVerify._bulk_copy_aligned (conv_len = Q + W - 2).
 *   [state]   "vllm.models.kimi_k3.nvidia.specialized_decode.recoverssm.state":
 *             deferred_recoverssm_verify (conv -> split q/k/v -> verify,
 *             records written to record rows).
 *
 * Every quantity after the convolution is computed in double from the exact
 * values of the bf16 / fp32 inputs.  Values the method stores in a narrower
 * type are rounded once, from the double result: outputs and key/gate records
 * to bf16 (round to nearest even), corrections and committed states to fp32.
 *
 * The convolution output is the one place where floating point decides a
 * stored code: the bf16 value that every later step consumes.  The oracle
 * takes that decision from the plain definition: y = sum_j w_j x_j in double
 * (each product of a bf16 input and a bf16 or fp32 weight is exact in double),
 * SiLU(y) = y / (1 + e^-y) with the C library's exp, and one rounding of that
 * double to bf16 (nearest; an exact tie, which only arises where double
 * cannot tell SiLU(y) from a large y, goes toward zero, the side the exact
 * value lies on).  The pins check the codes against an exact
 * (arbitrary-precision) evaluation, including inputs placed next to a bf16
 * rounding boundary and large sums that fall exactly on one.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - conv taps: w[c, W-1] multiplies the newest token (standard causal
 *     depthwise convolution), no bias, SiLU activation;
 *   - conv history: the W-1 stored taps starting at offset a-1, where
 *     a = clamp(num_accepted_prev[b], 1, Q) (1 when no counts are given);
 *     after the verify the slot stores seq[1 .. W-2+n] at taps 0 .. W-3+n
 *     (seq = history followed by the n window inputs), later taps untouched;
 *   - the conv output is rounded to bf16 before the recurrence uses it;
 *   - n = min(query_len, Q); tokens past Q are ignored; n <= 0 writes nothing;
 *   - a request whose slot is <= null_block_id writes zero outputs for its
 *     tokens and nothing else;
 *   - records go to row record_indices[b] (state_indices[b] when absent);
 *   - commit length m = min(max(num_accepted[b], 0), n).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Scalar conversions                                                         */
/* ------------------------------------------------------------------------- */

/* Exact value of a bf16 bit pattern (bf16 is the top half of an fp32). */
static double bf16_value(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Round a double straight to bf16, nearest, without passing through fp32
 * (which would round twice).  bf16 keeps 8 significant bits and shares fp32's
 * exponent range; its subnormal quantum is 2^-133.  A value exactly halfway
 * between two codes goes to the even one, or, with ties_down, to the one
 * nearer zero. */
static uint16_t bf16_round_ties(double x, int ties_down) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    if (isinf(ax)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(ax, &e); /* ax = f * 2^e, f in [0.5, 1) */
    int qexp = e - 8;
    if (qexp < -133) qexp = -133;
    double sc = ldexp(ax, -qexp); /* exact: a power-of-two scaling */
    double rq = nearbyint(sc);    /* ties to even */
    if (ties_down && sc - floor(sc) == 0.5) rq = floor(sc);
    double r = ldexp(rq, qexp);
    if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80);
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(sign | (uint16_t)(w >> 16));
}

static uint16_t bf16_round(double x) { return bf16_round_ties(x, 0); }

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------- */
/* The convolution output                                                     */
/* ------------------------------------------------------------------------- */

static double silu(double y) { return y / (1.0 + exp(-y)); }

/* The bf16 code of SiLU(y), correctly rounded.  For y > 0, SiLU(y) =
 * y - y e^-y / (1 + e^-y) lies strictly below y; past y of about 37, 1 + e^-y
 * rounds to 1 in double and the double SiLU equals y itself.  A y exactly
 * halfway between two codes then stands for a value just below the midpoint,
 * whose code is the one nearer zero, whichever of the two is even.  (SiLU(y)
 * itself is never a midpoint for y != 0: e^-y is transcendental.) */
static uint16_t silu_code(double y) {
    double s = silu(y);
    return bf16_round_ties(s, y > 0.0 && s == y);
}

/* [kernels] CuteRecoverSSMVerify.__call__ / [state] deferred_recoverssm_verify
 * (causal_conv1d_update with activation "silu"): y = sum_j w_j x_j over the W
 * taps, oldest first (w[W-1] on the newest input), SiLU, and the bf16 code of
 * the result.  Every product is exact in double. */
static uint16_t conv_silu_code(const double *w, const double *x, int W) {
    double y = 0.0;
    for (int j = 0; j < W; ++j) y += w[j] * x[j];
    return silu_code(y);
}

/* [ops] _kda_gate: gate_input = raw_g + dt_bias; the bounded form is
 * lower_bound * sigmoid(A * gate_input); otherwise -A * softplus(gate_input)
 * with softplus(x) = x for x > 20 and log(1 + e^x) below. */
static double kda_gate(double raw_g, double dt_bias, double A,
                       int use_lower_bound, double lower_bound) {
    double u = raw_g + dt_bias;
    if (use_lower_bound) return lower_bound * sigmoid(A * u);
    double sp = (u > 20.0) ? u : log(1.0 + exp(u));
    return -A * sp;
}

static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* ------------------------------------------------------------------------- */
/* Verify                                                                     */
/* ------------------------------------------------------------------------- */

typedef struct {
    int32_t B, H, K, V, Q, W, T, null_block_id;
    int64_t num_slots, num_record_rows;
    const uint16_t *mixed_qkv;  int64_t qkv_row_stride;  /* [T, 3HK] pre-conv */
    const uint16_t *raw_gate;   int64_t gate_row_stride; /* [T, HK]           */
    const uint16_t *raw_beta;   int64_t beta_row_stride; /* [T, H]            */
    const float *A_log;                                  /* [H]               */
    const float *dt_bias;                                /* [H*K]             */
    int32_t use_lower_bound;    double lower_bound;
    const void *conv_weight;    int32_t conv_weight_is_fp32; /* [3HK, W]      */
    uint16_t *conv_state;       int32_t conv_dim_first; int64_t conv_slot_stride;
    const float *state;         int64_t state_slot_stride;   /* [slots,H,V,K] */
    const int32_t *query_start_loc;   /* [B+1] */
    const int32_t *state_indices;     /* [B]   */
    const int32_t *record_indices;    /* [B] or NULL */
    const int32_t *num_accepted_prev; /* [B] or NULL */
    const uint8_t *item_mask;         /* [B*H] or NULL: compute only these */
    uint16_t *out;              int64_t out_row_stride;  /* [T, HV] bf16     */
    double *out_exact;                                   /* [T, HV] or NULL  */
    float *corr;                int64_t corr_row_stride; /* [rows,H,Q,V]     */
    double *corr_exact;                                  /* [rows,H,Q,V] or NULL */
    uint16_t *key_gate;         int64_t kg_row_stride;   /* [rows,H,Q,2K]    */
    double *running_state;      /* [B,H,Q,V,K] or NULL: S after each token */
    double *post_conv;          /* [T, 3HK] or NULL: conv outputs (bf16 values) */
    int32_t num_threads;
} kda_oracle_verify_args;

enum { ORACLE_OK = 0, ORACLE_BAD_ARGS = 1, ORACLE_BAD_DATA = 2 };

/* Index of conv-state element (slot s, channel c, tap j). */
static int64_t conv_index(const kda_oracle_verify_args *a, int64_t s, int64_t c, int64_t j) {
    int64_t C = 3LL * a->H * a->K;
    int64_t Lc = a->Q + a->W - 2;
    return a->conv_dim_first ? s * a->conv_slot_stride + c * Lc + j
                             : s * a->conv_slot_stride + j * C + c;
}

static double conv_weight_value(const kda_oracle_verify_args *a, int64_t c, int j) {
    if (a->conv_weight_is_fp32) return (double)((const float *)a->conv_weight)[c * a->W + j];
    return bf16_value(((const uint16_t *)a->conv_weight)[c * a->W + j]);
}

/* One (request b, head h) of the verify; returns ORACLE_BAD_DATA on an
 * out-of-range slot / row / token range (nothing is written then). */
static int verify_item(const kda_oracle_verify_args *a, int b, int h) {
    const int H = a->H, K = a->K, V = a->V, Q = a->Q, W = a->W;
    const int64_t HK = (int64_t)H * K;
    int64_t bos = a->query_start_loc[b], eos = a->query_start_loc[b + 1];
    int64_t len = eos - bos;
    if (len <= 0) return len < 0 ? ORACLE_BAD_DATA : ORACLE_OK;
    int n = len < Q ? (int)len : Q;
    if (bos < 0 || bos + n > a->T) return ORACLE_BAD_DATA;
    int64_t s = a->state_indices[b];

    /* [ops] _kda_recoverssm_verify_kernel, null-slot branch: zero outputs. */
    if (s <= a->null_block_id) {
        for (int t = 0; t < n; ++t)
            for (int v = 0; v < V; ++v) {
                a->out[(bos + t) * a->out_row_stride + (int64_t)h * V + v] = 0;
                if (a->out_exact) a->out_exact[(bos + t) * (int64_t)H * V + (int64_t)h * V + v] = 0.0;
            }
        return ORACLE_OK;
    }
    int64_t r = a->record_indices ? a->record_indices[b] : s;
    if (s >= a->num_slots || r < 0 || r >= a->num_record_rows) return ORACLE_BAD_DATA;
    int acc = a->num_accepted_prev ? clampi(a->num_accepted_prev[b], 1, Q) : 1;

    /* ---- short causal conv + SiLU over this head's q, k and v channels ----
     * [kernels] CuteRecoverSSMVerify.__call__ (the conv is fused into the
     * verify); [state] deferred_recoverssm_verify (conv output split into
     * q | k | v, each "n (h d)" head-contiguous). */
    const int nch = 3 * K;
    double *post = (double *)malloc(sizeof(double) * (size_t)nch * (size_t)n);
    uint16_t *seq = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(W - 1 + n));
    for (int g = 0; g < 3; ++g) {
        for (int i = 0; i < K; ++i) {
            int64_t c = g * HK + (int64_t)h * K + i;
            for (int j = 0; j < W - 1; ++j)
                seq[j] = a->conv_state[conv_index(a, s, c, acc - 1 + j)];
            for (int t = 0; t < n; ++t)
                seq[W - 1 + t] = a->mixed_qkv[(bos + t) * a->qkv_row_stride + c];
            for (int t = 0; t < n; ++t) {
                double wv[8], xv[8];
                for (int j = 0; j < W; ++j) {
                    wv[j] = conv_weight_value(a, c, j);
                    xv[j] = bf16_value(seq[t + j]);
                }
                post[(size_t)(g * K + i) * n + t] = bf16_value(conv_silu_code(wv, xv, W));
            }
            /* rolled state: taps 0 .. W-3+n <- seq[1 .. W-2+n] */
            for (int j = 0; j < W - 2 + n; ++j)
                a->conv_state[conv_index(a, s, c, j)] = seq[j + 1];
        }
    }
    free(seq);
    if (a->post_conv)
        for (int g = 0; g < 3; ++g)
            for (int i = 0; i < K; ++i)
                for (int t = 0; t < n; ++t)
                    a->post_conv[(bos + t) * 3 * HK + g * HK + (int64_t)h * K + i] =
                        post[(size_t)(g * K + i) * n + t];

    /* ---- gated delta rule over the window ---- [ops] verify kernel + step */
    double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
    const float *S0 = a->state + s * a->state_slot_stride + (int64_t)h * V * K;
    for (int64_t e = 0; e < (int64_t)V * K; ++e) S[e] = (double)S0[e];
    double A = exp((double)a->A_log[h]);
    double *kn = (double *)malloc(sizeof(double) * K);
    double *qn = (double *)malloc(sizeof(double) * K);
    double *eg = (double *)malloc(sizeof(double) * K);
    double *corr = (double *)malloc(sizeof(double) * V);

    for (int t = 0; t < n; ++t) {
        const int64_t tok = bos + t;
        double kk = 0.0, qq = 0.0;
        for (int k = 0; k < K; ++k) {
            double qv = post[(size_t)(0 * K + k) * n + t];
            double kv = post[(size_t)(1 * K + k) * n + t];
            qq += qv * qv;
            kk += kv * kv;
        }
        double kscale = 1.0 / sqrt(kk + 1e-6);
        double qscale = 1.0 / sqrt(qq + 1e-6) * pow((double)K, -0.5);
        for (int k = 0; k < K; ++k) {
            kn[k] = post[(size_t)(1 * K + k) * n + t] * kscale;
            qn[k] = post[(size_t)(0 * K + k) * n + t] * qscale;
            double rg = bf16_value(a->raw_gate[tok * a->gate_row_stride + (int64_t)h * K + k]);
            eg[k] = exp(kda_gate(rg, (double)a->dt_bias[(int64_t)h * K + k], A,
                                 a->use_lower_bound, a->lower_bound));
        }
        double beta = sigmoid(bf16_value(a->raw_beta[tok * a->beta_row_stride + h]));

        for (int v = 0; v < V; ++v) {
            double *row = S + (size_t)v * K;
            double p = 0.0;
            for (int k = 0; k < K; ++k) {
                row[k] *= eg[k];            /* S <- S diag(e^g) */
                p += row[k] * kn[k];        /* (S k^)[v]        */
            }
            double vv = post[(size_t)(2 * K + v) * n + t];
            corr[v] = (vv - p) * beta;      /* c = sigma(raw_beta)(v - S k^) */
            double o = 0.0;
            for (int k = 0; k < K; ++k) {
                row[k] += corr[v] * kn[k];  /* S <- S + c k^T   */
                o += row[k] * qn[k];        /* o = S q^         */
            }
            a->out[tok * a->out_row_stride + (int64_t)h * V + v] = bf16_round(o);
            if (a->out_exact) a->out_exact[tok * (int64_t)H * V + (int64_t)h * V + v] = o;
        }
        /* verify records: correction (fp32) and key/gate (k | raw_g). */
        int64_t cbase = r * a->corr_row_stride + ((int64_t)h * Q + t) * V;
        for (int v = 0; v < V; ++v) {
            a->corr[cbase + v] = (float)corr[v];
            if (a->corr_exact)
                a->corr_exact[(r * H + h) * (int64_t)Q * V + (int64_t)t * V + v] = corr[v];
        }
        int64_t kbase = r * a->kg_row_stride + ((int64_t)h * Q + t) * 2 * K;
        for (int k = 0; k < K; ++k) {
            a->key_gate[kbase + k] = bf16_round(post[(size_t)(1 * K + k) * n + t]);
            a->key_gate[kbase + K + k] = a->raw_gate[tok * a->gate_row_stride + (int64_t)h * K + k];
        }
        if (a->running_state) {
            double *dst = a->running_state + (((int64_t)b * H + h) * Q + t) * (int64_t)V * K;
            memcpy(dst, S, sizeof(double) * (size_t)V * K);
        }
    }
    free(kn); free(qn); free(eg); free(corr); free(S); free(post);
    return ORACLE_OK;
}

int kda_oracle_verify(const kda_oracle_verify_args *a) {
    if (!a || a->B < 0 || a->H <= 0 || a->K <= 0 || a->V != a->K || a->Q <= 0 || a->W < 2 || a->W > 8)
        return ORACLE_BAD_ARGS;
    int status = ORACLE_OK;
    const int items = a->B * a->H;
#ifdef _OPENMP
    int nt = a->num_threads > 0 ? a->num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(max : status)
#endif
    for (int it = 0; it < items; ++it) {
        if (a->item_mask && !a->item_mask[it]) continue;
        int st = verify_item(a, it / a->H, it % a->H);
        if (st > status) status = st;
    }
    return status;
}

/* ------------------------------------------------------------------------- */
/* Commit                                                                     */
/* ------------------------------------------------------------------------- */

typedef struct {
    int32_t B, H, K, V, Q, null_block_id;
    int64_t num_slots, num_record_rows;
    float *state;               int64_t state_slot_stride; /* in place        */
    double *state_exact;        /* [B,H,V,K] or NULL: unrounded new states    */
    const float *corr;          int64_t corr_row_stride;   /* [rows,H,Q,V]    */
    const uint16_t *key_gate;   int64_t kg_row_stride;     /* [rows,H,Q,2K]   */
    const float *A_log;         /* this layer's [H]   */
    const float *dt_bias;       /* this layer's [H*K] */
    int32_t use_lower_bound;    double lower_bound;
    const int32_t *query_start_loc, *state_indices, *record_indices, *num_accepted;
    const uint8_t *item_mask;   /* [B*H] or NULL */
    int32_t num_threads;
    /* align mode (prefix caching), all [B] or NULL: the slot the committed
     * state goes to (NULL: the source slot), and a boundary slot that receives
     * the state after the first boundary_recovery_lens[b] of the m tokens */
    const int32_t *final_state_indices, *boundary_state_indices, *boundary_recovery_lens;
    double *boundary_exact;     /* [B,H,V,K] or NULL: unrounded boundary states */
} kda_oracle_commit_args;

/* [ops] _commit_kda_state_kernel: the accepted state is the verify's running
 * state after m tokens.  Each recorded step is replayed in order from the
 * stored records: k^ and the gate are recomputed from the key/gate record,
 * c is the stored correction, and S <- S diag(e^g) + c k^T.
 * Align mode (the kernel's ALIGN_MODE): the state after the tokens before the
 * boundary recovery length R also goes to the boundary slot when that slot is
 * live, and the committed state goes to the final slot; a final slot at or
 * below the null block writes nothing. */
static int commit_item(const kda_oracle_commit_args *a, int b, int h) {
    const int K = a->K, V = a->V, Q = a->Q;
    int64_t s = a->state_indices[b];
    if (s <= a->null_block_id) return ORACLE_OK;
    int64_t len = (int64_t)a->query_start_loc[b + 1] - a->query_start_loc[b];
    int n = len < 0 ? 0 : (len < Q ? (int)len : Q);
    int m = a->num_accepted[b] < 0 ? 0 : a->num_accepted[b];
    if (m > n) m = n;
    if (m == 0) return ORACLE_OK;
    int64_t r = a->record_indices ? a->record_indices[b] : s;
    if (s >= a->num_slots || r < 0 || r >= a->num_record_rows) return ORACLE_BAD_DATA;
    const int64_t fs = a->final_state_indices ? a->final_state_indices[b] : s;
    if (fs <= a->null_block_id) return ORACLE_OK;
    const int64_t bs = a->boundary_state_indices ? a->boundary_state_indices[b] : a->null_block_id;
    if (fs >= a->num_slots || bs >= a->num_slots) return ORACLE_BAD_DATA;
    const int R = a->boundary_recovery_lens ? a->boundary_recovery_lens[b] : 0;

    float *S0 = a->state + s * a->state_slot_stride + (int64_t)h * V * K;
    double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
    double *Sb = (double *)malloc(sizeof(double) * (size_t)V * K);
    double *kn = (double *)malloc(sizeof(double) * K);
    double *eg = (double *)malloc(sizeof(double) * K);
    for (int64_t e = 0; e < (int64_t)V * K; ++e) S[e] = Sb[e] = (double)S0[e];
    double A = exp((double)a->A_log[h]);
    for (int t = 0; t < m; ++t) {
        const uint16_t *kg = a->key_gate + r * a->kg_row_stride + ((int64_t)h * Q + t) * 2 * K;
        const float *c = a->corr + r * a->corr_row_stride + ((int64_t)h * Q + t) * V;
        double kk = 0.0;
        for (int k = 0; k < K; ++k) kk += bf16_value(kg[k]) * bf16_value(kg[k]);
        double kscale = 1.0 / sqrt(kk + 1e-6);
        for (int k = 0; k < K; ++k) {
            kn[k] = bf16_value(kg[k]) * kscale;
            eg[k] = exp(kda_gate(bf16_value(kg[K + k]), (double)a->dt_bias[(int64_t)h * K + k], A,
                                 a->use_lower_bound, a->lower_bound));
        }
        for (int v = 0; v < V; ++v)
            for (int k = 0; k < K; ++k)
                S[(size_t)v * K + k] = S[(size_t)v * K + k] * eg[k] + (double)c[v] * kn[k];
        if (t + 1 == R)  /* the state after the tokens before the boundary */
            for (int64_t e = 0; e < (int64_t)V * K; ++e) Sb[e] = S[e];
    }
    if (R > m)  /* the boundary lies past the committed tokens: it holds them all */
        for (int64_t e = 0; e < (int64_t)V * K; ++e) Sb[e] = S[e];
    const int64_t off = (int64_t)h * V * K;
    if (bs > a->null_block_id) {  /* written first: a final slot equal to it wins */
        float *Bst = a->state + bs * a->state_slot_stride + off;
        for (int64_t e = 0; e < (int64_t)V * K; ++e) {
            Bst[e] = (float)Sb[e];
            if (a->boundary_exact) a->boundary_exact[((int64_t)b * a->H + h) * (int64_t)V * K + e] = Sb[e];
        }
    }
    float *F = a->state + fs * a->state_slot_stride + off;
    for (int64_t e = 0; e < (int64_t)V * K; ++e) {
        F[e] = (float)S[e];
        if (a->state_exact) a->state_exact[((int64_t)b * a->H + h) * (int64_t)V * K + e] = S[e];
    }
    free(S); free(Sb); free(kn); free(eg);
    return ORACLE_OK;
}

int kda_oracle_commit(const kda_oracle_commit_args *a) {
    if (!a || a->B < 0 || a->H <= 0 || a->K <= 0 || a->V <= 0 || a->Q <= 0) return ORACLE_BAD_ARGS;
    int status = ORACLE_OK;
    const int items = a->B * a->H;
#ifdef _OPENMP
    int nt = a->num_threads > 0 ? a->num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(max : status)
#endif
    for (int it = 0; it < items; ++it) {
        if (a->item_mask && !a->item_mask[it]) continue;
        int st = commit_item(a, it / a->H, it % a->H);
        if (st > status) status = st;
    }
    return status;
}

/* Exposed for the pin tests: the scalar pieces on their own. */
uint16_t kda_oracle_bf16_round(double x) { return bf16_round(x); }
double kda_oracle_gate(double raw_g, double dt_bias, double A, int use_lower_bound, double lower_bound) {
    return kda_gate(raw_g, dt_bias, A, use_lower_bound, lower_bound);
}
/* w, x: [n, W] row-major, taps oldest first; out: [n] bf16 codes. */
void kda_oracle_conv_silu_bf16(const double *w, const double *x, uint16_t *out, int64_t n, int W) {
    for (int64_t i = 0; i < n; ++i) out[i] = conv_silu_code(w + i * W, x + i * W, W);
}
