/*
 * dspark_oracle.h -- plain, slow CPU oracle for one DSpark draft round.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this code; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do. It shares no code, header, table or helper with the
 * CUDA library: it has its own Philox4x32-10 and its own arithmetic, all in
 * IEEE double precision, written as the plain definitions from
 * "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
 * Generation" (arXiv:2607.05147) as described on the pages it was built from:
 *   - semi-autoregressive factorisation, eq. (4); Markov bias, eq. (5);
 *     RNN head, eq. (6): z_k = [s_{k-1}; W_1[x_{k-1}]; h_k], s_k = g s_{k-1} + (1 - g) tanh(W_c z_k)
 *     with g = sigmoid(W_g z_k), s_0 = 0, B_k = W_2^T tanh(W_o z_k);
 *   - confidence head, eq. (7); survival products a_j = prod c_i;
 *   - Algorithm 1 (hardware-aware prefix scheduler) and the asynchronous
 *     capacity variant (section 5.2 of the paper);
 *   - rejection-sampling verification (Leviathan et al. 2023), the residual
 *     norm(max(0, p_t - p_d)) and the bonus token (dspark_cycle sketch,
 *     steps 5-6, on the caijizhuo.github.io page);
 *   - the static confidence-threshold admission used as the ablation baseline
 *     (zhongzhuzhou.org notes, figure 5 threshold sweep);
 *   - sequential temperature scaling of the confidences (same notes, "STS");
 *   - the flattened variable-length verify batch (same notes, physical
 *     execution without padding);
 *   - greedy decoding at temperature 0 (same notes, FAQ on temperature 0):
 *     the draft takes the arg-max of its logits, and acceptance is an exact
 *     match with the target's arg-max.
 * Every pointer is a host pointer owned by the caller.
 */
#ifndef DSPARK_ORACLE_H
#define DSPARK_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types accepted for tensor inputs */
enum { DSO_F32 = 0, DSO_BF16 = 1, DSO_F64 = 2 };

/* sequential heads: the Markov bias of eq. (5) or the gated recurrent state of eq. (6) */
enum { DSO_HEAD_MARKOV = 0, DSO_HEAD_RNN = 1 };

/* scheduler modes */
enum { DSO_SCHED_SYNC = 0, DSO_SCHED_ASYNC_CAPACITY = 1, DSO_SCHED_FULL_SCAN = 2, DSO_SCHED_THRESHOLD = 3 };

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): out = Philox(ctr, key). */
void dso_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* One uniform in (0,1) for a random purpose: counter (e>>2, pos, req, (round<<3)|purpose),
 * key (seed lo, seed hi), output word e&3, u = (2*(x>>9)+1) * 2^-24. */
double dso_uniform(uint64_t seed, uint64_t round, uint32_t purpose, uint32_t req, uint32_t pos,
                   uint32_t elem);

typedef struct {
    int R, gamma_max, V, r, d, dtype;   /* dtype of U, E, W, h */
    const int32_t* gamma;               /* [R] per-request gamma_r, or NULL = all gamma_max */
    const int32_t* req_ids;             /* [R] request ids used in random counters, NULL = 0..R-1 */
    const void* U;                      /* [R][gamma_max][V] base logits */
    const void* E;                      /* [V][r]  W_1 of eq. (5) */
    const void* W;                      /* [r][V]  W_2 of eq. (5) */
    const void* h;                      /* [R][gamma_max][d] draft hidden states */
    const float* w_h;                   /* [d]  confidence weights on h_k */
    const float* w_e;                   /* [r]  confidence weights on W_1[x] */
    float b;                            /* confidence bias */
    const float* temperature;           /* [R] */
    const int32_t* anchor;              /* [R] x_0 */
    uint64_t seed, round;
    int conf_token;                     /* 0: W_1[x_{k-1}] (eq. 7); 1: W_1[x_k] */
    int bias_first;                     /* 1: B_1 = W_1[x_0] W_2; 0: B_1 = 0 */
    int noise_block;                    /* vocabulary block width of the two-level Gumbel-max */
    const int32_t* forced_tokens;       /* [R][gamma_max] or NULL: committed tokens to condition on */
    /* outputs, all [R][gamma_max] */
    int32_t* tokens;                    /* the oracle's own draw at each position (-1 past gamma_r) */
    double* conf;                       /* c_k */
    double* surv;                       /* a_k = prod_{i<=k} c_i */
    double* lse;                        /* log sum_v exp((U_k + B_k)(v) / T) */
    double* logit;                      /* (U_k + B_k)(x_k) / T at the committed token */
    double* gap1;                       /* top-two gap of the block-level perturbed values */
    double* gap2;                       /* top-two gap of the element-level perturbed values */
    const double* sts_temp;             /* [gamma_max] or NULL: per-position temperature of the confidence
                                           logit (sequential temperature scaling), c_k = sigmoid(l_k / t_k) */
    int head;                           /* DSO_HEAD_MARKOV (eq. 5) or DSO_HEAD_RNN (eq. 6) */
    const void* W_rnn;                  /* [3r][2r+d] (dtype): rows W_g, then W_c, then W_o (RNN head) */
    double* a_rows;                     /* [R][gamma_max][r] or NULL: out, the bias operand of each step
                                           (W_1[x_{k-1}] for the Markov head, tanh(W_o z_k) for the RNN head) */
    float* logp;                        /* [R][gamma_max][V] or NULL: out, the draft distribution of each
                                           active position, log p_d(v) = l_k(v) - lse (a point mass at the
                                           committed token for temperature 0); 0 past gamma_r */
} dso_sample_args;

int dso_sample_block(const dso_sample_args* a);

typedef struct {
    int P;                              /* independent scheduling problems */
    int R, gamma_max;
    const int32_t* gamma;               /* [P][R] or NULL */
    const double* surv;                 /* [P][R][gamma_max] current survivals a_{r,j} */
    const double* surv_capacity;        /* [P][R][gamma_max] survivals two rounds old (async) */
    const double* sps;                  /* [n_sps], sps[B-1] = SPS(B) */
    int n_sps;
    int mode;
    /* outputs */
    int32_t* keep;                      /* [P][R] l_r */
    double* theta_best;                 /* [P] */
    int32_t* admitted;                  /* [P] */
    int32_t* capacity;                  /* [P] K (async), else -1 */
    int32_t* pool;                      /* [P] |E| */
    double* min_margin;                 /* [P] smallest relative margin of a decisive comparison */
    double* theta_curve;                /* [P][R*gamma_max+1] Theta_m of the (current) sorted pool for
                                           m = 0..|pool|, NaN beyond; may be NULL */
    double threshold;                   /* DSO_SCHED_THRESHOLD: admit (r, j) iff a_{r,j} >= threshold */
} dso_schedule_args;

int dso_schedule(const dso_schedule_args* a);

typedef struct {
    int R, gamma_max, V, r, dtype;      /* dtype of target, U, E, W */
    const int32_t* gamma;               /* [R] or NULL */
    const int32_t* req_ids;             /* [R] or NULL */
    const void* target;                 /* [R][gamma_max+1][V]; row i is the target's distribution for draft position i */
    const void* U;
    const void* E;
    const void* W;
    const int32_t* anchor;              /* [R] */
    const int32_t* tokens;              /* [R][gamma_max] draft tokens */
    const double* draft_lse;            /* [R][gamma_max] */
    const double* draft_logit;          /* [R][gamma_max] */
    const int32_t* keep;                /* [R] l_r */
    const float* temperature;           /* [R] */
    uint64_t seed, round;
    int bias_first, noise_block;
    const double* a_rows;               /* [R][gamma_max][r] or NULL: bias operand of each draft position
                                           (from dso_sample_block); NULL = W_1[x_{k-1}] (Markov head) */
    double res_rel_eps;                 /* relative error of the probabilities assumed for rgap1, rgap2 (0:
                                           rgap equals gap) */
    /* outputs */
    int32_t* accepted;                  /* [R] n_r */
    int32_t* next_token;                /* [R] residual or bonus token */
    int32_t* resampled;                 /* [R] 1 = residual, 0 = bonus */
    double* accept_margin;              /* [R][gamma_max] |log u - log(p_t/p_d)| of each tested position, NaN if untested */
    double* lse_t;                      /* [R][gamma_max+1] target log-normaliser of rows 0..l_r, NaN otherwise */
    double* gap1;                       /* [R] block-level top-two gap of the final draw */
    double* gap2;                       /* [R] element-level top-two gap of the final draw */
    double* rgap1;                      /* [R] block-level margin of the final draw when every probability
                                           carries a relative error up to res_rel_eps (residual draws; gap1
                                           otherwise): the winner's lowest value minus any other's highest */
    double* rgap2;                      /* [R] same, element level inside the winning block */
} dso_verify_args;

int dso_verify(const dso_verify_args* a);

/* Ragged verify batch: the admitted prefixes of all requests flattened into one token stream
 * (request r contributes its anchor, then its keep[r] admitted draft tokens), with the request
 * id and the causal position (0 for the anchor, j for draft token j) of every flat token and
 * the start offset of every request (offsets[R] = total). Entries past the total are -1.
 * Returns 1 if a keep value lies outside [0, gamma_max]. */
typedef struct {
    int R, gamma_max;
    const int32_t* keep;                /* [R] */
    const int32_t* anchor;              /* [R] */
    const int32_t* tokens;              /* [R][gamma_max] */
    int32_t* flat_tokens;               /* [R*(gamma_max+1)] */
    int32_t* flat_request;              /* [R*(gamma_max+1)] */
    int32_t* flat_position;             /* [R*(gamma_max+1)] */
    int32_t* offsets;                   /* [R+1] */
} dso_assemble_args;

int dso_assemble(const dso_assemble_args* a);

#ifdef __cplusplus
}
#endif
#endif
