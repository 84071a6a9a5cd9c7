/*
 * dspark.h -- C ABI of libdspark: the batched hot path of one DSpark
 * speculative-decoding round over R concurrent requests on one GB300 GPU.
 *
 * Method: "DSpark: Confidence-Scheduled Speculative Decoding with
 * Semi-Autoregressive Generation" (arXiv:2607.05147), as described on the
 * caijizhuo.github.io page (sections 2-4: serial sampling loop, survival /
 * expected-length / throughput table, "dspark_cycle" and "admit" sketches) and
 * the zhongzhuzhou.org reading notes (eq. 4-5 Markov head, eq. 7 confidence
 * head, Algorithm 1, Appendix A, section 5.2 asynchronous capacity).
 *
 * Conventions shared by every call
 *  - Every tensor pointer is a caller-owned DEVICE pointer (for example the
 *    storage of a torch tensor) in row-major layout with the shape stated. The
 *    library allocates nothing, keeps nothing between calls and never writes
 *    an input.
 *  - Scratch memory is a caller-owned device buffer of at least the size the
 *    matching *_workspace_size call reports; distinct concurrent calls need
 *    distinct workspaces. The workspace's first 256 bytes hold a device status
 *    word.
 *  - Calls are asynchronous on the caller's cudaStream_t (passed as void*,
 *    NULL = legacy default stream). Argument errors found on the host are
 *    returned before any launch. Errors found on the device (an out-of-range
 *    token id or length, a bounded wait that ran out) are recorded in the
 *    workspace status word, the kernels keep every access in bounds, and
 *    dspark_check() reports the word after synchronising the stream.
 *  - Argument structs start with struct_size = sizeof(struct); a mismatch
 *    returns DSPARK_ERR_INVALID_ARGUMENT.
 *  - Random numbers: Philox4x32-10 (Salmon et al., SC'11) with key
 *    (seed low word, seed high word) and counter (e>>2, position, request,
 *    (round<<3)|purpose); output word e&3; uniform u = (2*(x>>9)+1)*2^-24;
 *    Gumbel noise -log(-log u). round must be below 2^29.
 *  - Draws are two-level Gumbel-max samples from the normalised weights: a
 *    Gumbel-max over the log-masses of vocabulary blocks of DSPARK_NOISE_BLOCK
 *    ids picks a block, then a Gumbel-max over the log-weights inside it picks
 *    the token (exact sampling; for V <= DSPARK_NOISE_BLOCK the flat Gumbel-max).
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSPARK_ABI_VERSION 1
#define DSPARK_NOISE_BLOCK 128   /* vocabulary block width of the two-level Gumbel-max */
#define DSPARK_MAX_GAMMA 32      /* largest draft block length gamma_max */
#define DSPARK_MAX_SLOTS 8192    /* largest R * gamma_max the scheduler accepts */
#define DSPARK_STATIC_WORKSPACE_BYTES (8u << 20)  /* scratch of dspark_sample_block_static */

typedef int32_t dspark_status;
enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARGUMENT = 1,  /* null pointer, bad size, bad enum, struct_size mismatch */
    DSPARK_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside what the kernels handle (stated per call) */
    DSPARK_ERR_WORKSPACE = 3,         /* workspace missing or smaller than *_workspace_size */
    DSPARK_ERR_CUDA = 4,              /* a CUDA runtime / driver call failed */
    DSPARK_ERR_TIMEOUT = 5,           /* a bounded device-side wait ran out (device status word) */
    DSPARK_ERR_DEVICE_INPUT = 6,      /* an out-of-range device value was clamped (device status word) */
    DSPARK_ERR_NONFINITE_INPUT = 7    /* a NaN or +inf logit (U, target) or a non-finite confidence logit
                                         (h or a weight) was read (device status word); -inf logits are
                                         zero-probability entries, not errors */
};

enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 };

enum {
    DSPARK_HEAD_MARKOV = 0,          /* eq. 5: B_k = W_1[x_{k-1}] W_2 */
    DSPARK_HEAD_RNN = 1              /* eq. 6: gated recurrent state, B_k = W_2^T tanh(W_o z_k) */
};

enum {
    DSPARK_SCHED_SYNC = 0,           /* Algorithm 1: stop at the first Theta <= Theta_best */
    DSPARK_SCHED_ASYNC_CAPACITY = 1, /* section 5.2: capacity K from old survivals, current ranking */
    DSPARK_SCHED_FULL_SCAN = 2,      /* arg-max of Theta over every prefix of the sorted pool */
    DSPARK_SCHED_THRESHOLD = 3       /* static confidence threshold: admit every a_{r,j} >= threshold */
};

enum {
    DSPARK_PATH_AUTO = 0,            /* tensor cores per step when the shape allows, else CUDA cores */
    DSPARK_PATH_CUDA_CORE = 1,       /* fp32 FMA bias contraction */
    DSPARK_PATH_TENSOR_CORE = 2,     /* tcgen05 bias contraction, one launch per step (bf16, r % 64 == 0,
                                        V % 8 == 0) */
    DSPARK_PATH_RESIDENT = 3         /* sampler only, on request: every step in one persistent launch, one
                                        CTA per SM, each keeping its slice of W in tensor and shared memory
                                        between steps (bf16, Markov head, R <= 128, r = 256, V % 8 == 0,
                                        V >= 1024); with step_ready events it waits for all of them first.
                                        Same results as the other paths; slower than the per-step tensor-core
                                        kernels at the measured shapes */
};

/*
 * dspark_sample_block -- Markov-head serial sampling, confidence head and
 * survival products (eq. 4, 5, 7; "dspark_cycle" step 3).
 *
 * For each request r and draft position k = 0 .. gamma_r-1, with x_0 = anchor[r]:
 *   B_k  = W_1[x_{k-1}] W_2        (E row times W; zero for k = 0 when bias_first = 0)
 *   l_k  = (U[r][k] + B_k) / temperature[r]
 *   x_k  ~ softmax(l_k)            (two-level Gumbel-max, purposes 0 and 3)
 *   c_k  = sigmoid((w_h . h[r][k] + w_e . W_1[x] + b) / t_k), x = x_{k-1} (conf_token 0,
 *          eq. 7) or x_k (conf_token 1); t_k = sts_temp[k] (sequential temperature scaling of
 *          the confidences, zhongzhuzhou.org notes "STS": the temperatures are fitted
 *          elsewhere and only applied here) or 1 when sts_temp is NULL
 *   a_k  = a_{k-1} c_k             (a_0 = 1)
 * Outputs for k >= gamma_r are token -1 and zeros.
 * head = DSPARK_HEAD_RNN replaces the bias operand W_1[x_{k-1}] by the RNN head's output
 * (zhongzhuzhou.org notes, eq. 6):
 *   z_k = [s_{k-1}; W_1[x_{k-1}]; h[r][k]],  [y_g; y_c; y_o] = W_rnn z_k,  s_0 = 0,
 *   s_k = sigmoid(y_g) * s_{k-1} + (1 - sigmoid(y_g)) * tanh(y_c),  B_k = tanh(y_o) W_2.
 *   The h part of W_rnn z_k is one GEMM over all positions (this library's tcgen05 GEMM for bf16
 *   shapes the copy engine takes, else a CUDA-core GEMM; fp32 accumulation), the
 *   rest a per-step kernel. On the tensor-core path (bf16, r a multiple of 64 up to 256,
 *   (2r + d) a multiple of 8, 16-byte aligned W_rnn and a_rows) that kernel is a tcgen05 GEMM
 *   whose fp32 state enters as two bf16 operands (its rounding and the rounding of the
 *   remainder); elsewhere it runs on CUDA cores in fp32. On the tensor-core path tanh(y_o)
 *   likewise enters the bias contraction as two bf16 operands, so the bias keeps about 16
 *   significant bits.
 * a_rows (optional output) receives each step's bias operand in fp32 (W_1[x_{k-1}] or
 * tanh(y_o)); dspark_verify needs them for an RNN-head draft.
 * temperature[r] = 0 is greedy decoding (zhongzhuzhou.org notes, FAQ on temperature 0):
 *   x_k = arg-max of U[r][k] + B_k (lowest index on ties), draft_lse = draft_logit = its value
 *   (the draft is a point mass).
 */
typedef struct {
    uint32_t struct_size;
    int32_t R;            /* requests, >= 1 */
    int32_t gamma_max;    /* 1 .. DSPARK_MAX_GAMMA */
    int32_t V;            /* vocabulary, 1 .. 2^24 */
    int32_t r;            /* Markov rank, 1 .. 1024 */
    int32_t d;            /* hidden width, >= 1 */
    int32_t dtype;        /* element type of U, E, W, h: DSPARK_F32 or DSPARK_BF16 */
    int32_t conf_token;   /* 0 or 1, see above */
    int32_t bias_first;   /* 1: B_1 = W_1[x_0] W_2 (eq. 4-5); 0: B_1 = 0 */
    int32_t path;         /* DSPARK_PATH_* for the bias contraction */
    const int32_t* gamma; /* [R] per-request gamma_r in 0..gamma_max, or NULL = gamma_max */
    const void* U;        /* [R][gamma_max][V] parallel-backbone logits */
    const void* E;        /* [V][r] W_1 */
    const void* W;        /* [r][V] W_2 */
    const void* h;        /* [R][gamma_max][d] backbone hidden states */
    const float* w_h;     /* [d] */
    const float* w_e;     /* [r] */
    float b;
    const float* temperature; /* [R], > 0, or 0 for greedy decoding */
    const int32_t* anchor;    /* [R] x_0 in 0..V-1 */
    uint64_t seed;
    uint64_t round;
    int32_t* tokens;          /* out [R][gamma_max] */
    float* conf;              /* out [R][gamma_max] c_k */
    float* surv;              /* out [R][gamma_max] a_k */
    float* draft_lse;         /* out [R][gamma_max] log sum_v exp(l_k(v)) */
    float* draft_logit;       /* out [R][gamma_max] l_k(x_k) */
    const float* sts_temp;    /* [gamma_max] per-position confidence temperatures (> 0), or NULL */
    int32_t head;             /* DSPARK_HEAD_MARKOV or DSPARK_HEAD_RNN */
    const void* W_rnn;        /* [3r][2r+d] (dtype of E): rows W_g, W_c, W_o (RNN head only) */
    float* a_rows;            /* out [R][gamma_max][r] bias operand of each step, or NULL */
    const void* const* step_ready; /* [gamma_max] cudaEvent_t (host array), or NULL: step k's kernels
                                      wait for step_ready[k] (NULL entries: no wait), so that U[:, k, :]
                                      may still be arriving when the call is made */
} dspark_sample_args;

dspark_status dspark_sample_workspace_size(const dspark_sample_args* args, size_t* bytes);
/* The bias-contraction path these arguments select (DSPARK_PATH_CUDA_CORE,
 * DSPARK_PATH_TENSOR_CORE or DSPARK_PATH_RESIDENT), or -status for invalid arguments. */
int32_t dspark_sample_path(const dspark_sample_args* args);
dspark_status dspark_sample_block(const dspark_sample_args* args, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * dspark_sample_block_static -- dspark_sample_block for callers that cannot allocate device
 * memory (no counterpart in the paper: it is a deployment convenience). Some callers cannot
 * call cudaMalloc where they run a round -- code living inside another framework's memory pool
 * without access to its allocator, code that must not grow the device footprint after start-up,
 * or runtimes that only hand the library its input and output buffers. This entry point takes
 * no workspace: its scratch lives in one file-scope device array of
 * DSPARK_STATIC_WORKSPACE_BYTES (8 MiB) that every GPU loading the library holds until the
 * process exits. It calls no cudaMalloc, cudaFree or allocating library routine.
 *  - Arguments and results are those of dspark_sample_block.
 *  - Shapes whose dspark_sample_workspace_size exceeds DSPARK_STATIC_WORKSPACE_BYTES return
 *    DSPARK_ERR_UNSUPPORTED_SHAPE before any launch (the RNN head's scratch grows with
 *    R * gamma_max * 3r, so it fits only for small shapes).
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 *    that device current; make that first call before any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous call's contents (the
 *    call clears what must start at zero). Calls whose work overlaps on the GPU (other streams,
 *    other host threads) race on it: serialise them.
 *  - The status word at the start of the array collects what the kernels record on the device
 *    (a clamped out-of-range device input, a bounded wait that ran out, a non-finite input).
 *    The call clears it first; read it with dspark_check_static after the call and before the
 *    next one.
 */
dspark_status dspark_sample_block_static(const dspark_sample_args* args, void* stream);

/* Synchronise `stream`, then return the device status word of the static array of
 * dspark_sample_block_static on the current device (DSPARK_OK or the code a kernel of the last
 * call recorded) and clear it. Like the array itself, it has no counterpart in the paper. */
dspark_status dspark_check_static(void* stream);

/*
 * dspark_schedule -- hardware-aware prefix scheduler (Algorithm 1; "admit").
 *
 * Pool = {(r, j) : j <= gamma_r, a_{r,j} = surv[r][j-1] > 0}, sorted by a
 * descending, then r ascending, then j ascending. With tau_m = R + sum of the
 * first m a's and Theta_m = tau_m * SPS(R + m):
 *   SYNC:  m* = (first m >= 1 with Theta_m <= Theta_{m-1}) - 1, else |pool|
 *   FULL_SCAN: m* = smallest arg-max of Theta_m over m = 0..|pool|
 *   ASYNC_CAPACITY: K = FULL_SCAN count over the pool of surv_capacity
 *          (survivals two rounds old); m* = min(K, |pool|)
 * keep[r] = l_r, the largest admitted position j of request r (Algorithm 1 sets
 * l_r = j on each admission); with survivals non-increasing in j (true for
 * products of confidences in (0,1)) it is the number of admitted slots.
 * The prefix sums are exact fixed-point sums of the fp32 a's (2^-48 units) and
 * Theta is formed in double from them.
 *   threshold  (the static confidence-threshold admission the paper compares against,
 *          zhongzhuzhou.org notes figure 5): admit every candidate (r, j) of the pool
 *          with a_{r,j} >= threshold; no throughput model is consulted. keep and the
 *          stats follow the same definitions (Theta of the admitted set, capacity -1).
 * Unsupported: R * gamma_max > DSPARK_MAX_SLOTS.
 */
typedef struct {
    double theta_best;    /* Theta_{m*} with the current survivals */
    int32_t admitted;     /* m* */
    int32_t capacity;     /* K (async) or -1 */
    int32_t batch;        /* B = R + m* */
    int32_t pool;         /* |pool| */
} dspark_schedule_stats;

typedef struct {
    uint32_t struct_size;
    int32_t R;
    int32_t gamma_max;
    int32_t mode;                 /* DSPARK_SCHED_* */
    int32_t n_sps;                /* >= R * (1 + gamma_max) */
    const int32_t* gamma;         /* [R] or NULL */
    const float* surv;            /* [R][gamma_max] current survivals */
    const float* surv_capacity;   /* [R][gamma_max] survivals two rounds old (ASYNC_CAPACITY only) */
    const float* sps;             /* [n_sps] SPS(B) at index B-1 */
    int32_t* keep;                /* out [R] */
    dspark_schedule_stats* stats; /* out, one device struct */
    float threshold;              /* DSPARK_SCHED_THRESHOLD only */
} dspark_schedule_args;

dspark_status dspark_schedule_workspace_size(const dspark_schedule_args* args, size_t* bytes);
dspark_status dspark_schedule(const dspark_schedule_args* args, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * dspark_verify -- lossless rejection-sampling verification of the admitted
 * prefixes ("dspark_cycle" steps 5-6; accept rule min(1, p_t/p_d) and the
 * residual norm(max(0, p_t - p_d)) of Leviathan et al.).
 *
 * Target row i of request r (target[r][i]) is the target's distribution for
 * draft position i; row keep[r] supplies the bonus token. With
 * p_t = softmax(target[r][i] / T_r) and p_d(x) = exp(draft_logit - draft_lse):
 *   for j = 0 .. keep[r]-1: accept tokens[r][j] iff log u_j < log p_t(x) - log p_d(x)
 *     (u_j: purpose 1, position j); stop at the first rejection.
 *   accepted[r] = n, the accepted prefix length.
 *   n < keep[r]: next_token ~ norm(max(0, p_t - p_d)) at position n, with p_d
 *     recomputed from U, E, W (purposes 2 and 4); resampled[r] = 1.
 *     If that residual is zero everywhere (possible only through rounding)
 *     next_token ~ p_t of row n.
 *   n = keep[r]: next_token ~ p_t of row keep[r]; resampled[r] = 0.
 * The residual's p_d is rebuilt with the bias operand W_1[x_{n-1}] (Markov head) or, when
 *   a_rows is given, with a_rows[r][n] (the RNN head's operand reported by the sampler).
 * Committed tokens: tokens[r][0:n] followed by next_token[r] (the next anchor).
 * temperature[r] = 0 (greedy decoding): tokens[r][j] is accepted iff it equals the arg-max of
 *   target row j (lowest index on ties); the first mismatch is replaced by that arg-max
 *   (resampled 1), and when every admitted token matches, the arg-max of row keep[r] is the
 *   bonus token (resampled 0). No random numbers are drawn.
 */
typedef struct {
    uint32_t struct_size;
    int32_t R;
    int32_t gamma_max;
    int32_t V;
    int32_t r;
    int32_t dtype;               /* element type of target, U, E, W */
    int32_t bias_first;          /* as passed to dspark_sample_block */
    int32_t path;                /* DSPARK_PATH_* for the residual's bias recompute */
    const int32_t* gamma;        /* [R] or NULL */
    const void* target;          /* [R][gamma_max+1][V] */
    const void* U;               /* [R][gamma_max][V] */
    const void* E;               /* [V][r] */
    const void* W;               /* [r][V] */
    const int32_t* anchor;       /* [R] */
    const int32_t* tokens;       /* [R][gamma_max] */
    const float* draft_lse;      /* [R][gamma_max] */
    const float* draft_logit;    /* [R][gamma_max] */
    const int32_t* keep;         /* [R] */
    const float* temperature;    /* [R] */
    uint64_t seed;
    uint64_t round;
    int32_t* accepted;           /* out [R] */
    int32_t* next_token;         /* out [R] */
    uint8_t* resampled;          /* out [R] */
    const float* a_rows;         /* [R][gamma_max][r] bias operands from dspark_sample_block, or NULL */
} dspark_verify_args;

dspark_status dspark_verify_workspace_size(const dspark_verify_args* args, size_t* bytes);
dspark_status dspark_verify(const dspark_verify_args* args, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * dspark_assemble -- the verify batch as one flat token stream (zhongzhuzhou.org notes,
 * physical execution of variable-length batches without padding): every request contributes
 * its anchor followed by its keep[r] admitted draft tokens, the runs laid end to end in request
 * order. Alongside each flat token: its request id and its causal position inside the request's
 * run (0 for the anchor, j for draft token j) -- the marker tensor a target forward consumes.
 *   offsets[r] = sum_{q < r} (keep[q] + 1),  offsets[R] = total
 *   flat_*[offsets[r] + j] for j = 0 .. keep[r];  entries from total to R*(gamma_max+1) are -1.
 * keep[r] outside [0, gamma_max] is clamped and DSPARK_ERR_DEVICE_INPUT recorded in the
 * workspace status word. Unsupported: R > DSPARK_MAX_SLOTS.
 */
typedef struct {
    uint32_t struct_size;
    int32_t R;
    int32_t gamma_max;
    const int32_t* keep;         /* [R] admitted lengths (dspark_schedule) */
    const int32_t* anchor;       /* [R] the token each request's block follows */
    const int32_t* tokens;       /* [R][gamma_max] draft tokens */
    int32_t* flat_tokens;        /* out [R*(gamma_max+1)] */
    int32_t* flat_request;       /* out [R*(gamma_max+1)] */
    int32_t* flat_position;      /* out [R*(gamma_max+1)] */
    int32_t* offsets;            /* out [R+1] */
} dspark_assemble_args;

dspark_status dspark_assemble_workspace_size(const dspark_assemble_args* args, size_t* bytes);
dspark_status dspark_assemble(const dspark_assemble_args* args, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Launch accounting and timing (measurement support, not part of the method).
 *
 * dspark_launch_count: number of kernels this library has launched in this
 * process (all calls, all streams).
 *
 * dspark_time_kernel: while enabled, every launch of kernel family `kernel`
 * (DSPARK_KERNEL_*) records events[i].start on the call's stream just before
 * the launch and events[i].stop just after it, for i = *count, *count+1, ...
 * up to `capacity`; *count (a host int) is incremented per recorded pair. The
 * events are cudaEvent_t handles created by the caller and passed as void*.
 * kernel = -1 disables timing. The setting is process-wide and not
 * thread-safe; it adds one event record before and after each timed launch.
 */
enum {
    DSPARK_KERNEL_DRAFT_SETUP = 0,    /* sampler set-up: clears the block-draw slots, writes step 0's conditioning rows */
    DSPARK_KERNEL_DRAFT_STATS = 1,    /* bias contraction + block softmax statistics, one per draft step */
    DSPARK_KERNEL_DRAFT_COMMIT = 2,   /* two-level draw, confidence, survival, one per draft step */
    DSPARK_KERNEL_SCHEDULE = 3,
    DSPARK_KERNEL_VERIFY_ROWS = 4,
    DSPARK_KERNEL_VERIFY_DECIDE = 5,
    DSPARK_KERNEL_RESIDUAL_STATS = 6,
    DSPARK_KERNEL_RESIDUAL_PICK = 7,
    DSPARK_KERNEL_ASSEMBLE = 8,
    DSPARK_KERNEL_RNN_STEP = 9,      /* RNN head: the per-step state update */
    DSPARK_KERNEL_RNN_HIDDEN = 10,   /* RNN head: the h part of the projection, every position, once per call */
    DSPARK_KERNEL_DRAFT_LOOP = 11    /* the resident path's one launch: every draft step and its commit */
};

typedef struct {
    void* start;   /* cudaEvent_t */
    void* stop;    /* cudaEvent_t */
} dspark_event_pair;

uint64_t dspark_launch_count(void);
dspark_status dspark_time_kernel(int32_t kernel, dspark_event_pair* events, int32_t capacity, int32_t* count);

/* Synchronise `stream`, then return the device status word of `workspace`
 * (DSPARK_OK, DSPARK_ERR_TIMEOUT, DSPARK_ERR_DEVICE_INPUT or DSPARK_ERR_NONFINITE_INPUT: the
 * first code a kernel recorded since the last check) and clear it. */
dspark_status dspark_check(void* workspace, void* stream);

/* Bound, in nanoseconds of the device's global timer, of every device-side wait on another
 * agent (a copy, an MMA, another CTA) in the calls made after this one, process-wide; 0
 * restores the default of 4 s. Returns the previous bound. A wait that runs out records
 * DSPARK_ERR_TIMEOUT in the status word; its kernel stops issuing work, lets its own copies and
 * MMAs in flight complete, frees its tensor memory and returns, so the context stays usable.
 * Meant for tests and debugging: results of a call whose wait ran out are not defined. */
uint64_t dspark_set_wait_limit(uint64_t ns);

/* Description of the last CUDA failure seen by a call on this thread (the kernel
 * family and the CUDA error name and string), or "no error". */
const char* dspark_last_error(void);

/* Static description of a status code. */
const char* dspark_status_string(dspark_status status);

/* DSPARK_ABI_VERSION of the loaded library. */
int32_t dspark_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif
