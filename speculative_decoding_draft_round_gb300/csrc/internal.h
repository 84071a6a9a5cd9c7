// internal.h -- parameter blocks and launchers shared between the libdspark
// translation units (host side). Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// Copies of the next step's A rows the tensor-core draft path keeps, so that the 152 CTAs reading
// the same 64 KB tile spread over 8 copies instead of one.
constexpr int kAReplicas = 8;

// One serial step of the draft sampler (dspark_sample_block).
struct DraftStep {
    int R, G, V, r, d, k, nblk;
    int dtype, conf_token, bias_first;
    const int32_t* gamma;
    const void* U;
    const void* E;
    const void* W;
    const void* h;
    const float* w_h;
    const float* w_e;
    float b;
    const float* temperature;
    const int32_t* anchor;
    uint64_t seed, round;
    int32_t* tokens;
    float* conf;
    float* surv;
    float* draft_lse;
    float* draft_logit;
    const float* sts_temp;   // [G] confidence temperatures or NULL
    // workspace
    int* status;
    int32_t* x_cur;      // [R] token committed at the previous step
    float2* stats;       // [R][n_stats] (max, sum) of exp2, log2 units: per vocabulary block (CUDA-core
                         // path) or per CTA of the tensor-core kernel (its blocks merged), row-major
    int n_stats;         // entries per row of stats: nblk, or the tensor-core grid
    unsigned long long* pick;   // [G][R] packed block-level arg-max of each step (cleared per call)
    void* a_next;        // [a_replicas][R][r] (element type of E): W_1 row of the token each request
                         // conditions on next, in a_replicas identical copies (RNN head on the tensor-core
                         // path: the bf16 rounding of the step's bias operand)
    int a_replicas;      // 1 (CUDA-core path) or kAReplicas (tensor-core path: each CTA reads one copy)
    // RNN head (eq. 6)
    int head;            // DSPARK_HEAD_*
    const void* W_rnn;   // [3r][2r+d]
    float* a_rows;       // [R][G][r] fp32 bias operand of each step (RNN head: tanh(W_o z_k))
    float* yh;           // [R*G][3r] W_rnn[:, 2r:] h_k for every position
    float* state;        // [2][R][r] s_{k-1} / s_k by step parity
    void* a_lo;          // [R][r] bf16: operand minus its bf16 rounding (tensor-core path)
    void* zbuf;          // [2][R][3r] bf16 by step parity: [hi(s_{k-1}); lo(s_{k-1}); W_1[x_{k-1}]], the
                         // tensor-core RNN step's operand rows (NULL: the CUDA-core step)
    unsigned long long wait_ns;   // bound of each device-side wait (dspark_set_wait_limit)
};

// Verification (dspark_verify).
struct VerifyParams {
    int R, G, V, r, nblk;
    int dtype, bias_first;
    const int32_t* gamma;
    const void* target;
    const void* U;
    const void* E;
    const void* W;
    const int32_t* anchor;
    const int32_t* tokens;
    const float* draft_lse;
    const float* draft_logit;
    const int32_t* keep;
    const float* temperature;
    uint64_t seed, round;
    int32_t* accepted;
    int32_t* next_token;
    uint8_t* resampled;
    // workspace
    int* status;
    float2* row_stats;   // [R][G+1][nblk] block (max, sum) of the target rows, log2 units
    float2* row_part;    // [R][G+1][npart] per-warp merges of 8 blocks of row_stats
    int npart;           // ceil(nblk / 8)
    float* lse_t;        // [R][G+1]
    int32_t* rej;        // [R] rejected position, -1 if every admitted token was accepted
    int* n_rej;          // number of rejected requests (zeroed by verify_rows, counted by verify_decide)
    int32_t* rej_list;   // [R] the rejected requests, in the order verify_decide found them
    float* res_stats;    // [R_pad][nblk] block sums of max(0, p_t - p_d)
    const float* a_rows; // [R][G][r] bias operands reported by the sampler, or NULL (W_1[x_{n-1}])
    unsigned long long wait_ns;   // bound of each device-side wait (dspark_set_wait_limit)
};

struct ScheduleParams {
    int R, G, mode, n_sps;
    const int32_t* gamma;
    const float* surv;
    const float* surv_capacity;
    const float* sps;
    int32_t* keep;
    dspark_schedule_stats* stats;
    float threshold;
    int* status;
};

// The flattened verify batch (dspark_assemble).
struct AssembleParams {
    int R, G;
    const int32_t* keep;
    const int32_t* anchor;
    const int32_t* tokens;
    int32_t* flat_tokens;
    int32_t* flat_request;
    int32_t* flat_position;
    int32_t* offsets;
    int* status;
};

// sample.cu
cudaError_t launch_draft_setup(const DraftStep& p, cudaStream_t s);
cudaError_t launch_draft_stats_simt(const DraftStep& p, cudaStream_t s);
// wmap: the W block map of encode_w_block_map, or NULL (the commit then loads W with plain loads)
cudaError_t launch_draft_commit(const DraftStep& p, const CUtensorMap* wmap, cudaStream_t s);
// Tensor map of W [r][V] bf16 with one [r x 128] box per vocabulary block (r <= 256, V % 8 == 0,
// W 16-byte aligned): the commit's copy of the winning block.
cudaError_t encode_w_block_map(CUtensorMap* m, const void* W, int V, int r);

// sample_tc.cu
bool tc_supported(int dtype, int R, int V, int r, const void* U, const void* E, const void* W);
bool tc_residual_supported(int dtype, int R, int V, int r, const void* U, const void* E, const void* W);
size_t tc_stats_rows(int R);  // rows of the block-statistics workspace the tensor-core path writes
int tc_grid(int R, int nblk); // CTAs of the tensor-core statistics kernel
int num_sms();                 // streaming multiprocessors of the current device
// The scheduler's grid: one CTA that schedules and three that warm its code. Each holds every
// register of its SM (1024 threads x 64), so the verify row pass, launched while they run, leaves
// those SMs out of its persistent grid.
constexpr int kScheduleCtas = 4;
int verify_row_partials(int nblk);   // per-warp partials of one verified target row
cudaError_t launch_draft_stats_tc(const DraftStep& p, cudaStream_t s);
cudaError_t launch_residual_stats_tc(const VerifyParams& p, cudaStream_t s);

// draft_loop.cu (the persistent, W-resident draft loop: one launch for every step)
bool loop_supported(int dtype, int head, int R, int V, int r, const void* U, const void* E, const void* W,
                    const void* h, const void* w_h, const void* w_e);
int loop_ctas(int R, int V);                 // its grid, and the per-CTA partials of each row
size_t loop_slot_bytes(int R, int V);        // its leading-block logit slots
cudaError_t launch_draft_loop(const DraftStep& p, float* slots, float* hdot, unsigned int* gbar, int* gabort,
                              cudaStream_t s);

// verify.cu
cudaError_t launch_verify_rows(const VerifyParams& p, cudaStream_t s);
cudaError_t launch_verify_decide(const VerifyParams& p, cudaStream_t s);
cudaError_t launch_residual_stats_simt(const VerifyParams& p, cudaStream_t s);
cudaError_t launch_residual_pick(const VerifyParams& p, cudaStream_t s);

// schedule.cu
size_t schedule_smem_bytes();
cudaError_t launch_schedule(const ScheduleParams& p, cudaStream_t s);

// assemble.cu
cudaError_t launch_assemble(const AssembleParams& p, cudaStream_t s);

// rnn.cu (RNN head)
cudaError_t launch_rnn_hidden(const DraftStep& p, cudaStream_t s);   // rnn_hidden.cu: yh = W_rnn[:, 2r:] h, every position
cudaError_t launch_rnn_step(const DraftStep& p, cudaStream_t s);     // step k: state, bias operand
// rnn_tc.cu (RNN head on the tensor cores)
bool rnn_tc_supported(const DraftStep& p);
cudaError_t rnn_tc_maps(const DraftStep& p, CUtensorMap* zmap, CUtensorMap* wmap);
cudaError_t launch_rnn_z0(const DraftStep& p, cudaStream_t s);      // z[0]: zero state, W_1 of the anchor
cudaError_t launch_rnn_step_tc(const DraftStep& p, const CUtensorMap& zmap, const CUtensorMap& wmap, cudaStream_t s);

// Bound of the device-side waits on other agents (copies, MMAs, other CTAs) for the next
// launches; 4 s unless dspark_set_wait_limit changed it.
unsigned long long wait_limit_ns();

inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace dspark
