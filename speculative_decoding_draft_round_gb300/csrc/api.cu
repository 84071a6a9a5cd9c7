// api.cu -- the C ABI of libdspark (include/dspark.h): argument validation,
// workspace layout and the launch sequence of each call. Every step of the
// round runs in this library's kernels; nothing here computes on the host.
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

using namespace dspark;

namespace {

// ------------------------------------------------------------ launch accounting

std::atomic<unsigned long long> g_launches{0};

constexpr unsigned long long kDefaultWaitNs = 4000000000ull;   // 4 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

struct KernelTimer {
    int kernel = -1;
    dspark_event_pair* events = nullptr;
    int capacity = 0;
    int32_t* count = nullptr;
} g_timer;

bool timing(int kernel) { return g_timer.kernel == kernel && g_timer.count && *g_timer.count < g_timer.capacity; }

const char* kernel_name(int kernel)
{
    static const char* names[] = {"draft_setup", "draft_stats", "draft_commit", "schedule",
                                  "verify_rows", "verify_decide", "residual_stats", "residual_pick",
                                  "assemble", "rnn_step", "rnn_hidden", "draft_loop"};
    return kernel >= 0 && kernel <= DSPARK_KERNEL_DRAFT_LOOP ? names[kernel] : "?";
}

thread_local char g_last_error[256] = "no error";

// Launch one kernel family through `fn`, counting it and recording the timing events if enabled.
template <typename F>
cudaError_t launch(int kernel, cudaStream_t s, F&& fn)
{
    const bool t = timing(kernel);
    cudaError_t e = cudaSuccess;
    if (t) e = cudaEventRecord(static_cast<cudaEvent_t>(g_timer.events[*g_timer.count].start), s);
    if (e == cudaSuccess) e = fn();
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (t && e == cudaSuccess) {
        e = cudaEventRecord(static_cast<cudaEvent_t>(g_timer.events[*g_timer.count].stop), s);
        ++*g_timer.count;
    }
    if (e != cudaSuccess)
        snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", kernel_name(kernel), cudaGetErrorName(e),
                 cudaGetErrorString(e));
    return e;
}

// Clear a non-sticky error another library left in this thread's runtime state, so that
// the checks after our own launches report only our launches.
void clear_stale_error() { (void)cudaGetLastError(); }

constexpr size_t kAlign = 256;
constexpr size_t kStatusBytes = 256;


dspark_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

// ------------------------------------------------------------ sample_block

struct SampleLayout {
    size_t x_cur, stats, pick, a_next, yh, state, a_rows, a_lo, zbuf, slots, hdot, total;
};

// the status word sits at offset 0 of every workspace; the resident loop's grid barrier counter
// and abort flag share its 256-byte region
constexpr size_t kGridBarOffset = 64;
constexpr size_t kGridAbortOffset = 128;

dspark_status check_sample(const dspark_sample_args* a)
{
    if (!a || a->struct_size != sizeof(dspark_sample_args)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->R < 1 || a->gamma_max < 1 || a->gamma_max > DSPARK_MAX_GAMMA) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->V < 1 || a->V > (1 << 24) || a->r < 1 || a->r > 1024 || a->d < 1) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->dtype != DSPARK_F32 && a->dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARGUMENT;
    if ((a->conf_token | 1) != 1 || (a->bias_first | 1) != 1) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->head != DSPARK_HEAD_MARKOV && a->head != DSPARK_HEAD_RNN) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->head == DSPARK_HEAD_RNN && !a->W_rnn) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->path < DSPARK_PATH_AUTO || a->path > DSPARK_PATH_RESIDENT) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->round >= (1ull << 29)) return DSPARK_ERR_INVALID_ARGUMENT;
    if ((long long)a->R * a->gamma_max * a->V >= (1ll << 40)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (!a->U || !a->E || !a->W || !a->h || !a->w_h || !a->w_e || !a->temperature || !a->anchor)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (!a->tokens || !a->conf || !a->surv || !a->draft_lse || !a->draft_logit) return DSPARK_ERR_INVALID_ARGUMENT;
    return DSPARK_OK;
}

bool sample_uses_tc(const dspark_sample_args* a)
{
    if (a->path == DSPARK_PATH_CUDA_CORE) return false;
    return tc_supported(a->dtype, a->R, a->V, a->r, a->U, a->E, a->W);
}

// the persistent resident loop, when asked for. AUTO does not take it: measured at R = 128,
// V = 151936 it runs the draft in 1.18 ms against 0.48 ms for the per-step kernels (its transposed
// epilogue and the serial tail between steps cost more than the W traffic it saves)
bool sample_uses_loop(const dspark_sample_args* a)
{
    if (a->path != DSPARK_PATH_RESIDENT) return false;
    return sample_uses_tc(a) && loop_supported(a->dtype, a->head, a->R, a->V, a->r, a->U, a->E, a->W, a->h, a->w_h,
                                               a->w_e);
}

SampleLayout sample_layout(const dspark_sample_args* a)
{
    const int nblk = cdiv(a->V, kNoiseBlock);
    const size_t rows = sample_uses_tc(a) ? tc_stats_rows(a->R) : (size_t)a->R;
    const bool loop = sample_uses_loop(a);
    SampleLayout L;
    size_t o = kStatusBytes;
    L.x_cur = o;
    o = align_up(o + sizeof(int32_t) * a->R, kAlign);
    L.stats = o;   // per block (CUDA-core path), per CTA of the tensor-core kernel, or per CTA of the
                   // loop for two steps (its outputs of step k are written while step k + 1 runs)
    o = align_up(o + sizeof(float2) * rows *
                         (loop ? 2 * loop_ctas(a->R, a->V) : sample_uses_tc(a) ? tc_grid(a->R, nblk) : nblk),
                 kAlign);
    L.pick = o;
    o = align_up(o + sizeof(unsigned long long) * (size_t)a->R * a->gamma_max, kAlign);
    L.a_next = o;   // the tensor-core path keeps kAReplicas copies of the next step's A rows
    o = align_up(o + (sample_uses_tc(a) ? kAReplicas : 1) * (a->dtype == DSPARK_BF16 ? 2 : 4) * (size_t)a->R * a->r,
                 kAlign);
    const bool rnn = a->head == DSPARK_HEAD_RNN;
    L.yh = o;   // RNN head: the h part of the projection, every position
    o = align_up(o + (rnn ? sizeof(float) * (size_t)a->R * a->gamma_max * 3 * a->r : 0), kAlign);
    L.state = o;
    o = align_up(o + (rnn ? sizeof(float) * 2 * (size_t)a->R * a->r : 0), kAlign);
    L.a_rows = o;   // used when the caller does not take the bias operands
    o = align_up(o + (rnn && !a->a_rows ? sizeof(float) * (size_t)a->R * a->gamma_max * a->r : 0), kAlign);
    L.a_lo = o;
    o = align_up(o + (rnn ? 2 * (size_t)a->R * a->r : 0), kAlign);
    L.zbuf = o;   // RNN head on the tensor cores: the step's operand rows, two parities of [R][3r] bf16
    o = align_up(o + (rnn && sample_uses_tc(a) ? 2 * 2 * (size_t)a->R * 3 * a->r : 0), kAlign);
    L.slots = o;   // the loop: per CTA and request, the leading block's logits
    o = align_up(o + (loop ? loop_slot_bytes(a->R, a->V) : 0), kAlign);
    L.hdot = o;    // the loop: w_h . h_k of every position
    o = align_up(o + (loop ? sizeof(float) * (size_t)a->R * a->gamma_max : 0), kAlign);
    L.total = o;
    return L;
}

// ------------------------------------------------------------ verify

struct VerifyLayout {
    size_t row_stats, row_part, lse_t, rej, n_rej, rej_list, res_stats, total;
};

dspark_status check_verify(const dspark_verify_args* a)
{
    if (!a || a->struct_size != sizeof(dspark_verify_args)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->R < 1 || a->gamma_max < 1 || a->gamma_max > DSPARK_MAX_GAMMA) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->V < 1 || a->V > (1 << 24) || a->r < 1 || a->r > 1024) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->dtype != DSPARK_F32 && a->dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARGUMENT;
    if ((a->bias_first | 1) != 1) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->path < DSPARK_PATH_AUTO || a->path > DSPARK_PATH_TENSOR_CORE) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->round >= (1ull << 29)) return DSPARK_ERR_INVALID_ARGUMENT;
    if ((long long)a->R * (a->gamma_max + 1) * a->V >= (1ll << 40)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (!a->target || !a->U || !a->E || !a->W || !a->anchor || !a->tokens || !a->draft_lse || !a->draft_logit ||
        !a->keep || !a->temperature)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (!a->accepted || !a->next_token || !a->resampled) return DSPARK_ERR_INVALID_ARGUMENT;
    return DSPARK_OK;
}

bool verify_uses_tc(const dspark_verify_args* a)
{
    if (a->path == DSPARK_PATH_CUDA_CORE) return false;
    if (a->a_rows) return false;   // fp32 bias operands (RNN head): the CUDA-core residual keeps them exact
    return tc_residual_supported(a->dtype, a->R, a->V, a->r, a->U, a->E, a->W);
}

VerifyLayout verify_layout(const dspark_verify_args* a)
{
    const int nblk = cdiv(a->V, kNoiseBlock);
    const size_t rows = verify_uses_tc(a) ? tc_stats_rows(a->R) : (size_t)a->R;
    VerifyLayout L;
    size_t o = kStatusBytes;
    L.row_stats = o;
    o = align_up(o + sizeof(float2) * (size_t)a->R * (a->gamma_max + 1) * nblk, kAlign);
    L.row_part = o;
    o = align_up(o + sizeof(float2) * (size_t)a->R * (a->gamma_max + 1) * verify_row_partials(nblk), kAlign);
    L.lse_t = o;
    o = align_up(o + sizeof(float) * (size_t)a->R * (a->gamma_max + 1), kAlign);
    L.rej = o;
    o = align_up(o + sizeof(int32_t) * a->R, kAlign);
    L.n_rej = o;
    o = align_up(o + sizeof(int), kAlign);
    L.rej_list = o;
    o = align_up(o + sizeof(int32_t) * a->R, kAlign);
    L.res_stats = o;
    o = align_up(o + sizeof(float) * rows * nblk, kAlign);
    L.total = o;
    return L;
}

// ------------------------------------------------------------ schedule

dspark_status check_schedule(const dspark_schedule_args* a)
{
    if (!a || a->struct_size != sizeof(dspark_schedule_args)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->R < 1 || a->gamma_max < 1 || a->gamma_max > DSPARK_MAX_GAMMA) return DSPARK_ERR_INVALID_ARGUMENT;
    if ((long long)a->R * a->gamma_max > DSPARK_MAX_SLOTS) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (a->mode < DSPARK_SCHED_SYNC || a->mode > DSPARK_SCHED_THRESHOLD) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->mode == DSPARK_SCHED_THRESHOLD && !(a->threshold == a->threshold)) return DSPARK_ERR_INVALID_ARGUMENT;
    if ((long long)a->n_sps < (long long)a->R * (1 + a->gamma_max)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!a->surv || !a->sps || !a->keep || !a->stats) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->mode == DSPARK_SCHED_ASYNC_CAPACITY && !a->surv_capacity) return DSPARK_ERR_INVALID_ARGUMENT;
    return DSPARK_OK;
}

template <typename T>
T* at(void* ws, size_t off)
{
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

unsigned long long dspark::wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

extern "C" {

int32_t dspark_abi_version(void) { return DSPARK_ABI_VERSION; }

const char* dspark_status_string(dspark_status s)
{
    switch (s) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_INVALID_ARGUMENT: return "invalid argument";
    case DSPARK_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case DSPARK_ERR_WORKSPACE: return "workspace missing or too small";
    case DSPARK_ERR_CUDA: return "CUDA error";
    case DSPARK_ERR_TIMEOUT: return "bounded device wait ran out";
    case DSPARK_ERR_DEVICE_INPUT: return "out-of-range device input (clamped)";
    case DSPARK_ERR_NONFINITE_INPUT: return "NaN or +inf in a logit or hidden-state input";
    default: return "unknown status";
    }
}

dspark_status dspark_sample_workspace_size(const dspark_sample_args* a, size_t* bytes)
{
    const dspark_status st = check_sample(a);
    if (st != DSPARK_OK) return st;
    if (!bytes) return DSPARK_ERR_INVALID_ARGUMENT;
    *bytes = sample_layout(a).total;
    return DSPARK_OK;
}

int32_t dspark_sample_path(const dspark_sample_args* a)
{
    const dspark_status st = check_sample(a);
    if (st != DSPARK_OK) return -st;
    if (a->path == DSPARK_PATH_TENSOR_CORE && !sample_uses_tc(a)) return -DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (a->path == DSPARK_PATH_RESIDENT && !sample_uses_loop(a)) return -DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (sample_uses_loop(a)) return DSPARK_PATH_RESIDENT;
    return sample_uses_tc(a) ? DSPARK_PATH_TENSOR_CORE : DSPARK_PATH_CUDA_CORE;
}

dspark_status dspark_sample_block(const dspark_sample_args* a, void* ws, size_t ws_bytes, void* stream)
{
    clear_stale_error();
    dspark_status st = check_sample(a);
    if (st != DSPARK_OK) return st;
    if (a->path == DSPARK_PATH_TENSOR_CORE && !sample_uses_tc(a)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (a->path == DSPARK_PATH_RESIDENT && !sample_uses_loop(a)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    const SampleLayout L = sample_layout(a);
    if (!ws || ws_bytes < L.total) return DSPARK_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DraftStep p;
    memset(&p, 0, sizeof p);
    p.R = a->R;
    p.G = a->gamma_max;
    p.V = a->V;
    p.r = a->r;
    p.d = a->d;
    p.nblk = cdiv(a->V, kNoiseBlock);
    p.dtype = a->dtype;
    p.conf_token = a->conf_token;
    p.bias_first = a->bias_first;
    p.gamma = a->gamma;
    p.U = a->U;
    p.E = a->E;
    p.W = a->W;
    p.h = a->h;
    p.w_h = a->w_h;
    p.w_e = a->w_e;
    p.b = a->b;
    p.temperature = a->temperature;
    p.anchor = a->anchor;
    p.seed = a->seed;
    p.round = a->round;
    p.tokens = a->tokens;
    p.conf = a->conf;
    p.surv = a->surv;
    p.draft_lse = a->draft_lse;
    p.draft_logit = a->draft_logit;
    p.sts_temp = a->sts_temp;
    p.wait_ns = wait_limit_ns();
    p.status = at<int>(ws, 0);
    p.x_cur = at<int32_t>(ws, L.x_cur);
    p.stats = at<float2>(ws, L.stats);
    p.n_stats = sample_uses_tc(a) ? tc_grid(a->R, p.nblk) : p.nblk;
    p.pick = at<unsigned long long>(ws, L.pick);
    p.a_next = at<unsigned char>(ws, L.a_next);
    const bool tc = sample_uses_tc(a);
    p.a_replicas = tc && a->head != DSPARK_HEAD_RNN ? kAReplicas : 1;
    p.head = a->head;
    p.W_rnn = a->W_rnn;
    const bool rnn = a->head == DSPARK_HEAD_RNN;
    p.a_rows = rnn ? (a->a_rows ? a->a_rows : at<float>(ws, L.a_rows)) : a->a_rows;
    p.yh = rnn ? at<float>(ws, L.yh) : nullptr;
    p.state = rnn ? at<float>(ws, L.state) : nullptr;
    p.a_lo = rnn && tc ? at<unsigned char>(ws, L.a_lo) : nullptr;
    p.zbuf = rnn && tc ? at<unsigned char>(ws, L.zbuf) : nullptr;
    if (sample_uses_loop(a)) {
        // every step in one persistent launch (after every per-step input event, if any)
        p.n_stats = loop_ctas(a->R, a->V);
        cudaError_t e = cudaSuccess;
        for (int k = 0; a->step_ready && k < a->gamma_max && e == cudaSuccess; ++k)
            if (a->step_ready[k])
                e = cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(const_cast<void*>(a->step_ready[k])), 0);
        if (e == cudaSuccess)
            e = launch(DSPARK_KERNEL_DRAFT_LOOP, s, [&] {
                return launch_draft_loop(p, at<float>(ws, L.slots), at<float>(ws, L.hdot),
                                         at<unsigned int>(ws, kGridBarOffset), at<int>(ws, kGridAbortOffset), s);
            });
        return cuda_status(e);
    }
    cudaError_t e = launch(DSPARK_KERNEL_DRAFT_SETUP, s, [&] { return launch_draft_setup(p, s); });
    if (rnn && e == cudaSuccess) {
        // the h part of the RNN projection, every position: one GEMM before the serial loop
        e = launch(DSPARK_KERNEL_RNN_HIDDEN, s, [&] { return launch_rnn_hidden(p, s); });
        if (e != cudaSuccess)
            snprintf(g_last_error, sizeof g_last_error, "rnn hidden GEMM: %s (%s)", cudaGetErrorName(e),
                     cudaGetErrorString(e));
    }
    // RNN head on the tensor cores: operand-row and W_rnn tensor maps, and the step-0 operand rows
    CUtensorMap zmap, rmap;
    memset(&zmap, 0, sizeof zmap);
    memset(&rmap, 0, sizeof rmap);
    const bool rnn_tc = rnn && e == cudaSuccess && rnn_tc_supported(p) && rnn_tc_maps(p, &zmap, &rmap) == cudaSuccess;
    if (rnn && !rnn_tc) p.zbuf = nullptr;   // the CUDA-core step: the commit writes no operand rows
    if (rnn_tc) e = launch(DSPARK_KERNEL_RNN_STEP, s, [&] { return launch_rnn_z0(p, s); });
    // the commit copies the winning W block with one bulk copy when W admits the block map
    CUtensorMap wmap;
    memset(&wmap, 0, sizeof wmap);
    const bool use_wmap = a->dtype == DSPARK_BF16 && a->r % 16 == 0 && a->r <= 256 &&
                          encode_w_block_map(&wmap, a->W, a->V, a->r) == cudaSuccess;
    for (int k = 0; k < a->gamma_max && e == cudaSuccess; ++k) {
        p.k = k;
        // the caller may still be delivering this step's inputs (U[:, k, :]): wait for its event
        if (a->step_ready && a->step_ready[k]) {
            e = cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(const_cast<void*>(a->step_ready[k])), 0);
            if (e != cudaSuccess) {
                snprintf(g_last_error, sizeof g_last_error, "step_ready[%d]: %s", k, cudaGetErrorName(e));
                break;
            }
        }
        if (rnn)
            e = launch(DSPARK_KERNEL_RNN_STEP, s,
                       [&] { return rnn_tc ? launch_rnn_step_tc(p, zmap, rmap, s) : launch_rnn_step(p, s); });
        if (e == cudaSuccess)
            e = launch(DSPARK_KERNEL_DRAFT_STATS, s,
                       [&] { return tc ? launch_draft_stats_tc(p, s) : launch_draft_stats_simt(p, s); });
        if (e == cudaSuccess)
            e = launch(DSPARK_KERNEL_DRAFT_COMMIT, s, [&] { return launch_draft_commit(p, use_wmap ? &wmap : nullptr, s); });
    }
    return cuda_status(e);
}

dspark_status dspark_schedule_workspace_size(const dspark_schedule_args* a, size_t* bytes)
{
    const dspark_status st = check_schedule(a);
    if (st != DSPARK_OK) return st;
    if (!bytes) return DSPARK_ERR_INVALID_ARGUMENT;
    *bytes = kStatusBytes;
    return DSPARK_OK;
}

dspark_status dspark_schedule(const dspark_schedule_args* a, void* ws, size_t ws_bytes, void* stream)
{
    clear_stale_error();
    const dspark_status st = check_schedule(a);
    if (st != DSPARK_OK) return st;
    if (!ws || ws_bytes < kStatusBytes) return DSPARK_ERR_WORKSPACE;
    ScheduleParams p;
    p.R = a->R;
    p.G = a->gamma_max;
    p.mode = a->mode;
    p.n_sps = a->n_sps;
    p.gamma = a->gamma;
    p.surv = a->surv;
    p.surv_capacity = a->surv_capacity;
    p.sps = a->sps;
    p.keep = a->keep;
    p.stats = a->stats;
    p.threshold = a->threshold;
    p.status = at<int>(ws, 0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(launch(DSPARK_KERNEL_SCHEDULE, s, [&] { return launch_schedule(p, s); }));
}

dspark_status dspark_assemble_workspace_size(const dspark_assemble_args* a, size_t* bytes)
{
    if (!a || a->struct_size != sizeof(dspark_assemble_args) || !bytes) return DSPARK_ERR_INVALID_ARGUMENT;
    *bytes = kStatusBytes;
    return DSPARK_OK;
}

dspark_status dspark_assemble(const dspark_assemble_args* a, void* ws, size_t ws_bytes, void* stream)
{
    clear_stale_error();
    if (!a || a->struct_size != sizeof(dspark_assemble_args)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->R < 1 || a->gamma_max < 1 || a->gamma_max > DSPARK_MAX_GAMMA) return DSPARK_ERR_INVALID_ARGUMENT;
    if (a->R > DSPARK_MAX_SLOTS) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (!a->keep || !a->anchor || !a->tokens || !a->flat_tokens || !a->flat_request || !a->flat_position ||
        !a->offsets)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (!ws || ws_bytes < kStatusBytes) return DSPARK_ERR_WORKSPACE;
    AssembleParams p;
    p.R = a->R;
    p.G = a->gamma_max;
    p.keep = a->keep;
    p.anchor = a->anchor;
    p.tokens = a->tokens;
    p.flat_tokens = a->flat_tokens;
    p.flat_request = a->flat_request;
    p.flat_position = a->flat_position;
    p.offsets = a->offsets;
    p.status = at<int>(ws, 0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(launch(DSPARK_KERNEL_ASSEMBLE, s, [&] { return launch_assemble(p, s); }));
}

dspark_status dspark_verify_workspace_size(const dspark_verify_args* a, size_t* bytes)
{
    const dspark_status st = check_verify(a);
    if (st != DSPARK_OK) return st;
    if (!bytes) return DSPARK_ERR_INVALID_ARGUMENT;
    *bytes = verify_layout(a).total;
    return DSPARK_OK;
}

dspark_status dspark_verify(const dspark_verify_args* a, void* ws, size_t ws_bytes, void* stream)
{
    clear_stale_error();
    const dspark_status st = check_verify(a);
    if (st != DSPARK_OK) return st;
    if (a->path == DSPARK_PATH_TENSOR_CORE && !tc_supported(a->dtype, a->R, a->V, a->r, a->U, a->E, a->W))
        return DSPARK_ERR_UNSUPPORTED_SHAPE;
    const VerifyLayout L = verify_layout(a);
    if (!ws || ws_bytes < L.total) return DSPARK_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    VerifyParams p;
    memset(&p, 0, sizeof p);
    p.R = a->R;
    p.G = a->gamma_max;
    p.V = a->V;
    p.r = a->r;
    p.nblk = cdiv(a->V, kNoiseBlock);
    p.dtype = a->dtype;
    p.bias_first = a->bias_first;
    p.gamma = a->gamma;
    p.target = a->target;
    p.U = a->U;
    p.E = a->E;
    p.W = a->W;
    p.anchor = a->anchor;
    p.tokens = a->tokens;
    p.draft_lse = a->draft_lse;
    p.a_rows = a->a_rows;
    p.draft_logit = a->draft_logit;
    p.keep = a->keep;
    p.temperature = a->temperature;
    p.seed = a->seed;
    p.round = a->round;
    p.accepted = a->accepted;
    p.next_token = a->next_token;
    p.resampled = a->resampled;
    p.wait_ns = wait_limit_ns();
    p.status = at<int>(ws, 0);
    p.row_stats = at<float2>(ws, L.row_stats);
    p.row_part = at<float2>(ws, L.row_part);
    p.npart = verify_row_partials(p.nblk);
    p.lse_t = at<float>(ws, L.lse_t);
    p.rej = at<int32_t>(ws, L.rej);
    p.n_rej = at<int>(ws, L.n_rej);
    p.rej_list = at<int32_t>(ws, L.rej_list);
    p.res_stats = at<float>(ws, L.res_stats);
    const bool tc = verify_uses_tc(a);
    cudaError_t e = launch(DSPARK_KERNEL_VERIFY_ROWS, s, [&] { return launch_verify_rows(p, s); });
    if (e == cudaSuccess) e = launch(DSPARK_KERNEL_VERIFY_DECIDE, s, [&] { return launch_verify_decide(p, s); });
    if (e == cudaSuccess)
        e = launch(DSPARK_KERNEL_RESIDUAL_STATS, s,
                   [&] { return tc ? launch_residual_stats_tc(p, s) : launch_residual_stats_simt(p, s); });
    if (e == cudaSuccess) e = launch(DSPARK_KERNEL_RESIDUAL_PICK, s, [&] { return launch_residual_pick(p, s); });
    return cuda_status(e);
}

const char* dspark_last_error(void) { return g_last_error; }

uint64_t dspark_set_wait_limit(uint64_t ns)
{
    return g_wait_ns.exchange(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

uint64_t dspark_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

dspark_status dspark_time_kernel(int32_t kernel, dspark_event_pair* events, int32_t capacity, int32_t* count)
{
    if (kernel < 0) {
        g_timer = KernelTimer();
        return DSPARK_OK;
    }
    if (kernel > DSPARK_KERNEL_DRAFT_LOOP || !events || capacity < 0 || !count) return DSPARK_ERR_INVALID_ARGUMENT;
    g_timer.kernel = kernel;
    g_timer.events = events;
    g_timer.capacity = capacity;
    g_timer.count = count;
    return DSPARK_OK;
}

dspark_status dspark_check(void* ws, void* stream)
{
    if (!ws) return DSPARK_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, ws, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    return h;
}

}  // extern "C"
