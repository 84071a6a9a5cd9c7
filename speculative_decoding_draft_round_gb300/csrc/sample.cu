// sample.cu -- Markov-head serial sampling (CUDA-core contraction), confidence
// head and survival products.
//
// One draft step k of "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation" (caijizhuo.github.io, section 4 dspark_cycle
// step 3; zhongzhuzhou.org notes eq. 4, 5, 7):
//   B_k = W_1[x_{k-1}] W_2, l_k = (U_k + B_k) / T, x_k ~ softmax(l_k),
//   c_k = sigmoid(w_h . h_k + w_e . W_1[x] + b), a_k = a_{k-1} c_k.
// The step runs as two launches:
//   draft_stats   -- per (request, 128-wide vocabulary block): the bias
//                    contraction, then (max, sum exp2) of l_k over the block and
//                    the block's key of the two-level Gumbel-max, folded into one
//                    packed atomicMax per request. The V-wide bias never reaches
//                    global memory. (CUDA-core version here; tensor-core version in
//                    sample_tc.cu.)
//   draft_commit  -- per request: the winning block, the element-level Gumbel-max
//                    inside it (its 128 logits recomputed from W's block columns),
//                    the log-normaliser from the statistics, confidence and
//                    survival; x_k becomes the next step's previous token.
// w_h . h_k does not depend on the draws: each commit forms it from the inputs while the
// previous kernel finishes, and reduces it with the w_e part of eq. (7).
//   draft_setup   -- once per call: clears the block-draw slots and writes the first
//                    step's conditioning rows W_1[x_0].
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace dspark {

// ----------------------------------------------------------------- set-up of a call

template <typename T>
__global__ void __launch_bounds__(256) draft_setup_kernel(DraftStep p)
{
    pdl_enter();   // the previous call's kernels read the slots and rows written here
    // clear the per-step block-draw slots of this call, and set the first step's conditioning rows
    // (W_1[x_0], x_0 = anchor) for the tensor-core statistics kernel
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.R * p.G; i += gridDim.x * blockDim.x) p.pick[i] = 0ull;
    {
        const T* E = static_cast<const T*>(p.E);
        T* an = static_cast<T*>(p.a_next);
        const size_t n = (size_t)p.R * p.r;
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)n;
             i += (long long)gridDim.x * blockDim.x) {
            const int q = (int)(i / p.r), c = (int)(i % p.r);
            const int x0 = checked_index(p.anchor[q], p.V, p.status);
            const T v = E[(size_t)x0 * p.r + c];
            for (int rp = 0; rp < p.a_replicas; ++rp) an[rp * n + i] = v;
        }
    }
}

// ----------------------------------------------------------------- block statistics (CUDA cores)

constexpr int kSimtReq = 8;   // requests per block of the CUDA-core contraction

struct StepRequest {
    int active, prev, use_bias;
    float scale;              // log2(e) / T (log2(e) for greedy requests)
    int greedy;               // temperature 0: the draw is the arg-max (no noise)
};

__device__ __forceinline__ StepRequest draft_request(const DraftStep& p, int q)
{
    StepRequest s{0, 0, 0, 0.f, 0};
    if (q >= p.R) return s;
    int g = p.gamma ? p.gamma[q] : p.G;
    if (g < 0 || g > p.G) {
        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
        g = g < 0 ? 0 : p.G;
    }
    if (p.k >= g) return s;
    s.active = 1;
    s.prev = checked_index(p.k == 0 ? p.anchor[q] : p.x_cur[q], p.V, p.status);
    s.use_bias = (p.k > 0) || p.bias_first;
    s.greedy = p.temperature[q] == 0.f;
    s.scale = s.greedy ? kLog2e : kLog2e / p.temperature[q];
    return s;
}

// the part of draft_request that reads only inputs (no earlier kernel's output)
__device__ __forceinline__ StepRequest draft_request_inputs(const DraftStep& p, int q)
{
    StepRequest s{0, 0, 0, 0.f, 0};
    if (q >= p.R) return s;
    int g = p.gamma ? p.gamma[q] : p.G;
    if (g < 0 || g > p.G) {
        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
        g = g < 0 ? 0 : p.G;
    }
    if (p.k >= g) return s;
    s.active = 1;
    s.use_bias = (p.k > 0) || p.bias_first;
    s.greedy = p.temperature[q] == 0.f;
    s.scale = s.greedy ? kLog2e : kLog2e / p.temperature[q];
    return s;
}

template <typename T>
__global__ void __launch_bounds__(kNoiseBlock) draft_stats_simt_kernel(DraftStep p)
{
    pdl_enter();   // x_cur, the operand rows and the pick slots come from the previous kernels
    extern __shared__ float es[];   // [kSimtReq][r]
    __shared__ StepRequest req[kSimtReq];
    __shared__ float red[8];
    const int b = blockIdx.x;
    const int q0 = blockIdx.y * kSimtReq;
    const int t = threadIdx.x;
    if (t < kSimtReq) req[t] = draft_request(p, q0 + t);
    __syncthreads();
    const T* E = static_cast<const T*>(p.E);
    const T* W = static_cast<const T*>(p.W);
    for (int i = t; i < kSimtReq * p.r; i += blockDim.x) {
        const int j = i / p.r, c = i % p.r;
        // the bias operand: W_1[x_{k-1}] (Markov head) or the RNN head's tanh(W_o z_k) row
        const size_t ar = ((size_t)(q0 + j) * p.G + p.k) * p.r + c;
        es[i] = (req[j].active && req[j].use_bias)
                    ? (p.head == DSPARK_HEAD_RNN ? p.a_rows[ar] : ld(E, (size_t)req[j].prev * p.r + c))
                    : 0.f;
    }
    __syncthreads();
    const int v = b * kNoiseBlock + t;
    float acc[kSimtReq];
#pragma unroll
    for (int j = 0; j < kSimtReq; ++j) acc[j] = 0.f;
    if (v < p.V) {
        for (int i = 0; i < p.r; ++i) {
            const float w = ld(W, (size_t)i * p.V + v);
#pragma unroll
            for (int j = 0; j < kSimtReq; ++j) acc[j] = fmaf(es[j * p.r + i], w, acc[j]);
        }
    }
    const T* U = static_cast<const T*>(p.U);
#pragma unroll 1
    for (int j = 0; j < kSimtReq; ++j) {
        if (!req[j].active) continue;   // uniform across the block
        const int q = q0 + j;
        float x = -INFINITY;
        if (v < p.V) x = (ld(U, ((size_t)q * p.G + p.k) * p.V + v) + acc[j]) * req[j].scale;
        const float m = block_max<kNoiseBlock>(x, red);
        const float e = v < p.V ? exp2f(x - m) : 0.f;
        const float s = block_sum<kNoiseBlock>(e, red);
        if (t == 0) {
            // a NaN or +inf logit leaves a NaN sum or an infinite maximum (-inf is a zero weight)
            if (!(s >= 0.f) || m == INFINITY || m != m) raise_status(p.status, DSPARK_ERR_NONFINITE_INPUT);
            p.stats[(size_t)q * p.n_stats + b] = make_float2(m, s);
            // block key of the two-level draw; greedy requests take the block holding the maximum
            const float z = req[j].greedy ? m
                                          : (m + log2f(s)) * kLn2 -
                                                logf(-logf(uniform_at(make_key(p.seed), p.round, kDraftBlock,
                                                                      (uint32_t)q, (uint32_t)p.k, (uint32_t)b)));
            atomicMax(p.pick + (size_t)p.k * p.R + q, pack_pick(z, b));
        }
    }
}

// ----------------------------------------------------------------- commit

constexpr int kCommitThreads = kBlockGemvThreads;

// Online (max, sum) pair in log2 units: represents sum_i 2^{x_i} as s * 2^m.
struct LseAcc {
    float m, s;
};

__device__ __forceinline__ LseAcc lse_add(LseAcc a, float L2)
{
    if (L2 <= a.m) return LseAcc{a.m, a.s + exp2f(L2 - a.m)};
    return LseAcc{L2, a.s * exp2f(a.m - L2) + 1.f};
}

__device__ __forceinline__ LseAcc lse_merge(LseAcc a, LseAcc b)
{
    if (b.m == -INFINITY) return a;
    if (a.m == -INFINITY) return b;
    return a.m >= b.m ? LseAcc{a.m, a.s + b.s * exp2f(b.m - a.m)} : LseAcc{b.m, b.s + a.s * exp2f(a.m - b.m)};
}

// Phase structure (each phase issues all of its global reads before using any):
//   A  pick slot of this step, every block statistic, W_1[prev], per-request scalars
//   B  (needs b*) the block's W columns (one 16-byte vector per K-slice row) and U values,
//      while the log-normaliser of phase A is reduced
//   C  (needs x_k) W_1[x_k]: the next step's conditioning row and, for conf_token = 1, eq. (7)
constexpr int kStatsPerThread = 8;       // block statistics held in registers per thread (nblk <= 2048)
constexpr int kBiasRows = 16;            // W rows per thread in the fast path (r <= 256)

constexpr unsigned long long kCommitDrainNs = 4000000000ull;   // 4 s: a copy in flight lands long before

// Bounded wait for phase `parity` of a shared-memory barrier; false (and DSPARK_ERR_TIMEOUT
// recorded) when it runs out.
__device__ __forceinline__ bool commit_wait(uint32_t bar, uint32_t parity, int* status, unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > limit_ns) {
            raise_status(status, DSPARK_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Shared memory of the commit: [r] W_1[prev] (padded to 4), [16][128] K-slice partials, and with
// the W block map the block's W columns [r][128] bf16 (128-byte aligned for the copy) and the
// copy's barrier.
__host__ __device__ inline size_t commit_smem_wtile(int r) { return (size_t)(((r + 3) & ~3) + 16 * kNoiseBlock) * 4; }
constexpr size_t kCommitTmaSlack = 128 + 16;   // alignment of the tile, then the barrier

template <typename T, bool RNN>
__global__ void __launch_bounds__(kCommitThreads)
    draft_commit_kernel(DraftStep p, const __grid_constant__ CUtensorMap wmap, int use_wmap)
{
    extern __shared__ __align__(16) float sm_dyn[];
    float* erow = sm_dyn;
    float* part = sm_dyn + ((p.r + 3) & ~3);
    unsigned char* wtile = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(sm_dyn) + commit_smem_wtile(p.r) + 127) & ~uintptr_t(127));
    const uint32_t wbar = smem_addr(wtile + (size_t)p.r * kNoiseBlock * 2);
    if (use_wmap && threadIdx.x == 0) {
        mbar_init(wbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __shared__ float sv[kCommitThreads / 32];
    __shared__ int si[kCommitThreads / 32];
    __shared__ float lm_s[kCommitThreads / 32], ls_s[kCommitThreads / 32];
    __shared__ float red[kCommitThreads / 32];
    __shared__ int s_tok;
    __shared__ float s_logit;
    const int q = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    // inputs that no earlier kernel writes can be read before the dependency wait
    const StepRequest rq = draft_request_inputs(p, q);
    const size_t o = (size_t)q * p.G + p.k;
    const bool greedy = p.temperature[q] == 0.f;   // temperature 0: arg-max draft
    const float invT = greedy ? 1.f : 1.f / p.temperature[q];
    // w_h . h[q][k], the confidence head's hidden part (eq. 7): h and w_h are inputs, so this
    // thread's share of the dot product is formed while the previous kernel finishes, and is
    // reduced with the w_e part after the draw
    float hdot = 0.f;
    if (rq.active) {
        const T* h = static_cast<const T*>(p.h) + o * p.d;
        if (sizeof(T) == 2 && p.d % 8 == 0 && ((reinterpret_cast<uintptr_t>(p.h) & 15u) == 0) &&
            ((reinterpret_cast<uintptr_t>(p.w_h) & 15u) == 0)) {
            for (int c = t * 8; c < p.d; c += 8 * kCommitThreads) {
                float x[8], w[8];
                load8<T>(h + c, x);
                load8<float>(p.w_h + c, w);
#pragma unroll
                for (int e = 0; e < 8; ++e) hdot = fmaf(w[e], x[e], hdot);
            }
        } else {
            for (int c = t; c < p.d; c += kCommitThreads) hdot = fmaf(p.w_h[c], ld(h, c), hdot);
        }
    }
    pdl_wait();      // block statistics, pick slots and x_cur come from the kernels before this one
    pdl_trigger();   // the next step's statistics kernel may start its prefetch
    if (!rq.active) {
        if (p.a_rows && !RNN)
            for (int i = t; i < p.r; i += kCommitThreads) p.a_rows[o * p.r + i] = 0.f;
        if (t == 0) {
            p.tokens[o] = -1;
            p.conf[o] = p.surv[o] = p.draft_lse[o] = p.draft_logit[o] = 0.f;
        }
        return;
    }
    // W_1[x_{k-1}] is the conditioning row the previous commit (or draft_setup for k = 0) wrote
    const T* prev_row = static_cast<const T*>(p.a_next) + (size_t)q * p.r;
    const T* E = static_cast<const T*>(p.E);
    const T* W = static_cast<const T*>(p.W);
    const T* U = static_cast<const T*>(p.U);
    const PhiloxKey key = make_key(p.seed);
    const float2* st = p.stats + (size_t)q * p.n_stats;

    // ---- phase A
    const unsigned long long pk = p.pick[(size_t)p.k * p.R + q];
    const float surv_prev = p.k == 0 ? 1.f : p.surv[o - 1];
    const bool fast_stats = p.n_stats <= kStatsPerThread * kCommitThreads;
    float2 ms[kStatsPerThread];
    if (fast_stats) {
#pragma unroll
        for (int u = 0; u < kStatsPerThread; ++u) {
            const int b = t + u * kCommitThreads;
            ms[u] = b < p.n_stats ? st[b] : make_float2(-INFINITY, 0.f);
        }
    }
    const bool need_prev_row = rq.use_bias || !p.conf_token;
    constexpr bool rnn = RNN;
    // RNN head: the bias operand is the step's tanh(W_o z_k); W_1[x_{k-1}] feeds eq. (7) only
    const int prevtok = rnn ? checked_index(p.k == 0 ? p.anchor[q] : p.x_cur[q], p.V, p.status) : 0;
    // the conditioning row is loaded now and stored to shared memory after the phase-B loads are
    // issued, so that no use of a load holds up the next one (r <= 4 * kCommitThreads here)
    constexpr int kErowPer = 4;
    float ev[kErowPer];
#pragma unroll
    for (int j = 0; j < kErowPer; ++j) {
        const int i = t + j * kCommitThreads;
        ev[j] = 0.f;
        if (i < p.r) {
            if (rnn)
                ev[j] = rq.use_bias ? p.a_rows[o * p.r + i] : 0.f;
            else
                ev[j] = (need_prev_row || p.a_rows) ? ld(prev_row, i) : 0.f;
        }
    }
    int bstar = pk == 0ull ? -1 : unpack_pick_index(pk);
    if (bstar < 0 || bstar >= p.nblk) {
        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
        bstar = 0;
    }

    // ---- phase B: the chosen block's W columns and U values
    const int v = bstar * kNoiseBlock + t;
    const bool fast_bias = rq.use_bias && sizeof(T) == 2 && p.V % 8 == 0 && p.r % 16 == 0 &&
                           p.r <= 16 * kBiasRows && ((reinterpret_cast<uintptr_t>(W) & 15u) == 0);
    const int cg = t & 15, ks = t >> 4;
    const int c0 = bstar * kNoiseBlock + cg * 8;
    uint4 wv[kBiasRows];
    // With the W block map one bulk copy brings the block's [r x 128] columns into shared memory
    // (64 KB at r = 256: more than per-thread loads keep in flight); columns past V read as zero.
    const bool tma_w = fast_bias && use_wmap;
    if (tma_w && t == 0) {
        mbar_expect_tx(wbar, (uint32_t)p.r * kNoiseBlock * 2);
        tma_load_2d(smem_addr(wtile), &wmap, bstar * kNoiseBlock, 0, wbar, l2_policy_evict_normal());
    }
    if (fast_bias && !tma_w) {
#pragma unroll
        for (int j = 0; j < kBiasRows; ++j) {
            const int i = ks + 16 * j;
            wv[j] = (i < p.r && c0 < p.V) ? __ldg(reinterpret_cast<const uint4*>(W + (size_t)i * p.V + c0))
                                          : make_uint4(0, 0, 0, 0);
        }
    }
    // U at this thread's column of the block, kept in its own type until it is used
    T u_raw = T(0.f);
    if (t < kNoiseBlock && v < p.V) u_raw = U[o * p.V + v];
    // the element Gumbel of this column: it needs only the picked block, so it is formed under the W copy
    const float gum = (t < kNoiseBlock && v < p.V && !greedy)
                          ? gumbel_at(key, p.round, kDraftElem, (uint32_t)q, (uint32_t)p.k, (uint32_t)v) : 0.f;
#pragma unroll
    for (int j = 0; j < kErowPer; ++j) {
        const int i = t + j * kCommitThreads;
        if (i < p.r) {
            erow[i] = (rnn || need_prev_row) ? ev[j] : 0.f;
            if (!rnn && p.a_rows) p.a_rows[o * p.r + i] = ev[j];   // Markov operand W_1[x_{k-1}]
        }
    }
    // log-normaliser from phase A while the phase-B loads fly
    LseAcc acc{-INFINITY, 0.f};
    if (fast_stats) {
#pragma unroll
        for (int u = 0; u < kStatsPerThread; ++u)
            if (ms[u].y > 0.f) acc = lse_add(acc, ms[u].x + log2f(ms[u].y));   // empty entries hold zero mass
    } else {
        for (int b = t; b < p.n_stats; b += kCommitThreads)
            if (st[b].y > 0.f) acc = lse_add(acc, st[b].x + log2f(st[b].y));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const LseAcc other{__shfl_xor_sync(0xffffffffu, acc.m, off), __shfl_xor_sync(0xffffffffu, acc.s, off)};
        acc = lse_merge(acc, other);
    }
    if (lane == 0) {
        lm_s[warp] = acc.m;
        ls_s[warp] = acc.s;
    }
    __syncthreads();   // also publishes erow
    LseAcc tot{-INFINITY, 0.f};
#pragma unroll
    for (int w = 0; w < kCommitThreads / 32; ++w) tot = lse_merge(tot, LseAcc{lm_s[w], ls_s[w]});
    float bias = 0.f;
    bool w_ok = true;
    if (tma_w) {
        w_ok = commit_wait(wbar, 0u, p.status, p.wait_ns);
        const uint4* wt = reinterpret_cast<const uint4*>(wtile);
#pragma unroll
        for (int j = 0; j < kBiasRows; ++j) {
            const int i = ks + 16 * j;
            wv[j] = (w_ok && i < p.r) ? wt[i * (kNoiseBlock / 8) + cg] : make_uint4(0, 0, 0, 0);
        }
    }
    if (fast_bias) {
        float a8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kBiasRows; ++j) {
            const int i = ks + 16 * j;
            if (i < p.r) {
                const float ei = erow[i];
                const uint32_t u4[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    a8[2 * h] = fmaf(ei, __uint_as_float(u4[h] << 16), a8[2 * h]);
                    a8[2 * h + 1] = fmaf(ei, __uint_as_float(u4[h] & 0xFFFF0000u), a8[2 * h + 1]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) part[ks * kNoiseBlock + cg * 8 + j] = a8[j];
        __syncthreads();
        if (t < kNoiseBlock)
            for (int s2 = 0; s2 < 16; ++s2) bias += part[s2 * kNoiseBlock + t];
    } else if (rq.use_bias) {
        bias = block_bias<T>(erow, W, p.V, p.r, bstar * kNoiseBlock, part);
    }
    ArgMax cand{-INFINITY, -1};
    float lv = 0.f;
    if (t < kNoiseBlock && v < p.V) {
        lv = (to_f32<T>(u_raw) + bias) * invT;
        cand = ArgMax{greedy ? lv : lv + gum, v};
    }
    const ArgMax win = block_argmax<kCommitThreads>(cand, sv, si);
    int tok = win.i;
    if (tok < 0) {
        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
        tok = min(bstar * kNoiseBlock, p.V - 1);
    }
    if (t < kNoiseBlock && v == tok) {
        s_tok = tok;
        s_logit = lv;
    }

    // ---- phase C: W_1[x_k] for the next step's conditioning rows and the confidence head (eq. 7)
    float dot = 0.f;
    T* an = static_cast<T*>(p.a_next) + (size_t)q * p.r;
    const size_t rep_stride = (size_t)p.R * p.r;
    for (int i = t; i < p.r; i += kCommitThreads) {
        const T et = E[(size_t)tok * p.r + i];
        if (!rnn)   // the RNN head's next operand comes from its state update
            for (int rp = 0; rp < p.a_replicas; ++rp) an[rp * rep_stride + i] = et;
        else if (p.zbuf)   // the tensor-core RNN step's next operand rows: W_1[x_k]
            static_cast<T*>(p.zbuf)[(((size_t)((p.k + 1) & 1) * p.R + q) * 3 + 2) * p.r + i] = et;
        const float xprev = rnn ? (p.conf_token ? 0.f : ld(E, (size_t)prevtok * p.r + i)) : erow[i];
        dot = fmaf(p.w_e[i], p.conf_token ? to_f32<T>(et) : xprev, dot);   // eq. (7) reads W_1[x_{k-1}]
    }
    dot = block_sum<kCommitThreads>(dot + hdot, red);
    if (t == 0) {
        // sequential temperature scaling of the confidence: the head's logit over t_k
        const float logit = (dot + p.b) / (p.sts_temp ? p.sts_temp[p.k] : 1.f);
        if (!isfinite(logit)) raise_status(p.status, DSPARK_ERR_NONFINITE_INPUT);   // h, or a weight
        const float c = 1.f / (1.f + expf(-logit));
        p.tokens[o] = s_tok;
        p.conf[o] = c;
        p.surv[o] = surv_prev * c;
        // greedy: the draft is a point mass, reported as lse = logit (log p_d(x_k) = 0)
        p.draft_lse[o] = greedy ? s_logit : (tot.m + log2f(tot.s)) * kLn2;
        p.draft_logit[o] = s_logit;
        p.x_cur[q] = s_tok;
    }
    // a copy whose wait gave up may still be writing shared memory: let it land before exit
    if (tma_w && !w_ok && t == 0) (void)commit_wait(wbar, 0u, nullptr, kCommitDrainNs);
}

// ----------------------------------------------------------------- launchers

cudaError_t launch_draft_setup(const DraftStep& p, cudaStream_t s)
{
    const int blocks = cdiv(std::max(p.R * p.G, p.R * p.r), 256);
    const cudaError_t e = p.dtype == DSPARK_BF16 ? launch_pdl(draft_setup_kernel<__nv_bfloat16>, blocks, 256, 0, s, p)
                                                 : launch_pdl(draft_setup_kernel<float>, blocks, 256, 0, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_draft_stats_simt(const DraftStep& p, cudaStream_t s)
{
    const dim3 grid(p.nblk, cdiv(p.R, kSimtReq));
    const size_t smem = (size_t)kSimtReq * p.r * sizeof(float);
    if (p.dtype == DSPARK_BF16) {
        cudaFuncSetAttribute(draft_stats_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        const cudaError_t e = launch_pdl(draft_stats_simt_kernel<__nv_bfloat16>, grid, kNoiseBlock, smem, s, p);
        if (e != cudaSuccess) return e;
    } else {
        cudaFuncSetAttribute(draft_stats_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const cudaError_t e = launch_pdl(draft_stats_simt_kernel<float>, grid, kNoiseBlock, smem, s, p);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

template <typename T, bool RNN>
cudaError_t launch_commit_instance(const DraftStep& p, const CUtensorMap* wmap, cudaStream_t s)
{
    const bool use = wmap != nullptr;
    const size_t smem = commit_smem_wtile(p.r) + (use ? (size_t)p.r * kNoiseBlock * 2 + kCommitTmaSlack : 0);
    static size_t smem_set = 0;   // the largest dynamic shared memory this instance was opened to
    if (smem > 48 * 1024 && smem > smem_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(draft_commit_kernel<T, RNN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    CUtensorMap none;
    memset(&none, 0, sizeof none);
    return launch_pdl(draft_commit_kernel<T, RNN>, dim3(p.R), dim3(kCommitThreads), smem, s, p, use ? *wmap : none,
                      use ? 1 : 0);
}

cudaError_t launch_draft_commit(const DraftStep& p, const CUtensorMap* wmap, cudaStream_t s)
{
    // the RNN head takes its own instance: the Markov head's commit carries none of its branches
    const bool rnn = p.head == DSPARK_HEAD_RNN;
    if (p.dtype == DSPARK_BF16)
        return rnn ? launch_commit_instance<__nv_bfloat16, true>(p, wmap, s)
                   : launch_commit_instance<__nv_bfloat16, false>(p, wmap, s);
    return rnn ? launch_commit_instance<float, true>(p, nullptr, s) : launch_commit_instance<float, false>(p, nullptr, s);
}

}  // namespace dspark
