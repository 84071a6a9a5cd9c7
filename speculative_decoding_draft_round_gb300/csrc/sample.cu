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
//                    contraction, then (max, sum exp2) of l_k over the block.
//                    The V-wide bias never reaches global memory.
//   draft_commit  -- per request: block-level Gumbel-max over the block
//                    log-masses, element-level Gumbel-max inside the winning
//                    block (its 128 logits recomputed), log-normaliser,
//                    confidence and survival; x_k becomes the next step's
//                    previous token.
// w_h . h_k does not depend on the draws, so conf_hidden computes it for every
// (request, position) in one pass before the serial loop.
#include "common.cuh"
#include "internal.h"

namespace dspark {

// ----------------------------------------------------------------- w_h . h

template <typename T>
__global__ void __launch_bounds__(256) conf_hidden_kernel(DraftStep p)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= p.R * p.G) return;
    const int q = warp / p.G, k = warp % p.G;
    const int g = p.gamma ? p.gamma[q] : p.G;
    if (k >= g) return;
    const T* h = static_cast<const T*>(p.h) + (size_t)warp * p.d;
    float acc = 0.f;
    const bool vec = (p.d % 8 == 0) && ((reinterpret_cast<uintptr_t>(p.h) & 15u) == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.w_h) & 15u) == 0);
    if (vec) {
        // 8 elements (16 bytes of bf16, 32 of fp32) per lane per step, all loads independent
        for (int j = lane * 8; j < p.d; j += 256) {
            float w[8], x[8];
            load8<T>(h + j, x);
            load8<float>(p.w_h + j, w);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(w[e], x[e], acc);
        }
    } else {
        for (int j = lane; j < p.d; j += 32) acc += p.w_h[j] * ld(h, j);
    }
    acc = warp_sum(acc);
    if (lane == 0) p.hw[warp] = acc;
}

// ----------------------------------------------------------------- block statistics (CUDA cores)

constexpr int kSimtReq = 8;   // requests per block of the CUDA-core contraction

struct StepRequest {
    int active, prev, use_bias;
    float scale;              // log2(e) / T
};

__device__ __forceinline__ StepRequest draft_request(const DraftStep& p, int q)
{
    StepRequest s{0, 0, 0, 0.f};
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
    s.scale = kLog2e / p.temperature[q];
    return s;
}

template <typename T>
__global__ void __launch_bounds__(kNoiseBlock) draft_stats_simt_kernel(DraftStep p)
{
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
        es[i] = (req[j].active && req[j].use_bias) ? ld(E, (size_t)req[j].prev * p.r + c) : 0.f;
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
        if (t == 0) p.stats[(size_t)q * p.nblk + b] = make_float2(m, s);
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

template <typename T>
__global__ void __launch_bounds__(kCommitThreads) draft_commit_kernel(DraftStep p)
{
    extern __shared__ float sm_dyn[];   // [r] W_1[prev], then [16][128] K-slice partials
    float* erow = sm_dyn;
    float* part = sm_dyn + ((p.r + 3) & ~3);
    __shared__ float sv[kCommitThreads / 32];
    __shared__ int si[kCommitThreads / 32];
    __shared__ float lm_s[kCommitThreads / 32], ls_s[kCommitThreads / 32];
    __shared__ float red[kCommitThreads / 32];
    __shared__ int s_tok;
    __shared__ float s_logit;
    const int q = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const StepRequest rq = draft_request(p, q);
    const size_t o = (size_t)q * p.G + p.k;
    if (!rq.active) {
        if (t == 0) {
            p.tokens[o] = -1;
            p.conf[o] = p.surv[o] = p.draft_lse[o] = p.draft_logit[o] = 0.f;
        }
        return;
    }
    const T* E = static_cast<const T*>(p.E);
    const T* W = static_cast<const T*>(p.W);
    const PhiloxKey key = make_key(p.seed);
    const float2* st = p.stats + (size_t)q * p.nblk;

    // W_1[prev] for the element-level recompute (independent of the block draw)
    for (int i = t; i < p.r; i += kCommitThreads) erow[i] = rq.use_bias ? ld(E, (size_t)rq.prev * p.r + i) : 0.f;

    // block level: Gumbel-max over ln(block mass), one Philox call per 4 consecutive blocks,
    // and the log-normaliser accumulated in the same pass
    ArgMax best{-INFINITY, -1};
    LseAcc acc{-INFINITY, 0.f};
    for (int g4 = t; g4 * 4 < p.nblk; g4 += kCommitThreads) {
        const uint4 w = philox4x32_10(
            make_uint4((uint32_t)g4, (uint32_t)p.k, (uint32_t)q, counter_word3(p.round, kDraftBlock)), key);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = g4 * 4 + j;
            if (b < p.nblk) {
                const float2 ms = st[b];
                const float L2 = ms.x + log2f(ms.y);
                acc = lse_add(acc, L2);
                const float z = L2 * kLn2 - logf(-logf(bits_to_uniform(words[j])));
                best = argmax_better(best, ArgMax{z, b});
            }
        }
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
    best = block_argmax<kCommitThreads>(best, sv, si);   // contains __syncthreads
    LseAcc tot{-INFINITY, 0.f};
#pragma unroll
    for (int w = 0; w < kCommitThreads / 32; ++w) tot = lse_merge(tot, LseAcc{lm_s[w], ls_s[w]});
    int bstar = best.i;
    if (bstar < 0) {
        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
        bstar = 0;
    }

    // element level inside the chosen block: recompute its 128 logits
    float bias = 0.f;
    if (rq.use_bias) bias = block_bias<T>(erow, W, p.V, p.r, bstar * kNoiseBlock, part);
    const int v = bstar * kNoiseBlock + t;
    ArgMax cand{-INFINITY, -1};
    float lv = 0.f;
    if (t < kNoiseBlock && v < p.V) {
        const T* U = static_cast<const T*>(p.U);
        lv = (ld(U, o * p.V + v) + bias) / p.temperature[q];
        cand = ArgMax{lv + gumbel_at(key, p.round, kDraftElem, (uint32_t)q, (uint32_t)p.k, (uint32_t)v), v};
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

    // confidence head (eq. 7) on W_1[x_{k-1}] or W_1[x_k]
    const int xc = p.conf_token ? tok : rq.prev;
    float dot = 0.f;
    for (int i = t; i < p.r; i += kCommitThreads) dot = fmaf(p.w_e[i], ld(E, (size_t)xc * p.r + i), dot);
    dot = block_sum<kCommitThreads>(dot, red);
    if (t == 0) {
        const float logit = p.hw[o] + dot + p.b;
        const float c = 1.f / (1.f + expf(-logit));
        const float prev_s = p.k == 0 ? 1.f : p.surv[o - 1];
        p.tokens[o] = s_tok;
        p.conf[o] = c;
        p.surv[o] = prev_s * c;
        p.draft_lse[o] = (tot.m + log2f(tot.s)) * kLn2;
        p.draft_logit[o] = s_logit;
        p.x_cur[q] = s_tok;
    }
}

// ----------------------------------------------------------------- launchers

cudaError_t launch_conf_hidden(const DraftStep& p, cudaStream_t s)
{
    const int rows = p.R * p.G;
    const int blocks = cdiv(rows, 8);
    if (p.dtype == DSPARK_BF16)
        conf_hidden_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(p);
    else
        conf_hidden_kernel<float><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_draft_stats_simt(const DraftStep& p, cudaStream_t s)
{
    const dim3 grid(p.nblk, cdiv(p.R, kSimtReq));
    const size_t smem = (size_t)kSimtReq * p.r * sizeof(float);
    if (p.dtype == DSPARK_BF16) {
        cudaFuncSetAttribute(draft_stats_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        draft_stats_simt_kernel<__nv_bfloat16><<<grid, kNoiseBlock, smem, s>>>(p);
    } else {
        cudaFuncSetAttribute(draft_stats_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        draft_stats_simt_kernel<float><<<grid, kNoiseBlock, smem, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_draft_commit(const DraftStep& p, cudaStream_t s)
{
    const size_t smem = (size_t)(((p.r + 3) & ~3) + 16 * kNoiseBlock) * sizeof(float);
    if (p.dtype == DSPARK_BF16)
        draft_commit_kernel<__nv_bfloat16><<<p.R, kCommitThreads, smem, s>>>(p);
    else
        draft_commit_kernel<float><<<p.R, kCommitThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace dspark
