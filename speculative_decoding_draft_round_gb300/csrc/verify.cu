// verify.cu -- lossless rejection-sampling verification of the admitted prefixes.
//
// "DSpark" dspark_cycle steps 5-6 (caijizhuo.github.io, section 4) with the
// standard accept rule min(1, p_t/p_d) and residual norm(max(0, p_t - p_d))
// (Leviathan et al. 2023; zhongzhuzhou.org notes, eq. 8a). Target row i is the
// target's distribution for draft position i; row keep[r] supplies the bonus.
// Launches:
//   verify_rows      -- per (request, row i <= keep, vocabulary chunk): block
//                       (max, sum exp2) of target/T, one warp per 128-block.
//   verify_decide    -- per request: target log-normalisers, accept tests,
//                       first rejection; bonus draw when nothing was rejected.
//   residual_stats   -- per (rejecting request, vocabulary block): p_d
//                       recomputed with the Markov bias of the rejected
//                       position, block sums of max(0, p_t - p_d).
//   residual_pick    -- per rejecting request: two-level Gumbel-max over the
//                       residual (p_t of the same row if the residual is zero).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dspark {

__device__ __forceinline__ int request_gamma(const VerifyParams& p, int q)
{
    int g = p.gamma ? p.gamma[q] : p.G;
    if (g < 0 || g > p.G) {
        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
        g = g < 0 ? 0 : p.G;
    }
    return g;
}

__device__ __forceinline__ int request_keep(const VerifyParams& p, int q)
{
    const int g = request_gamma(p, q);
    int ell = p.keep[q];
    if (ell < 0 || ell > g) {
        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
        ell = ell < 0 ? 0 : g;
    }
    return ell;
}

// ----------------------------------------------------------------- target row statistics

constexpr int kRowWarps = 8;
constexpr int kRowBlocksPerWarp = 8;   // 1024 columns per warp: four 16-byte loads per lane

// Block (max, sum exp2) of z/T (log2 units) for the 8 consecutive 128-wide blocks starting at
// block b0, one warp; lane bb < 8 receives block b0 + bb. In the bf16 vector path four lanes share
// a block: lane 4bb + qq reads columns 32j + 8qq .. +7 (j = 0..3) of block b0 + bb, so each of the
// four 16-byte loads (row_load8, all issued before any use) covers 64 contiguous bytes of every
// block; row_reduce8 takes the maximum on packed bf16 pairs and the sum with one fused
// multiply-add and one SFU exponential an element, then two shuffle steps within the four lanes.
template <typename T>
__device__ __forceinline__ void row_load8(const T* row, int V, int b0, int lane, uint4 (&raw)[4])
{
    const int bb = lane >> 2, qq = lane & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int v = (b0 + bb) * kNoiseBlock + j * 32 + qq * 8;
        raw[j] = v < V ? __ldg(reinterpret_cast<const uint4*>(row + v)) : make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float2 row_reduce8(const uint4 (&raw)[4], int V, int b0, float scale, int lane)
{
    const int bb = lane >> 2, qq = lane & 3;
    // columns past V: the whole 8-column group is out (V % 8 == 0)
    bool in[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) in[j] = (b0 + bb) * kNoiseBlock + j * 32 + qq * 8 < V;
    uint32_t mx2 = 0xFF80FF80u;   // (-inf, -inf)
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (in[j]) mx2 = bf16x2_max(bf16x2_max(mx2, bf16x2_max(raw[j].x, raw[j].y)), bf16x2_max(raw[j].z, raw[j].w));
    float mr = fmaxf(__uint_as_float(mx2 << 16), __uint_as_float(mx2 & 0xFFFF0000u));
    mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 1));
    mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, 2));
    const float m = mr * scale;   // the block maximum of z/T in log2 units (scale > 0)
    float s0 = 0.f, s1 = 0.f;
    if (m > -INFINITY) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (!in[j]) continue;
            const uint32_t w4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                s0 += ex2(fmaf(__uint_as_float(w4[h] << 16), scale, -m));
                s1 += ex2(fmaf(__uint_as_float(w4[h] & 0xFFFF0000u), scale, -m));
            }
        }
    }
    float sacc = s0 + s1;
    sacc += __shfl_xor_sync(0xffffffffu, sacc, 1);
    sacc += __shfl_xor_sync(0xffffffffu, sacc, 2);
    // lane bb < 8 takes block bb's statistics from lane 4bb
    const int src = (lane & 7) * 4;
    return make_float2(__shfl_sync(0xffffffffu, m, src), __shfl_sync(0xffffffffu, sacc, src));
}

template <typename T>
__device__ __forceinline__ float2 row_block_stats8(const T* row, int V, int b0, float scale, int lane, bool vec)
{
    if (vec && sizeof(T) == 2) {
        uint4 raw[4];
        row_load8(row, V, b0, lane, raw);
        return row_reduce8(raw, V, b0, scale, lane);
    }
    float2 mine = make_float2(-INFINITY, 0.f);
#pragma unroll 1
    for (int bb = 0; bb < kRowBlocksPerWarp; ++bb) {
        const int b = b0 + bb;
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int v = b * kNoiseBlock + e * 32 + lane;
            x[e] = v < V ? ld(row, v) * scale : -INFINITY;
        }
        float m = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        m = warp_max(m);
        float sacc = 0.f;
        if (m > -INFINITY) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc += exp2f(x[e] - m);
        }
        sacc = warp_sum(sacc);
        if (lane == bb) mine = make_float2(m, sacc);
    }
    return mine;
}

// Greedy requests (temperature 0): per 128-wide block the maximum of the raw target logits and
// the lowest index attaining it, stored as (max, index) in the statistics slot.
template <typename T>
__device__ __forceinline__ float2 row_block_argmax(const T* row, int V, int b, int lane, bool& nonfinite)
{
    float m = -INFINITY;
    int mi = -1;
#pragma unroll
    for (int e = 0; e < 4; ++e) {   // lane's columns in increasing order: a later equal value never wins
        const int v = b * kNoiseBlock + e * 32 + lane;
        if (v < V) {
            const float x = ld(row, v);
            if (x != x || x == INFINITY) nonfinite = true;
            if (x > m || mi < 0) {
                m = x;
                mi = v;
            }
        }
    }
    const ArgMax best = warp_argmax(ArgMax{m, mi});
    return make_float2(best.v, (float)best.i);   // indices below 2^24 are exact in fp32
}

// grid (vocabulary chunks, R): the CTA walks target rows 0..keep[r] of its request. Row 0 is
// verified whatever keep is (rows 0..keep), and its statistics read only inputs: they are formed
// before the dependency wait, while the scheduler runs, and stored after it (the workspace may
// still be read by the kernel before this one); rows 1..keep follow once keep exists.
//
// a NaN or +inf logit leaves a NaN sum or an infinite maximum (-inf is a zero weight)
__device__ __forceinline__ void check_row_stats(const VerifyParams& p, int b0, int lane, float2 st, bool& nonfinite)
{
    if (lane < kRowBlocksPerWarp && b0 + lane < p.nblk && (!(st.y >= 0.f) || st.x == INFINITY || st.x != st.x))
        nonfinite = true;
}

// This warp's statistics of row i for blocks b0 .. b0 + 7, held by lanes 0-7 (lane bb: block b0 + bb)
template <typename T>
__device__ __forceinline__ float2 row_stats_of(const VerifyParams& p, int q, int i, int b0, bool greedy, float scale,
                                               bool vec, int lane, bool& nonfinite)
{
    const T* row = static_cast<const T*>(p.target) + ((size_t)q * (p.G + 1) + i) * p.V;
    float2 mine = make_float2(-INFINITY, 0.f);
    if (greedy) {
        for (int bb = 0; bb < kRowBlocksPerWarp && b0 + bb < p.nblk; ++bb) {
            const float2 st = row_block_argmax<T>(row, p.V, b0 + bb, lane, nonfinite);
            if (lane == bb) mine = st;
        }
        return mine;
    }
    mine = row_block_stats8<T>(row, p.V, b0, scale, lane, vec);
    check_row_stats(p, b0, lane, mine, nonfinite);
    return mine;
}

// The merge of this warp's 8 block statistics (lanes 0-7; lane 0 receives it): (max, sum) in log2
// units, or the (max, lowest index) of a greedy row.
__device__ __forceinline__ float2 merge_row_part(const VerifyParams& p, int b0, int lane, float2 v, bool greedy)
{
    const bool in = lane < kRowBlocksPerWarp && b0 + lane < p.nblk;
    float m = in ? v.x : -INFINITY, x = in ? v.y : (greedy ? -1.f : 0.f);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {   // lanes 0-7: the eight blocks (xor within the group of 8)
        const float mo = __shfl_xor_sync(0xffffffffu, m, o), xo = __shfl_xor_sync(0xffffffffu, x, o);
        if (greedy) {
            const ArgMax r = argmax_better(ArgMax{m, (int)x}, ArgMax{mo, (int)xo});
            m = r.v;
            x = (float)r.i;
        } else if (mo > -INFINITY) {
            const float M = fmaxf(m, mo);
            x = x * ex2(m - M) + xo * ex2(mo - M);
            m = M;
        }
    }
    return make_float2(m, x);
}

// This warp's statistics of row i, blocks b0 .. b0 + 7 (lane bb holds block b0 + bb), and their
// merge at partial slot b0 / 8.
__device__ __forceinline__ void store_row_stats(const VerifyParams& p, int q, int i, int b0, int lane, float2 v,
                                                bool greedy)
{
    const size_t row = (size_t)q * (p.G + 1) + i;
    if (lane < kRowBlocksPerWarp && b0 + lane < p.nblk) p.row_stats[row * p.nblk + b0 + lane] = v;
    const float2 part = merge_row_part(p, b0, lane, v, greedy);
    if (lane == 0) p.row_part[row * p.npart + b0 / kRowBlocksPerWarp] = part;
}

// A persistent grid walks items (request q, target row i, chunk c of 64 blocks), every warp taking
// 8 blocks of the chunk. Row 0 is verified whatever keep is and reads only inputs: each CTA forms
// up to kRowPre row-0 items before the dependency wait, while the scheduler runs, and stores them
// after it (the workspace may still be read by the kernel before this one). Then the items of
// rows 1..keep[q], numbered through the prefix sum of keep over the requests, are dealt to the
// CTAs in turn, so that a request with many admitted tokens spreads over the whole GPU instead of
// walking its rows one after the other. In the bf16 vector path each warp issues the next item's
// loads before it reduces the current one.
constexpr int kRowPre = 16;
constexpr int kRowCtasPerSm = 4;   // 256 threads at 64 registers: four CTAs fill an SM's registers
__device__ __forceinline__ int cdiv_dev(int a, int b) { return (a + b - 1) / b; }
constexpr int kRowChunk = kRowWarps * kRowBlocksPerWarp;   // blocks per item

struct RowItem {
    int q, i, b0;   // q < 0: none
};

// Issue the loads of item `it` (bf16 vector path, temperature > 0); false: row_finish reads it
// itself. s_scale[q]: log2(e) / T of request q, 0 for a greedy request.
template <typename T>
__device__ __forceinline__ bool row_start(const VerifyParams& p, const float* s_scale, const RowItem& it, bool vec,
                                          int lane, uint4 (&raw)[4])
{
    if (sizeof(T) != 2 || !vec || it.q < 0 || it.b0 >= p.nblk || s_scale[it.q] == 0.f) return false;
    row_load8(static_cast<const T*>(p.target) + ((size_t)it.q * (p.G + 1) + it.i) * p.V, p.V, it.b0, lane, raw);
    return true;
}

// The warp's 8 block statistics of item `it` (lanes 0-7); greedy for a temperature-0 request
template <typename T>
__device__ __forceinline__ float2 row_finish(const VerifyParams& p, const float* s_scale, const RowItem& it,
                                             bool started, const uint4 (&raw)[4], bool vec, int lane,
                                             bool& nonfinite, bool& greedy)
{
    greedy = s_scale[it.q] == 0.f;
    const float scale = greedy ? 1.f : s_scale[it.q];
    if (!started) return row_stats_of<T>(p, it.q, it.i, it.b0, greedy, scale, vec, lane, nonfinite);
    const float2 st = row_reduce8(raw, p.V, it.b0, scale, lane);
    check_row_stats(p, it.b0, lane, st, nonfinite);
    return st;
}

template <typename T>
__global__ void __launch_bounds__(kRowWarps * 32) verify_rows_kernel(VerifyParams p)
{
    extern __shared__ int s_pref[];   // [R + 1]: rows 1..keep of requests 0 .. q-1, then s_scale [R]
    float* s_scale = reinterpret_cast<float*>(s_pref + p.R + 1);
    __shared__ int s_wsum[kRowWarps];
    // row-0 statistics formed before the wait, held until it: lane l < 8 of each warp per item, the
    // warp's merge of them, and the item's request (-1: none)
    __shared__ float2 s_pre[kRowPre][kRowWarps][kRowBlocksPerWarp];
    __shared__ float2 s_pre_part[kRowPre][kRowWarps];
    __shared__ int s_pre_q[kRowPre];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool vec = (p.V % 8 == 0) && ((reinterpret_cast<uintptr_t>(p.target) & 15u) == 0);
    const int nch = cdiv_dev(p.nblk, kRowChunk);
    const int n0 = p.R * nch;   // row-0 items
    const int wb = warp * kRowBlocksPerWarp;
    bool nonfinite = false;
    uint4 rc[4], rn[4];
    for (int q = threadIdx.x; q < p.R; q += kRowWarps * 32) {   // an input: read before the wait
        const float temp = p.temperature[q];
        s_scale[q] = temp == 0.f ? 0.f : kLog2e / temp;
    }
    __syncthreads();

    // before the wait: row 0 of items blockIdx.x + k * gridDim.x, k < kRowPre (a warp whose 8
    // blocks lie past the vocabulary skips its part)
    const auto pre_item = [&](int k) {
        const int it = blockIdx.x + k * gridDim.x;
        if (k >= kRowPre || it >= n0) return RowItem{-1, 0, 0};
        return RowItem{it / nch, 0, (it % nch) * kRowChunk + wb};
    };
    {
        RowItem c = pre_item(0);
        bool fc = row_start<T>(p, s_scale, c, vec, lane, rc);
        for (int k = 0; c.q >= 0; ++k) {
            const RowItem n = pre_item(k + 1);
            const bool fn = row_start<T>(p, s_scale, n, vec, lane, rn);
            if (c.b0 < p.nblk) {
                bool greedy;
                const float2 st = row_finish<T>(p, s_scale, c, fc, rc, vec, lane, nonfinite, greedy);
                const float2 part = merge_row_part(p, c.b0, lane, st, greedy);
                if (lane < kRowBlocksPerWarp) s_pre[k][warp][lane] = st;
                if (lane == 0) s_pre_part[k][warp] = part;
            }
            if (threadIdx.x == 0) s_pre_q[k] = c.q;
            c = n;
            fc = fn;
#pragma unroll
            for (int j = 0; j < 4; ++j) rc[j] = rn[j];
        }
    }
    if (threadIdx.x == 0)
        for (int k = 0; k < kRowPre; ++k)
            if (blockIdx.x + k * gridDim.x >= n0) s_pre_q[k] = -1;
    __syncthreads();
    pdl_enter();   // keep comes from the scheduler
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.n_rej = 0;   // verify_decide counts from zero
    for (int k = 0; k < kRowPre && s_pre_q[k] >= 0; ++k) {
        const int b0 = ((blockIdx.x + k * gridDim.x) % nch) * kRowChunk + wb;
        if (b0 < p.nblk) {
            const size_t row = (size_t)s_pre_q[k] * (p.G + 1);   // row 0 of the request
            if (lane < kRowBlocksPerWarp && b0 + lane < p.nblk) p.row_stats[row * p.nblk + b0 + lane] = s_pre[k][warp][lane];
            if (lane == 0) p.row_part[row * p.npart + b0 / kRowBlocksPerWarp] = s_pre_part[k][warp];
        }
    }
    // exclusive prefix over the requests of their rows 1..keep (each thread a run of requests)
    const int per = cdiv_dev(p.R, kRowWarps * 32), q_lo = threadIdx.x * per, q_hi = min(p.R, q_lo + per);
    int run = 0;
    for (int q = q_lo; q < q_hi; ++q) run += request_keep(p, q);
    int inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_wsum[warp] = inc;
    __syncthreads();
    int base = inc - run;
    for (int w = 0; w < warp; ++w) base += s_wsum[w];
    for (int q = q_lo; q < q_hi; ++q) {
        s_pref[q] = base;
        base += request_keep(p, q);
    }
    if (threadIdx.x == kRowWarps * 32 - 1) s_pref[p.R] = base;
    __syncthreads();
    const int n_left0 = max(0, n0 - kRowPre * (int)gridDim.x);   // row-0 items not formed before the wait
    const int n_items = n_left0 + s_pref[p.R] * nch;
    const auto post_item = [&](int it) {
        if (it >= n_items) return RowItem{-1, 0, 0};
        if (it < n_left0) {
            const int j = kRowPre * gridDim.x + it;
            return RowItem{j / nch, 0, (j % nch) * kRowChunk + wb};
        }
        const int rr = (it - n_left0) / nch;
        int lo = 0, hi = p.R - 1;   // the last q with s_pref[q] <= rr: its row rr - s_pref[q] + 1
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pref[mid] <= rr)
                lo = mid;
            else
                hi = mid - 1;
        }
        return RowItem{lo, rr - s_pref[lo] + 1, ((it - n_left0) % nch) * kRowChunk + wb};
    };
    int it = blockIdx.x;
    RowItem c = post_item(it);
    bool fc = row_start<T>(p, s_scale, c, vec, lane, rc);
    while (c.q >= 0) {
        it += gridDim.x;
        const RowItem n = post_item(it);
        const bool fn = row_start<T>(p, s_scale, n, vec, lane, rn);
        if (c.b0 < p.nblk) {
            bool greedy;
            const float2 st = row_finish<T>(p, s_scale, c, fc, rc, vec, lane, nonfinite, greedy);
            store_row_stats(p, c.q, c.i, c.b0, lane, st, greedy);
        }
        c = n;
        fc = fn;
#pragma unroll
        for (int j = 0; j < 4; ++j) rc[j] = rn[j];
    }
    if (nonfinite) raise_status(p.status, DSPARK_ERR_NONFINITE_INPUT);
}

// ----------------------------------------------------------------- accept tests and bonus

constexpr int kDecideThreads = 256;
constexpr int kDecidePre = 2;   // block Gumbels formed before the wait: nblk <= 4 * 2 * 256

template <typename T>
__global__ void __launch_bounds__(kDecideThreads) verify_decide_kernel(VerifyParams p)
{
    __shared__ float red[8];
    __shared__ float sv[8];
    __shared__ int si[8];
    __shared__ float lse_s[DSPARK_MAX_GAMMA + 1];
    const int q = blockIdx.x, t = threadIdx.x;
    // keep, the draft outputs and the inputs were complete before the previous kernel started (it
    // waited for the scheduler): the acceptance tests' operands are gathered before the wait, so
    // that only the row log-normalisers are read after it
    const int ell = request_keep(p, q);
    const T* target = static_cast<const T*>(p.target);
    const bool greedy_q = p.temperature[q] == 0.f;
    float a_zt = 0.f, a_lpd = 0.f, a_lu = 0.f;   // thread t < ell: position t's z_t(x) / T, log p_d(x), log u
    if (!greedy_q && t < ell) {
        const size_t o = (size_t)q * p.G + t;
        const int x = checked_index(p.tokens[o], p.V, p.status);
        a_zt = ld(target, ((size_t)q * (p.G + 1) + t) * p.V + x) * (1.f / p.temperature[q]);
        a_lpd = p.draft_logit[o] - p.draft_lse[o];
        a_lu = logf(uniform_at(make_key(p.seed), p.round, kAccept, (uint32_t)q, (uint32_t)t, 0u));
    }
    // the bonus draw's block Gumbels -log(-log u) need only the seed, the round and the request: formed
    // before the wait for blocks 4g4 .. 4g4 + 3, g4 = t + u * kDecideThreads (u < kDecidePre)
    const PhiloxKey key = make_key(p.seed);
    float gb[kDecidePre][4];
#pragma unroll
    for (int u = 0; u < kDecidePre; ++u) {
        const int g4 = t + u * kDecideThreads;
        if (!greedy_q && g4 * 4 < p.nblk) {
            const uint4 w = philox4x32_10(make_uint4((uint32_t)g4, 0u, (uint32_t)q, counter_word3(p.round, kFinalBlock)), key);
            const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) gb[u][j] = -logf(-logf(bits_to_uniform(words[j])));
        }
    }
    pdl_enter();   // the row statistics and the zeroed rejection counter come from verify_rows
    if (greedy_q) {
        // greedy decoding: accept while the draft token equals the target's arg-max; the first
        // mismatch is replaced by that arg-max, else the arg-max of row ell is the bonus token
        __shared__ int s_next;
        int n = ell;
        for (int j = 0; j <= ell; ++j) {
            const float2* pp = p.row_part + ((size_t)q * (p.G + 1) + j) * p.npart;
            ArgMax best{-INFINITY, -1};
            for (int b = t; b < p.npart; b += kDecideThreads) best = argmax_better(best, ArgMax{pp[b].x, (int)pp[b].y});
            best = block_argmax<kDecideThreads>(best, sv, si);
            const int tgt = best.i < 0 ? 0 : best.i;
            if (j == ell || checked_index(p.tokens[(size_t)q * p.G + j], p.V, p.status) != tgt) {
                n = j;
                if (t == 0) s_next = tgt;
                break;   // uniform: every thread sees the same reduction
            }
        }
        __syncthreads();
        if (t == 0) {
            p.accepted[q] = n;
            p.rej[q] = -1;   // nothing for the residual kernels
            p.next_token[q] = s_next;
            p.resampled[q] = n < ell ? 1 : 0;
        }
        return;
    }
    const float invT = 1.f / p.temperature[q];

    // log-normalisers of target rows 0..ell (natural log), one warp per row, from the rows' per-warp
    // partials (max, sum of 2^(z/T log2 e - max)) over 8 blocks each
    const int warp = t >> 5, lane = t & 31;
    for (int i = warp; i <= ell; i += kDecideThreads / 32) {
        const float2* pp = p.row_part + ((size_t)q * (p.G + 1) + i) * p.npart;
        float lm = -INFINITY;
        for (int b = lane; b < p.npart; b += 32) lm = fmaxf(lm, pp[b].x);
        lm = warp_max(lm);
        float acc = 0.f;
        if (lm > -INFINITY)
            for (int b = lane; b < p.npart; b += 32) acc += exp2f(pp[b].x - lm) * pp[b].y;
        acc = warp_sum(acc);
        if (lane == 0) {
            lse_s[i] = (lm + log2f(acc)) * kLn2;
            p.lse_t[(size_t)q * (p.G + 1) + i] = lse_s[i];
        }
    }
    __syncthreads();

    // accept x_j with probability min(1, p_t / p_d): log u < log p_t(x) - log p_d(x)
    int first_reject = ell;
    static_assert(DSPARK_MAX_GAMMA <= kDecideThreads, "one position per thread");
    if (t < ell) {
        const float log_pt = a_zt - lse_s[t];
        if (!(a_lu < log_pt - a_lpd)) first_reject = t;
    }
    const int n = block_min_int<kDecideThreads>(first_reject, si);
    if (t == 0) {
        p.accepted[q] = n;
        p.rej[q] = n < ell ? n : -1;
        if (n < ell) p.rej_list[atomicAdd(p.n_rej, 1)] = q;   // the residual kernel tiles these rows
    }
    if (n < ell) return;   // residual draw happens in residual_pick

    // bonus token from target row ell: two-level Gumbel-max over z_t / T
    const float2* st = p.row_stats + ((size_t)q * (p.G + 1) + ell) * p.nblk;
    ArgMax best{-INFINITY, -1};
#pragma unroll
    for (int u = 0; u < kDecidePre; ++u) {
        const int g4 = t + u * kDecideThreads;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = g4 * 4 + j;
            if (b < p.nblk) best = argmax_better(best, ArgMax{(st[b].x + log2f(st[b].y)) * kLn2 + gb[u][j], b});
        }
    }
    for (int g4 = t + kDecidePre * kDecideThreads; g4 * 4 < p.nblk; g4 += kDecideThreads) {   // V > 2^18
        const uint4 w = philox4x32_10(make_uint4((uint32_t)g4, 0u, (uint32_t)q, counter_word3(p.round, kFinalBlock)), key);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = g4 * 4 + j;
            if (b < p.nblk) {
                const float z = (st[b].x + log2f(st[b].y)) * kLn2 - logf(-logf(bits_to_uniform(words[j])));
                best = argmax_better(best, ArgMax{z, b});
            }
        }
    }
    best = block_argmax<kDecideThreads>(best, sv, si);
    const int bstar = best.i < 0 ? 0 : best.i;
    const int v = bstar * kNoiseBlock + t;
    ArgMax cand{-INFINITY, -1};
    if (t < kNoiseBlock && v < p.V) {   // one thread per column of the block
        const float zt = ld(target, ((size_t)q * (p.G + 1) + ell) * p.V + v) * invT;
        cand = ArgMax{zt + gumbel_at(key, p.round, kFinalElem, (uint32_t)q, 0u, (uint32_t)v), v};
    }
    const ArgMax win = block_argmax<kDecideThreads>(cand, sv, si);
    if (t == 0) {
        int tok = win.i;
        if (tok < 0) {
            raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
            tok = min(bstar * kNoiseBlock, p.V - 1);
        }
        p.next_token[q] = tok;
        p.resampled[q] = 0;
    }
}

// ----------------------------------------------------------------- residual block sums (CUDA cores)

constexpr int kResReq = 8;

struct ResRequest {
    int active, n, prev, use_bias;
    float invT, lse_d, lse_t;
};

__device__ __forceinline__ ResRequest residual_request(const VerifyParams& p, int q)
{
    ResRequest s{0, 0, 0, 0, 0.f, 0.f, 0.f};
    if (q >= p.R) return s;
    const int n = p.rej[q];
    if (n < 0) return s;
    s.active = 1;
    s.n = n;
    s.prev = checked_index(n == 0 ? p.anchor[q] : p.tokens[(size_t)q * p.G + n - 1], p.V, p.status);
    s.use_bias = (n > 0) || p.bias_first;
    s.invT = 1.f / p.temperature[q];
    s.lse_d = p.draft_lse[(size_t)q * p.G + n];
    s.lse_t = p.lse_t[(size_t)q * (p.G + 1) + n];
    return s;
}

template <typename T>
__global__ void __launch_bounds__(kNoiseBlock) residual_stats_simt_kernel(VerifyParams p)
{
    pdl_enter();   // the rejected positions come from verify_decide
    extern __shared__ float es[];   // [kResReq][r]
    __shared__ ResRequest req[kResReq];
    __shared__ float red[8];
    const int b = blockIdx.x, q0 = blockIdx.y * kResReq, t = threadIdx.x;
    if (t < kResReq) req[t] = residual_request(p, q0 + t);
    __syncthreads();
    bool any = false;
#pragma unroll
    for (int j = 0; j < kResReq; ++j) any |= req[j].active != 0;
    if (!any) return;
    const T* E = static_cast<const T*>(p.E);
    const T* W = static_cast<const T*>(p.W);
    for (int i = t; i < kResReq * p.r; i += blockDim.x) {
        const int j = i / p.r, c = i % p.r;
        // the bias operand of the rejected position: the sampler's reported row, else W_1[x_{n-1}]
        es[i] = (req[j].active && req[j].use_bias)
                    ? (p.a_rows ? p.a_rows[((size_t)(q0 + j) * p.G + req[j].n) * p.r + c]
                                : ld(E, (size_t)req[j].prev * p.r + c))
                    : 0.f;
    }
    __syncthreads();
    const int v = b * kNoiseBlock + t;
    float acc[kResReq];
#pragma unroll
    for (int j = 0; j < kResReq; ++j) acc[j] = 0.f;
    if (v < p.V) {
        for (int i = 0; i < p.r; ++i) {
            const float w = ld(W, (size_t)i * p.V + v);
#pragma unroll
            for (int j = 0; j < kResReq; ++j) acc[j] = fmaf(es[j * p.r + i], w, acc[j]);
        }
    }
    const T* U = static_cast<const T*>(p.U);
    const T* target = static_cast<const T*>(p.target);
#pragma unroll 1
    for (int j = 0; j < kResReq; ++j) {
        if (!req[j].active) continue;
        const int q = q0 + j;
        float res = 0.f;
        if (v < p.V) {
            const float ldv = (ld(U, ((size_t)q * p.G + req[j].n) * p.V + v) + acc[j]) * req[j].invT;
            const float pd = expf(ldv - req[j].lse_d);
            const float zt = ld(target, ((size_t)q * (p.G + 1) + req[j].n) * p.V + v) * req[j].invT;
            const float pt = expf(zt - req[j].lse_t);
            res = fmaxf(pt - pd, 0.f);
        }
        const float s = block_sum<kNoiseBlock>(res, red);
        if (t == 0) p.res_stats[(size_t)q * p.nblk + b] = s;
    }
}

// ----------------------------------------------------------------- residual draw

constexpr int kPickThreads = kBlockGemvThreads;
constexpr int kPickPre = 2;   // block Gumbels formed before the wait: nblk <= 4 * 2 * kPickThreads

template <typename T>
__global__ void __launch_bounds__(kPickThreads) residual_pick_kernel(VerifyParams p)
{
    extern __shared__ float sm_dyn[];   // [r] W_1[prev], then [16][128] K-slice partials
    float* erow = sm_dyn;
    float* part = sm_dyn + ((p.r + 3) & ~3);
    __shared__ float sv[kPickThreads / 32];
    __shared__ int si[kPickThreads / 32];
    __shared__ float red[kPickThreads / 32];
    const int q = blockIdx.x, t = threadIdx.x;
    // The rejected position, the row log-normalisers and the bias operand row come from verify_decide
    // and the sampler, both complete before the kernel this one follows started (it waited for
    // verify_decide): they, and the block Gumbels of the draw, are formed before the dependency wait;
    // only the residual block sums come from that kernel.
    const ResRequest rq = residual_request(p, q);
    if (!rq.active) return;
    const PhiloxKey key = make_key(p.seed);
    const float* rs = p.res_stats + (size_t)q * p.nblk;
    const float2* st = p.row_stats + ((size_t)q * (p.G + 1) + rq.n) * p.nblk;
    const T* E = static_cast<const T*>(p.E);
    const T* W = static_cast<const T*>(p.W);
    for (int i = t; i < p.r; i += kPickThreads)
        erow[i] = rq.use_bias ? (p.a_rows ? p.a_rows[((size_t)q * p.G + rq.n) * p.r + i] : ld(E, (size_t)rq.prev * p.r + i))
                              : 0.f;
    float gb[kPickPre][4];   // -log(-log u) of blocks 4g4 .. 4g4 + 3, g4 = t + u * kPickThreads
#pragma unroll
    for (int u = 0; u < kPickPre; ++u) {
        const int g4 = t + u * kPickThreads;
        if (g4 * 4 < p.nblk) {
            const uint4 w = philox4x32_10(make_uint4((uint32_t)g4, 0u, (uint32_t)q, counter_word3(p.round, kFinalBlock)), key);
            const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) gb[u][j] = -logf(-logf(bits_to_uniform(words[j])));
        }
    }
    pdl_enter();   // the residual block sums come from the residual statistics kernel
    // residual mass anywhere?
    float tot = 0.f;
    for (int b = t; b < p.nblk; b += kPickThreads) tot += rs[b];
    tot = block_sum<kPickThreads>(tot, red);
    const bool fallback = !(tot > 0.f);   // zero only through rounding: draw from p_t of the row
    // block level, one Philox call per 4 consecutive blocks (formed above for the first kPickPre)
    ArgMax best{-INFINITY, -1};
    const auto block_key = [&](int b, float g) {
        float L;
        if (fallback) {
            L = (st[b].x + log2f(st[b].y)) * kLn2;
        } else {
            if (!(rs[b] > 0.f)) return;
            L = logf(rs[b]);
        }
        best = argmax_better(best, ArgMax{L + g, b});
    };
#pragma unroll
    for (int u = 0; u < kPickPre; ++u) {
        const int g4 = t + u * kPickThreads;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (g4 * 4 + j < p.nblk) block_key(g4 * 4 + j, gb[u][j]);
    }
    for (int g4 = t + kPickPre * kPickThreads; g4 * 4 < p.nblk; g4 += kPickThreads) {   // V > 2^18
        const uint4 w = philox4x32_10(make_uint4((uint32_t)g4, 0u, (uint32_t)q, counter_word3(p.round, kFinalBlock)), key);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (g4 * 4 + j < p.nblk) block_key(g4 * 4 + j, -logf(-logf(bits_to_uniform(words[j]))));
    }
    best = block_argmax<kPickThreads>(best, sv, si);
    const int bstar = best.i < 0 ? 0 : best.i;
    // element level inside the chosen block
    float bias = 0.f;
    if (!fallback && rq.use_bias) bias = block_bias<T>(erow, W, p.V, p.r, bstar * kNoiseBlock, part);
    const int v = bstar * kNoiseBlock + t;
    ArgMax cand{-INFINITY, -1};
    if (t < kNoiseBlock && v < p.V) {
        const T* target = static_cast<const T*>(p.target);
        const float zt = ld(target, ((size_t)q * (p.G + 1) + rq.n) * p.V + v) * rq.invT;
        float L = -INFINITY;
        if (fallback) {
            L = zt;
        } else {
            const T* U = static_cast<const T*>(p.U);
            const float ldv = (ld(U, ((size_t)q * p.G + rq.n) * p.V + v) + bias) * rq.invT;
            const float res = expf(zt - rq.lse_t) - expf(ldv - rq.lse_d);
            if (res > 0.f) L = logf(res);
        }
        if (L > -INFINITY) cand = ArgMax{L + gumbel_at(key, p.round, kFinalElem, (uint32_t)q, 0u, (uint32_t)v), v};
    }
    const ArgMax win = block_argmax<kPickThreads>(cand, sv, si);
    if (t == 0) {
        int tok = win.i;
        if (tok < 0) {
            raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
            tok = min(bstar * kNoiseBlock, p.V - 1);
        }
        p.next_token[q] = tok;
        p.resampled[q] = 1;
    }
}

// ----------------------------------------------------------------- launchers

template <typename T>
int row_grid(const VerifyParams& p, size_t smem)
{
    // as many CTAs as are resident at once while the scheduler still runs, at most one per item: a
    // CTA that started late would form its row-0 items after the wait
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_rows_kernel<T>, kRowWarps * 32, smem) !=
            cudaSuccess ||
        per_sm <= 0) {
        (void)cudaGetLastError();
        per_sm = 1;
    }
    const long long items = (long long)p.R * (p.G + 1) * cdiv(p.nblk, kRowChunk);
    const int sms = std::max(1, num_sms() - kScheduleCtas);   // the scheduler's SMs are full until it ends
    return (int)std::min<long long>(items, (long long)std::min(per_sm, kRowCtasPerSm) * sms);
}

cudaError_t launch_verify_rows(const VerifyParams& p, cudaStream_t s)
{
    const size_t smem = sizeof(int) * ((size_t)p.R + 1) + sizeof(float) * (size_t)p.R;   // R <= DSPARK_MAX_SLOTS
    static bool smem_set = false;
    if (!smem_set) {   // above the default 48 KB at the largest R
        const int most = (int)(sizeof(int) * (DSPARK_MAX_SLOTS + 1) + sizeof(float) * DSPARK_MAX_SLOTS);
        if (cudaFuncSetAttribute(verify_rows_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, most) !=
                cudaSuccess ||
            cudaFuncSetAttribute(verify_rows_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, most) !=
                cudaSuccess)
            return cudaGetLastError();
        smem_set = true;
    }
    const cudaError_t e =
        p.dtype == DSPARK_BF16
            ? launch_pdl(verify_rows_kernel<__nv_bfloat16>, row_grid<__nv_bfloat16>(p, smem), kRowWarps * 32, smem, s, p)
            : launch_pdl(verify_rows_kernel<float>, row_grid<float>(p, smem), kRowWarps * 32, smem, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

int verify_row_partials(int nblk) { return cdiv(nblk, kRowBlocksPerWarp); }

cudaError_t launch_verify_decide(const VerifyParams& p, cudaStream_t s)
{
    const cudaError_t e = p.dtype == DSPARK_BF16
                              ? launch_pdl(verify_decide_kernel<__nv_bfloat16>, p.R, kDecideThreads, 0, s, p)
                              : launch_pdl(verify_decide_kernel<float>, p.R, kDecideThreads, 0, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_residual_stats_simt(const VerifyParams& p, cudaStream_t s)
{
    const dim3 grid(p.nblk, cdiv(p.R, kResReq));
    const size_t smem = (size_t)kResReq * p.r * sizeof(float);
    if (p.dtype == DSPARK_BF16) {
        cudaFuncSetAttribute(residual_stats_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        const cudaError_t e = launch_pdl(residual_stats_simt_kernel<__nv_bfloat16>, grid, kNoiseBlock, smem, s, p);
        if (e != cudaSuccess) return e;
    } else {
        cudaFuncSetAttribute(residual_stats_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        const cudaError_t e = launch_pdl(residual_stats_simt_kernel<float>, grid, kNoiseBlock, smem, s, p);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_residual_pick(const VerifyParams& p, cudaStream_t s)
{
    const size_t smem = (size_t)(((p.r + 3) & ~3) + 16 * kNoiseBlock) * sizeof(float);
    const cudaError_t e = p.dtype == DSPARK_BF16
                              ? launch_pdl(residual_pick_kernel<__nv_bfloat16>, p.R, kPickThreads, smem, s, p)
                              : launch_pdl(residual_pick_kernel<float>, p.R, kPickThreads, smem, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
