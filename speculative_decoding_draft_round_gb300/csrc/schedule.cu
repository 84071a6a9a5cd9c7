// schedule.cu -- hardware-aware prefix scheduler, one CTA.
//
// Algorithm 1 of "DSpark" (zhongzhuzhou.org notes, hardware-aware prefix
// scheduler; caijizhuo.github.io section 4 "admit"), plus the asynchronous
// capacity variant of the paper's section 5.2:
//   pool   {(r, j): j <= gamma_r, a_{r,j} > 0}, sorted by a descending, then
//          r, then j ascending (ties keep prefixes closed, Lemma 1);
//   tau_m  = R + sum of the first m a's;  Theta_m = tau_m * SPS(R + m);
//   sync   m* = (first m with Theta_m <= Theta_{m-1}) - 1;
//   full   m* = smallest arg-max of Theta_m;
//   async  K  = full-scan count over the survivals two rounds old,
//          m* = min(K, |pool|) over the current ranking.
// GB300 mapping: up to 8192 slots live in shared memory. A positive float's bit
// pattern orders like an unsigned integer, so the sort is a stable LSD radix
// sort (four 8-bit digits, warp-aggregated ranks via __match_any_sync) of the
// complemented bits; stability in slot order gives the (r, j) tie-break for
// free. Prefix sums are exact 64-bit fixed-point sums (a in units of 2^-48),
// so they do not depend on the summation order; Theta is formed in double.
#include "common.cuh"
#include "internal.h"

namespace dspark {

constexpr int kSchedThreads = 1024;
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr int kKeysPerWarp = DSPARK_MAX_SLOTS / kSchedWarps;   // 256
constexpr int kItems = kKeysPerWarp / 32;                      // 8 per lane
constexpr int kDigits = 256;

struct SchedSmem {
    uint32_t key[2][DSPARK_MAX_SLOTS];
    uint16_t val[2][DSPARK_MAX_SLOTS];
    uint32_t hist[kSchedWarps * kDigits];   // per-warp digit counts, then offsets; reused for keep counts
    uint32_t dbase[kDigits];
    uint32_t wtot[kDigits / 32];
    unsigned long long wsum[kSchedWarps];
    double wbest[kSchedWarps];
    int wbest_m[kSchedWarps];
    int n_pool;
    int first_bad;
};

size_t schedule_smem_bytes() { return sizeof(SchedSmem); }

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Load the pool keys of `src` ([R][G] survivals) into key[0]/val[0]; returns |pool|.
__device__ int load_pool(SchedSmem& sm, const ScheduleParams& p, const float* src, int n_slots, int n_pad)
{
    if (threadIdx.x == 0) sm.n_pool = 0;
    __syncthreads();
    int cnt = 0;
    for (int s = threadIdx.x; s < n_pad; s += kSchedThreads) {
        uint32_t key = 0xFFFFFFFFu;
        if (s < n_slots) {
            const int q = s / p.G, j = s % p.G;
            int g = p.gamma ? p.gamma[q] : p.G;
            if (g < 0 || g > p.G) {
                raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                g = g < 0 ? 0 : p.G;
            }
            float a = src[s];
            if (j < g && a > 0.f) {   // NaN and non-positive survivals are not in the pool
                if (!(a <= 1.f)) {
                    raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                    a = 1.f;
                }
                key = ~__float_as_uint(a);
                ++cnt;
            }
        }
        sm.key[0][s] = key;
        sm.val[0][s] = (uint16_t)s;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(&sm.n_pool, cnt);
    __syncthreads();
    return sm.n_pool;
}

// One stable counting pass on 8 bits of the key, buffer `in` -> 1 - in.
__device__ void radix_pass(SchedSmem& sm, int in, int shift, int active_warps)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < kSchedWarps * kDigits; i += kSchedThreads) sm.hist[i] = 0;
    __syncthreads();
    uint32_t key[kItems], dig[kItems], rank[kItems];
    uint16_t val[kItems];
    if (warp < active_warps) {
        uint32_t* h = sm.hist + warp * kDigits;
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int idx = warp * kKeysPerWarp + it * 32 + lane;   // striped: order = (warp, it, lane)
            key[it] = sm.key[in][idx];
            val[it] = sm.val[in][idx];
            dig[it] = (key[it] >> shift) & (kDigits - 1);
            const uint32_t peers = __match_any_sync(0xffffffffu, dig[it]);
            const uint32_t base = h[dig[it]];
            __syncwarp();
            if (lane == __ffs(peers) - 1) h[dig[it]] = base + __popc(peers);
            __syncwarp();
            rank[it] = base + __popc(peers & lanemask_lt());
        }
    }
    __syncthreads();
    // exclusive offsets in digit-major, warp-minor order: thread d turns the
    // per-warp counts of digit d into offsets within the digit, then the 256
    // digit totals are scanned (8 warps: shuffle scan + warp totals)
    uint32_t tot = 0, inc = 0;
    if (tid < kDigits) {
        for (int w = 0; w < kSchedWarps; ++w) {
            const uint32_t c = sm.hist[w * kDigits + tid];
            sm.hist[w * kDigits + tid] = tot;
            tot += c;
        }
        inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) sm.wtot[warp] = inc;
    }
    __syncthreads();
    if (tid < kDigits) {
        uint32_t add = 0;
        for (int w = 0; w < warp; ++w) add += sm.wtot[w];
        sm.dbase[tid] = add + inc - tot;
    }
    __syncthreads();
    const int out = 1 - in;
    if (warp < active_warps) {
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const uint32_t pos = sm.dbase[dig[it]] + sm.hist[warp * kDigits + dig[it]] + rank[it];
            sm.key[out][pos] = key[it];
            sm.val[out][pos] = val[it];
        }
    }
    __syncthreads();
}

// Sort key[0]/val[0] ascending (a descending); result in buffer 0.
__device__ void sort_pool(SchedSmem& sm, int n_pad)
{
    const int active_warps = n_pad / kKeysPerWarp;
    radix_pass(sm, 0, 0, active_warps);
    radix_pass(sm, 1, 8, active_warps);
    radix_pass(sm, 0, 16, active_warps);
    radix_pass(sm, 1, 24, active_warps);
}

__device__ __forceinline__ unsigned long long fixed48(uint32_t key)
{
    const float a = __uint_as_float(~key);
    return __float2ull_rn(a * 281474976710656.0f);   // a * 2^48, exact scaling
}

__device__ __forceinline__ double theta_of(int R, int m, unsigned long long S, const float* sps)
{
    const double tau = (double)R + (double)S * 0x1p-48;
    return tau * (double)sps[R + m - 1];
}

// Inclusive prefix sums S_i (i = sorted index) of the fixed-point a's for the
// `kItems` consecutive indices this thread owns, plus the exclusive prefix.
__device__ void prefix_sums(SchedSmem& sm, int n, unsigned long long S[kItems], unsigned long long& excl)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned long long run = 0;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const int i = tid * kItems + it;
        run += i < n ? fixed48(sm.key[0][i]) : 0ull;
        S[it] = run;
    }
    unsigned long long inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) sm.wsum[warp] = inc;
    __syncthreads();
    unsigned long long wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += sm.wsum[w];
    excl = wbase + inc - run;
#pragma unroll
    for (int it = 0; it < kItems; ++it) S[it] += excl;
    __syncthreads();
}

// Smallest arg-max of Theta_m over m = 0..n (full scan).
__device__ int full_scan(SchedSmem& sm, int R, int n, const float* sps)
{
    unsigned long long S[kItems], excl;
    prefix_sums(sm, n, S, excl);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    double best = -1.0;
    int bm = INT32_MAX;
    if (tid == 0) {
        best = theta_of(R, 0, 0ull, sps);
        bm = 0;
    }
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const int i = tid * kItems + it;
        if (i < n) {
            const double th = theta_of(R, i + 1, S[it], sps);
            if (th > best) {
                best = th;
                bm = i + 1;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int om = __shfl_xor_sync(0xffffffffu, bm, o);
        if (ob > best || (ob == best && om < bm)) {
            best = ob;
            bm = om;
        }
    }
    if (lane == 0) {
        sm.wbest[warp] = best;
        sm.wbest_m[warp] = bm;
    }
    __syncthreads();
    double b = -1.0;
    int m = INT32_MAX;
    for (int w = 0; w < kSchedWarps; ++w) {
        if (sm.wbest[w] > b || (sm.wbest[w] == b && sm.wbest_m[w] < m)) {
            b = sm.wbest[w];
            m = sm.wbest_m[w];
        }
    }
    __syncthreads();
    return m;
}

// First m >= 1 with Theta_m <= Theta_{m-1}, minus one (|pool| if none).
__device__ int sync_scan(SchedSmem& sm, int R, int n, const float* sps)
{
    unsigned long long S[kItems], excl;
    prefix_sums(sm, n, S, excl);
    const int tid = threadIdx.x;
    if (tid == 0) sm.first_bad = INT32_MAX;
    __syncthreads();
    int bad = INT32_MAX;
    double prev = (tid * kItems < n) ? theta_of(R, tid * kItems, excl, sps) : 0.0;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const int i = tid * kItems + it;
        if (i < n) {
            const double th = theta_of(R, i + 1, S[it], sps);
            if (!(th > prev) && bad == INT32_MAX) bad = i + 1;
            prev = th;
        }
    }
    bad = __reduce_min_sync(0xffffffffu, bad);
    if ((tid & 31) == 0 && bad != INT32_MAX) atomicMin(&sm.first_bad, bad);
    __syncthreads();
    const int fb = sm.first_bad;
    __syncthreads();
    return fb == INT32_MAX ? n : fb - 1;
}

__global__ void __launch_bounds__(kSchedThreads, 1) schedule_kernel(ScheduleParams p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SchedSmem& sm = *reinterpret_cast<SchedSmem*>(smem_raw);
    const int n_slots = p.R * p.G;
    const int n_pad = (n_slots + kKeysPerWarp - 1) / kKeysPerWarp * kKeysPerWarp;

    int capacity = -1;
    if (p.mode == DSPARK_SCHED_ASYNC_CAPACITY) {
        const int n_old = load_pool(sm, p, p.surv_capacity, n_slots, n_pad);
        sort_pool(sm, n_pad);
        capacity = full_scan(sm, p.R, n_old, p.sps);
    }
    const int n = load_pool(sm, p, p.surv, n_slots, n_pad);
    sort_pool(sm, n_pad);
    int m_star;
    if (p.mode == DSPARK_SCHED_SYNC)
        m_star = sync_scan(sm, p.R, n, p.sps);
    else if (p.mode == DSPARK_SCHED_FULL_SCAN)
        m_star = full_scan(sm, p.R, n, p.sps);
    else
        m_star = min(capacity, n);

    // keep[r] = l_r, the largest admitted position of request r (Algorithm 1 sets l_r = j on
    // each admission); with survivals non-increasing in j it is also the admitted count
    uint32_t* cnt = sm.hist;
    for (int q = threadIdx.x; q < p.R; q += kSchedThreads) cnt[q] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m_star; i += kSchedThreads) {
        const int slot = sm.val[0][i];
        atomicMax(&cnt[slot / p.G], (uint32_t)(slot % p.G + 1));
    }
    __syncthreads();
    for (int q = threadIdx.x; q < p.R; q += kSchedThreads) p.keep[q] = (int32_t)cnt[q];

    // Theta of the admitted set with the current survivals
    unsigned long long S[kItems], excl;
    prefix_sums(sm, m_star, S, excl);
    const int last = m_star - 1;
    if (m_star == 0 && threadIdx.x == 0) {
        p.stats->theta_best = theta_of(p.R, 0, 0ull, p.sps);
    } else if (last >= 0 && last / kItems == (int)threadIdx.x) {
        p.stats->theta_best = theta_of(p.R, m_star, S[last % kItems], p.sps);
    }
    if (threadIdx.x == 0) {
        p.stats->admitted = m_star;
        p.stats->capacity = capacity;
        p.stats->batch = p.R + m_star;
        p.stats->pool = n;
    }
}

cudaError_t launch_schedule(const ScheduleParams& p, cudaStream_t s)
{
    const size_t smem = sizeof(SchedSmem);
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    schedule_kernel<<<1, kSchedThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace dspark
