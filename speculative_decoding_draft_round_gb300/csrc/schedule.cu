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
// GB300 mapping: up to 8192 slots live in shared memory, spread over all 32
// warps. A positive float's bit pattern orders like an unsigned integer, so the
// sort is a stable LSD radix sort (four 8-bit digits, warp-aggregated ranks via
// __match_any_sync, digit offsets from one block-wide scan of the [digit][warp]
// counts) of the complemented bits; stability in slot order gives the (r, j)
// tie-break for free. Prefix sums are exact 64-bit fixed-point sums (a in units
// of 2^-48), so they do not depend on the summation order, and every Theta
// comparison is exact: tau * 2^48 is an integer below 2^62 and SPS(B) a float,
// so Theta is compared through the 128-bit product of the integer and the
// float's 24-bit significand (normalised to 64 bits: ties closer than 2^-63
// relative compare equal). Only the reported Theta_best is formed in double.
#include "common.cuh"
#include "internal.h"

namespace dspark {

constexpr int kSchedThreads = 1024;
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr int kMaxItems = DSPARK_MAX_SLOTS / kSchedThreads;   // keys per thread, at most 8

struct ThetaKey {
    int e;                  // Theta = m * 2^e with m normalised (bit 63 set); zero: e = INT_MIN, m = 0
    unsigned long long m;
};

constexpr int kDigits = 256;
constexpr int kHist = kDigits * kSchedWarps;                  // [digit][warp] counts

// Position x of a key array lives at sk(x) = x + x / 32: a thread's run of 2, 4 or 8 consecutive
// positions and a warp's 32 consecutive positions both fall in distinct banks.
__device__ __forceinline__ int sk(int x) { return x + (x >> 5); }
constexpr int kSkewed = DSPARK_MAX_SLOTS + DSPARK_MAX_SLOTS / 32;

struct SchedSmem {
    uint32_t key[2][kSkewed];
    uint16_t val[2][kSkewed];
    uint32_t hist[kHist];                   // digit counts, then offsets; reused for keep counts
    uint32_t wpart[kSchedWarps];
    unsigned long long wsum[kSchedWarps];
    ThetaKey wbest[kSchedWarps];
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

// Sorting position of (warp, item, lane): warp-major, then item, then lane; with ni items per
// lane, position order equals slot order when the keys are loaded.
__device__ __forceinline__ int striped(int warp, int it, int lane, int ni) { return (warp * ni + it) * 32 + lane; }

// Load the pool keys of `src` ([R][G] survivals) into key[0]/val[0]; returns |pool|. Every load
// of a thread is issued before any is used.
__device__ __noinline__ int load_pool(SchedSmem& sm, const ScheduleParams& p, const float* src, int n_slots, int ni)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) sm.n_pool = 0;
    float a[kMaxItems];
    int g[kMaxItems];
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        const int s = striped(warp, it, lane, ni);
        const bool in = it < ni && s < n_slots;
        a[it] = in ? src[s] : 0.f;
        g[it] = in ? (p.gamma ? p.gamma[s / p.G] : p.G) : 0;
    }
    int cnt = 0;
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        if (it >= ni) break;
        const int s = striped(warp, it, lane, ni);
        uint32_t key = 0xFFFFFFFFu;
        if (s < n_slots) {
            int gg = g[it];
            if (gg < 0 || gg > p.G) {
                raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                gg = gg < 0 ? 0 : p.G;
            }
            float av = a[it];
            if (s % p.G < gg && av > 0.f) {   // NaN and non-positive survivals are not in the pool
                if (!(av <= 1.f)) {
                    raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                    av = 1.f;
                }
                key = ~__float_as_uint(av);
                ++cnt;
            }
        }
        sm.key[0][sk(s)] = key;
        sm.val[0][sk(s)] = (uint16_t)s;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    __syncthreads();
    if (lane == 0 && cnt) atomicAdd(&sm.n_pool, cnt);
    __syncthreads();
    return sm.n_pool;
}

// Exclusive prefix over the kHist counts in [digit][warp] order, in place (1024 threads, 8 each).
__device__ __noinline__ void scan_hist(SchedSmem& sm)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int per = kHist / kSchedThreads;   // 8
    const uint4 c0 = reinterpret_cast<uint4*>(sm.hist)[2 * tid];
    const uint4 c1 = reinterpret_cast<uint4*>(sm.hist)[2 * tid + 1];
    uint32_t c[per] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint32_t run = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        const uint32_t v = c[i];
        c[i] = run;
        run += v;
    }
    uint32_t inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) sm.wpart[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = sm.wpart[lane];
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        sm.wpart[lane] = wi - w;
    }
    __syncthreads();
    const uint32_t base = sm.wpart[warp] + inc - run;
    reinterpret_cast<uint4*>(sm.hist)[2 * tid] = make_uint4(base + c[0], base + c[1], base + c[2], base + c[3]);
    reinterpret_cast<uint4*>(sm.hist)[2 * tid + 1] = make_uint4(base + c[4], base + c[5], base + c[6], base + c[7]);
}

// One stable counting pass on 8 bits of the key, buffer `in` -> 1 - in.
__device__ __noinline__ void radix_pass(SchedSmem& sm, int in, int shift, int ni)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    reinterpret_cast<uint4*>(sm.hist)[2 * tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(sm.hist)[2 * tid + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    uint32_t key[kMaxItems], dig[kMaxItems], rank[kMaxItems];
    uint16_t val[kMaxItems];
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        if (it >= ni) break;
        const int idx = striped(warp, it, lane, ni);
        key[it] = sm.key[in][sk(idx)];
        val[it] = sm.val[in][sk(idx)];
    }
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        if (it >= ni) break;
        dig[it] = (key[it] >> shift) & (kDigits - 1);
        uint32_t* h = sm.hist + dig[it] * kSchedWarps + warp;
        const uint32_t peers = __match_any_sync(0xffffffffu, dig[it]);
        const uint32_t base = *h;
        __syncwarp();
        if (lane == __ffs(peers) - 1) *h = base + __popc(peers);
        __syncwarp();
        rank[it] = base + __popc(peers & lanemask_lt());
    }
    __syncthreads();
    scan_hist(sm);
    __syncthreads();
    const int out = 1 - in;
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        if (it >= ni) break;
        const uint32_t pos = sm.hist[dig[it] * kSchedWarps + warp] + rank[it];
        sm.key[out][sk(pos)] = key[it];
        sm.val[out][sk(pos)] = val[it];
    }
    __syncthreads();
}

// (key, slot) order: the sort order of the pool (a descending, then slot ascending)
__device__ __forceinline__ bool kv_less(uint32_t ka, uint16_t va, uint32_t kb, uint16_t vb)
{
    return ka < kb || (ka == kb && va < vb);
}

// One level of a merge sort: the sorted runs [2pL, 2pL + L) and [2pL + L, 2pL + 2L) of buffer `in`
// (clipped to n) merge into [2pL, 2pL + 2L) of buffer 1 - in. Thread t writes outputs
// t*ni .. t*ni + ni - 1; it finds where its first output of each pair starts on the merge path by
// a binary search, then merges element by element with the two candidates held in registers.
__device__ __noinline__ void merge_level(SchedSmem& sm, int in, int n, int L, int ni)
{
    const uint32_t* ka = sm.key[in];
    const uint16_t* va = sm.val[in];
    uint32_t* ko = sm.key[1 - in];
    uint16_t* vo = sm.val[1 - in];
    const int o0 = threadIdx.x * ni, o1 = min(o0 + ni, n);
    if (o0 >= o1) return;
    int p0 = o0 / (2 * L) * (2 * L);
    int a = 0, a_end = 0, b = 0, b_end = 0;
    uint32_t kA = 0, kB = 0;
    uint16_t vA = 0, vB = 0;
    for (int o = o0; o < o1; ++o) {
        if (o == p0 + 2 * L) p0 = o;   // the chunk runs into the next pair
        if (o == o0 || o == p0) {      // locate on the merge path of this pair
            const int a0 = p0, a1 = min(p0 + L, n), b0 = a1, b1 = min(p0 + 2 * L, n);
            const int na = a1 - a0, nb = b1 - b0, k = o - p0;
            int lo = max(0, k - nb), hi = min(k, na);
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                const int ai = sk(a0 + mid), bj = sk(b0 + k - mid - 1);
                if (kv_less(ka[ai], va[ai], ka[bj], va[bj]))
                    lo = mid + 1;
                else
                    hi = mid;
            }
            a = a0 + lo;
            a_end = a1;
            b = b0 + k - lo;
            b_end = b1;
            if (a < a_end) {
                kA = ka[sk(a)];
                vA = va[sk(a)];
            }
            if (b < b_end) {
                kB = ka[sk(b)];
                vB = va[sk(b)];
            }
        }
        const bool take_a = b >= b_end || (a < a_end && kv_less(kA, vA, kB, vB));
        const int w = sk(o);
        if (take_a) {
            ko[w] = kA;
            vo[w] = vA;
            if (++a < a_end) {
                kA = ka[sk(a)];
                vA = va[sk(a)];
            }
        } else {
            ko[w] = kB;
            vo[w] = vB;
            if (++b < b_end) {
                kB = ka[sk(b)];
                vB = va[sk(b)];
            }
        }
    }
}

// Sort key[0]/val[0] ascending (a descending, then slot); result in buffer 0. When every
// request's G slots are already in order -- the sampler's survivals are running products of
// confidences below one, so they never increase along a request -- the R runs are merged
// pairwise (log2 R levels); any other input takes the stable LSD radix sort.
__device__ __noinline__ void sort_pool(SchedSmem& sm, int n, int G, int ni)
{
    bool unsorted = false;
    for (int s = threadIdx.x; s < n; s += kSchedThreads)
        if (s % G != G - 1 && s + 1 < n && sm.key[0][sk(s + 1)] < sm.key[0][sk(s)]) unsorted = true;
    if (__syncthreads_or(unsorted)) {
        radix_pass(sm, 0, 0, ni);
        radix_pass(sm, 1, 8, ni);
        radix_pass(sm, 0, 16, ni);
        radix_pass(sm, 1, 24, ni);
        return;
    }
    int in = 0;
    for (int L = G; L < n; L *= 2) {
        merge_level(sm, in, n, L, ni);
        __syncthreads();
        in = 1 - in;
    }
    if (in == 1) {
        for (int s = threadIdx.x; s < n; s += kSchedThreads) {
            sm.key[0][sk(s)] = sm.key[1][sk(s)];
            sm.val[0][sk(s)] = sm.val[1][sk(s)];
        }
        __syncthreads();
    }
}

// a * 2^48 rounded to nearest (ties to even), a in (0, 1] from its word, with integer operations
__device__ __forceinline__ unsigned long long fixed48(uint32_t key)
{
    const uint32_t b = ~key;
    const uint32_t ex = (b >> 23) & 0xFFu;
    const unsigned long long M = ex ? ((b & 0x7FFFFFu) | 0x800000u) : (b & 0x7FFFFFu);
    const int sh = (ex ? (int)ex - 150 : -149) + 48;   // a * 2^48 = M * 2^sh
    if (sh >= 0) return M << sh;
    if (sh < -25) return 0ull;
    const unsigned long long q = M >> -sh, rem = M & ((1ull << -sh) - 1ull), half = 1ull << (-sh - 1);
    return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

// Exact Theta_m = (R + S * 2^-48) * SPS(R + m) as a normalised key (see the header comment).
__device__ __forceinline__ ThetaKey theta_key(int R, unsigned long long S, float sv, int* status)
{
    const unsigned long long T = ((unsigned long long)R << 48) + S;   // < 2^62
    if (!(sv > 0.f) || sv == INFINITY) {
        raise_status(status, DSPARK_ERR_DEVICE_INPUT);   // a throughput table entry must be positive and finite
        return ThetaKey{INT32_MIN, 0ull};
    }
    const uint32_t b = __float_as_uint(sv);
    const uint32_t ex = (b >> 23) & 0xFFu;
    const unsigned long long M = ex ? ((b & 0x7FFFFFu) | 0x800000u) : (b & 0x7FFFFFu);
    const int E = ex ? (int)ex - 150 : -149;   // SPS = M * 2^E
    const unsigned long long lo = T * M, hi = __umul64hi(T, M);
    if (hi == 0ull && lo == 0ull) return ThetaKey{INT32_MIN, 0ull};
    // Theta = (hi * 2^64 + lo) * 2^(E - 48)
    if (hi) {
        const int lz = __clzll(hi);
        const unsigned long long m64 = (hi << lz) | (lz ? lo >> (64 - lz) : 0ull);
        // m64 holds bits [127 - lz - 63, 127 - lz] of the product: Theta = m64 * 2^(64 - lz + E - 48)
        return ThetaKey{64 - lz + E - 48, m64};
    }
    const int lz = __clzll(lo);
    return ThetaKey{E - 48 - lz, lo << lz};   // Theta = (lo << lz) * 2^(E - 48 - lz)
}

__device__ __forceinline__ bool key_gt(ThetaKey a, ThetaKey b) { return a.e > b.e || (a.e == b.e && a.m > b.m); }

__device__ __forceinline__ double theta_of(int R, int m, unsigned long long S, const float* sps)
{
    const double tau = (double)R + (double)S * 0x1p-48;
    return tau * (double)sps[R + m - 1];
}

// Inclusive prefix sums S (sorted index tid * ni + it) of the fixed-point a's, and the exclusive
// prefix of the thread's first index.
__device__ __noinline__ void prefix_sums(SchedSmem& sm, int n, int ni, unsigned long long (&S)[kMaxItems], unsigned long long& excl)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned long long run = 0;
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        const int i = tid * ni + it;
        run += (it < ni && i < n) ? fixed48(sm.key[0][sk(i)]) : 0ull;
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
    if (warp == 0) {
        const unsigned long long w = sm.wsum[lane];
        unsigned long long wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        sm.wsum[lane] = wi - w;
    }
    __syncthreads();
    excl = sm.wsum[warp] + inc - run;
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) S[it] += excl;
    __syncthreads();
}

// Smallest arg-max of Theta_m over m = 0..n (full scan), from the prefix sums.
__device__ __noinline__ int full_scan(SchedSmem& sm, const ScheduleParams& p, int n, int ni, const unsigned long long (&S)[kMaxItems],
                         const float (&sv)[kMaxItems + 1])
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    ThetaKey best{INT32_MIN, 0ull};
    int bm = INT32_MAX;
    if (tid == 0) {
        best = theta_key(p.R, 0ull, sv[0], p.status);
        bm = 0;
    }
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        const int i = tid * ni + it;
        if (it < ni && i < n) {
            const ThetaKey th = theta_key(p.R, S[it], sv[it + 1], p.status);
            if (key_gt(th, best) || bm == INT32_MAX) {
                best = th;
                bm = i + 1;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const ThetaKey ob{__shfl_xor_sync(0xffffffffu, best.e, o), __shfl_xor_sync(0xffffffffu, best.m, o)};
        const int om = __shfl_xor_sync(0xffffffffu, bm, o);
        if (om != INT32_MAX && (bm == INT32_MAX || key_gt(ob, best) || (!key_gt(best, ob) && om < bm))) {
            best = ob;
            bm = om;
        }
    }
    if (lane == 0) {
        sm.wbest[warp] = best;
        sm.wbest_m[warp] = bm;
    }
    __syncthreads();
    ThetaKey b{INT32_MIN, 0ull};
    int m = INT32_MAX;
    for (int w = 0; w < kSchedWarps; ++w) {
        const ThetaKey wb = sm.wbest[w];
        const int wm = sm.wbest_m[w];
        if (wm != INT32_MAX && (m == INT32_MAX || key_gt(wb, b) || (!key_gt(b, wb) && wm < m))) {
            b = wb;
            m = wm;
        }
    }
    __syncthreads();
    return m;
}

// First m >= 1 with Theta_m <= Theta_{m-1}, minus one (|pool| if none).
__device__ __noinline__ int sync_scan(SchedSmem& sm, const ScheduleParams& p, int n, int ni, const unsigned long long (&S)[kMaxItems],
                         unsigned long long excl, const float (&sv)[kMaxItems + 1])
{
    const int tid = threadIdx.x;
    if (tid == 0) sm.first_bad = INT32_MAX;
    __syncthreads();
    int bad = INT32_MAX;
    if (tid * ni < n) {
        ThetaKey prev = theta_key(p.R, excl, sv[0], p.status);
#pragma unroll
        for (int it = 0; it < kMaxItems; ++it) {
            const int i = tid * ni + it;
            if (it < ni && i < n) {
                const ThetaKey th = theta_key(p.R, S[it], sv[it + 1], p.status);
                if (!key_gt(th, prev) && bad == INT32_MAX) bad = i + 1;
                prev = th;
            }
        }
    }
    bad = __reduce_min_sync(0xffffffffu, bad);
    if ((tid & 31) == 0 && bad != INT32_MAX) atomicMin(&sm.first_bad, bad);
    __syncthreads();
    const int fb = sm.first_bad;
    __syncthreads();
    return fb == INT32_MAX ? n : fb - 1;
}

// Static confidence threshold: every pool candidate with a_{r,j} >= threshold, no sort and no
// throughput model; keep and the stats as for the other modes.
__device__ void threshold_admit(SchedSmem& sm, const ScheduleParams& p, int n_slots)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t* cnt = sm.hist;
    for (int q = tid; q < p.R; q += kSchedThreads) cnt[q] = 0;
    if (tid == 0) {
        sm.n_pool = 0;
        sm.first_bad = 0;   // admitted count
    }
    __syncthreads();
    int n_pool = 0, n_adm = 0;
    unsigned long long sum = 0;
    for (int s = tid; s < n_slots; s += kSchedThreads) {
        const int q = s / p.G, j = s % p.G;
        int g = p.gamma ? p.gamma[q] : p.G;
        if (g < 0 || g > p.G) {
            raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
            g = g < 0 ? 0 : p.G;
        }
        float a = p.surv[s];
        if (j < g && a > 0.f) {   // the pool, as for the other modes
            if (!(a <= 1.f)) {
                raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                a = 1.f;
            }
            ++n_pool;
            if (a >= p.threshold) {
                ++n_adm;
                sum += fixed48(~__float_as_uint(a));
                atomicMax(&cnt[q], (uint32_t)(j + 1));   // l_r = the largest admitted j
            }
        }
    }
    n_pool = __reduce_add_sync(0xffffffffu, n_pool);
    n_adm = __reduce_add_sync(0xffffffffu, n_adm);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
        sm.wsum[warp] = sum;
        if (n_pool) atomicAdd(&sm.n_pool, n_pool);
        if (n_adm) atomicAdd(&sm.first_bad, n_adm);
    }
    __syncthreads();
    for (int q = tid; q < p.R; q += kSchedThreads) p.keep[q] = (int32_t)cnt[q];
    if (tid == 0) {
        unsigned long long S = 0;
        for (int w = 0; w < kSchedWarps; ++w) S += sm.wsum[w];
        const int m = sm.first_bad;
        p.stats->theta_best = theta_of(p.R, m, S, p.sps);
        p.stats->admitted = m;
        p.stats->capacity = -1;
        p.stats->batch = p.R + m;
        p.stats->pool = sm.n_pool;
    }
}

__global__ void __launch_bounds__(kSchedThreads, 1) schedule_kernel(ScheduleParams p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SchedSmem& sm = *reinterpret_cast<SchedSmem*>(smem_raw);
    const int n_slots = p.R * p.G;
    const int ni = (n_slots + kSchedThreads - 1) / kSchedThreads;   // keys per thread, 1..8
    // The throughput-table entries of this thread's scan positions, SPS(R + m) for
    // m = tid*ni .. tid*ni + ni (index R + m - 1; n_sps >= R (1 + G) covers every m <= R G). The
    // table is an input: it is read before the dependency wait, so the scans never wait on memory.
    float sv[kMaxItems + 1];
#pragma unroll
    for (int u = 0; u <= kMaxItems; ++u) {
        const int m = (int)threadIdx.x * ni + u;
        sv[u] = (u <= ni && m <= n_slots && p.R + m >= 1) ? p.sps[p.R + m - 1] : 0.f;
    }
    pdl_enter();   // the survivals come from the sampler's last commit
    if (p.mode == DSPARK_SCHED_THRESHOLD) {
        threshold_admit(sm, p, n_slots);
        return;
    }

    unsigned long long S[kMaxItems], excl;
    int capacity = -1;
    if (p.mode == DSPARK_SCHED_ASYNC_CAPACITY) {
        const int n_old = load_pool(sm, p, p.surv_capacity, n_slots, ni);
        sort_pool(sm, n_slots, p.G, ni);
        prefix_sums(sm, n_old, ni, S, excl);
        capacity = full_scan(sm, p, n_old, ni, S, sv);
    }
    const int n = load_pool(sm, p, p.surv, n_slots, ni);
    sort_pool(sm, n_slots, p.G, ni);
    prefix_sums(sm, n, ni, S, excl);
    int m_star;
    if (p.mode == DSPARK_SCHED_SYNC)
        m_star = sync_scan(sm, p, n, ni, S, excl, sv);
    else if (p.mode == DSPARK_SCHED_FULL_SCAN)
        m_star = full_scan(sm, p, n, ni, S, sv);
    else
        m_star = min(capacity, n);

    // keep[r] = l_r, the largest admitted position of request r (Algorithm 1 sets l_r = j on
    // each admission); with survivals non-increasing in j it is also the admitted count
    uint32_t* cnt = sm.hist;
    for (int q = threadIdx.x; q < p.R; q += kSchedThreads) cnt[q] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m_star; i += kSchedThreads) {
        const int slot = sm.val[0][sk(i)];
        atomicMax(&cnt[slot / p.G], (uint32_t)(slot % p.G + 1));
    }
    __syncthreads();
    for (int q = threadIdx.x; q < p.R; q += kSchedThreads) p.keep[q] = (int32_t)cnt[q];

    // Theta of the admitted set with the current survivals, from the prefix sums
    const int last = m_star - 1;
    if (m_star == 0 && threadIdx.x == 0) {
        p.stats->theta_best = theta_of(p.R, 0, 0ull, p.sps);
    } else if (last >= 0 && last / ni == (int)threadIdx.x) {
        p.stats->theta_best = theta_of(p.R, m_star, S[last % ni], p.sps);
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
    static bool smem_set = false;
    const size_t smem = sizeof(SchedSmem);
    if (!smem_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = true;
    }
    const cudaError_t e = launch_pdl(schedule_kernel, 1, kSchedThreads, smem, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
