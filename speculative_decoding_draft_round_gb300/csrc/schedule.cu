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
// warps. A positive float's bit pattern orders like an unsigned integer, so keys
// are the complemented bits. When every request's keys are already in order (the
// sampler's survivals are running products of confidences) the R runs are merged
// pairwise on merge paths; any other input takes a stable LSD radix sort (four
// 8-bit digits, warp-aggregated ranks via __match_any_sync, digit offsets from one
// block-wide scan of the [digit][warp] counts); stability in slot order gives the
// (r, j) tie-break for free. Sync mode with a table that forces the first decrease
// within 64 admissions (a staircase edge) takes only the top 64 keys, selected
// by bitonic networks in registers, instead of sorting the whole pool.
// Prefix sums are exact 64-bit fixed-point sums (a in units
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

constexpr int kTopMax = 64;      // sync mode: the latest forced first decrease that takes the top-keys path

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
    // sync mode, top-keys path
    unsigned long long tlist[kSchedWarps][kTopMax];   // per-warp top lists, (key << 32) | slot ascending
    float tsps[kTopMax + 1];                           // SPS(R + m), m = 0 .. kTopMax
    unsigned long long s_star;                         // fixed-point sum of the admitted a's
    int m_bound;   // first m at which the throughput table forces Theta down
    // the table entries SPS(R + m) of each thread's scan positions m = tid*ni + u, read before the
    // dependency wait; kept here, not in registers, so that no out-of-line call has to save them
    float sv[kMaxItems + 1][kSchedThreads];
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
// of a thread is issued before any is used. (Scalar arguments: a reference to the kernel's
// parameter block would put a copy of it in local memory.)
__device__ __noinline__ int load_pool(SchedSmem& sm, const int32_t* gamma, int G, int* status, const float* src,
                                      int n_slots, int ni)
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
        g[it] = in ? (gamma ? gamma[s / G] : G) : 0;
    }
    int cnt = 0;
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        if (it >= ni) break;
        const int s = striped(warp, it, lane, ni);
        uint32_t key = 0xFFFFFFFFu;
        if (s < n_slots) {
            int gg = g[it];
            if (gg < 0 || gg > G) {
                raise_status(status, DSPARK_ERR_DEVICE_INPUT);
                gg = gg < 0 ? 0 : G;
            }
            float av = a[it];
            if (s % G < gg && av > 0.f) {   // NaN and non-positive survivals are not in the pool
                if (!(av <= 1.f)) {
                    raise_status(status, DSPARK_ERR_DEVICE_INPUT);
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
__device__ __forceinline__ void scan_hist(SchedSmem& sm)
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

// One stable counting pass on 8 bits of the key, buffer `in` -> 1 - in. A thread's keys and, per
// key, its slot (low 16 bits) with its rank among the equal digits of its warp (high 16 bits, below
// 256) stay in registers across the histogram scan; the digit is formed again for the scatter.
__device__ __noinline__ void radix_pass(SchedSmem& sm, int in, int shift, int ni)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    reinterpret_cast<uint4*>(sm.hist)[2 * tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(sm.hist)[2 * tid + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    uint32_t key[kMaxItems], vr[kMaxItems];
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        if (it >= ni) break;
        const int idx = striped(warp, it, lane, ni);
        key[it] = sm.key[in][sk(idx)];
        vr[it] = sm.val[in][sk(idx)];
    }
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        if (it >= ni) break;
        const uint32_t dig = (key[it] >> shift) & (kDigits - 1);
        uint32_t* h = sm.hist + dig * kSchedWarps + warp;
        const uint32_t peers = __match_any_sync(0xffffffffu, dig);
        const uint32_t base = *h;
        __syncwarp();
        if (lane == __ffs(peers) - 1) *h = base + __popc(peers);
        __syncwarp();
        vr[it] |= (base + __popc(peers & lanemask_lt())) << 16;
    }
    __syncthreads();
    scan_hist(sm);
    __syncthreads();
    const int out = 1 - in;
#pragma unroll
    for (int it = 0; it < kMaxItems; ++it) {
        if (it >= ni) break;
        const uint32_t dig = (key[it] >> shift) & (kDigits - 1);
        const uint32_t pos = sm.hist[dig * kSchedWarps + warp] + (vr[it] >> 16);
        sm.key[out][sk(pos)] = key[it];
        sm.val[out][sk(pos)] = (uint16_t)(vr[it] & 0xFFFFu);
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

// Are every request's G keys in order? The sampler's survivals are running products of
// confidences below one, so they never increase along a request.
__device__ __noinline__ bool runs_sorted(SchedSmem& sm, int n, int G)
{
    bool unsorted = false;
    for (int s = threadIdx.x; s < n; s += kSchedThreads)
        if (s % G != G - 1 && s + 1 < n && sm.key[0][sk(s + 1)] < sm.key[0][sk(s)]) unsorted = true;
    return !__syncthreads_or(unsorted);
}

// Sort key[0]/val[0] ascending (a descending, then slot); result in buffer 0. When the R runs of
// G keys are in order they are merged pairwise (log2 R levels); any other input takes the
// stable LSD radix sort.
__device__ __noinline__ void sort_pool(SchedSmem& sm, int n, int G, int ni)
{
    if (!runs_sorted(sm, n, G)) {
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
__device__ __forceinline__ void prefix_sums(SchedSmem& sm, int n, int ni, unsigned long long (&S)[kMaxItems], unsigned long long& excl)
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
__device__ __forceinline__ int full_scan(SchedSmem& sm, const ScheduleParams& p, int n, int ni, const unsigned long long (&S)[kMaxItems])
{
    const float* sv = &sm.sv[0][threadIdx.x];   // sv[u * kSchedThreads]: SPS at position tid*ni + u
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
            const ThetaKey th = theta_key(p.R, S[it], sv[(it + 1) * kSchedThreads], p.status);
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
__device__ __forceinline__ int sync_scan(SchedSmem& sm, const ScheduleParams& p, int n, int ni, const unsigned long long (&S)[kMaxItems],
                         unsigned long long excl)
{
    const float* sv = &sm.sv[0][threadIdx.x];   // sv[u * kSchedThreads]: SPS at position tid*ni + u
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
                const ThetaKey th = theta_key(p.R, S[it], sv[(it + 1) * kSchedThreads], p.status);
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

// ---- sync mode, top-keys path
// Admitting an m-th key adds a <= 1 to tau >= R, so Theta_m <= Theta_{m-1} whatever the keys are
// once SPS(R + m - 1) * R >= SPS(R + m) * (R + 1). With M the first such m (the table is an input,
// so M is known before the dependency wait) the first decrease comes at m <= M, and only the top M
// keys decide m*. For M <= kTopMax the kernel takes the kTopMax smallest (key, slot) pairs with
// bitonic networks in registers -- no sort of the whole pool -- and scans Theta over them in one
// warp. A lane holds elements `lane` and `lane + 32` of a 64-element list in x0 and x1.

__device__ __forceinline__ unsigned long long packed_key(const SchedSmem& sm, int i, int n)
{
    return i < n ? ((unsigned long long)sm.key[0][sk(i)] << 32) | sm.val[0][sk(i)] : ~0ull;
}

// compare-exchange of element i with element i ^ j (j < 32, another lane), in the direction of
// i's block of size k (ascending when i & k == 0)
__device__ __forceinline__ unsigned long long cmp_x(unsigned long long x, int i, int j, int k)
{
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, x, j);
    return (((i & k) == 0) == ((i & j) == 0)) ? min(x, o) : max(x, o);
}

// sort 64 values ascending
__device__ __forceinline__ void bitonic_sort64(unsigned long long& x0, unsigned long long& x1, int lane)
{
#pragma unroll
    for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j == 32) {   // k == 64: the partner is this lane's other element, ascending
                const unsigned long long lo = min(x0, x1), hi = max(x0, x1);
                x0 = lo;
                x1 = hi;
            } else {
                x0 = cmp_x(x0, lane, j, k);
                x1 = cmp_x(x1, lane + 32, j, k);
            }
        }
    }
}

// (x0, x1) = the 64 smallest of two ascending lists (x0, x1) and (y0, y1), ascending:
// min(A_i, B_{63-i}) is a bitonic sequence that holds them, then a bitonic merge sorts it
__device__ __forceinline__ void merge_top64(unsigned long long& x0, unsigned long long& x1, unsigned long long y0,
                                            unsigned long long y1, int lane)
{
    x0 = min(x0, __shfl_sync(0xffffffffu, y1, 31 - lane));   // B_{63 - lane}
    x1 = min(x1, __shfl_sync(0xffffffffu, y0, 31 - lane));   // B_{31 - lane}
    const unsigned long long lo = min(x0, x1), hi = max(x0, x1);
    x0 = lo;
    x1 = hi;
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        x0 = cmp_x(x0, lane, j, 64);
        x1 = cmp_x(x1, lane + 32, j, 64);
    }
}

// m* of the sync scan from the top keys of buffer 0 (n_slots positions, n of them in the pool):
// every warp sorts 64-position chunks and folds them into its own top list, the 32 lists are
// merged pairwise in five levels, and warp 0 scans Theta over the first min(kTopMax, n). Returns
// m* to every thread, with the admitted keys' slots at val[0] positions 0 .. m*-1 and their
// fixed-point sum in s_star; -1 (buffers untouched) when those keys showed no decrease and the pool
// holds more, so that the full sort decides.
__device__ __noinline__ int top_scan(SchedSmem& sm, int R, int* status, int n_slots, int n)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned long long x0 = ~0ull, x1 = ~0ull;
    for (int c = warp * 64; c < n_slots; c += kSchedWarps * 64) {
        unsigned long long y0 = packed_key(sm, c + lane, n_slots), y1 = packed_key(sm, c + 32 + lane, n_slots);
        bitonic_sort64(y0, y1, lane);
        merge_top64(x0, x1, y0, y1, lane);
    }
    sm.tlist[warp][lane] = x0;
    sm.tlist[warp][lane + 32] = x1;
    __syncthreads();
    for (int w = kSchedWarps / 2; w >= 1; w >>= 1) {
        if (warp < w) {
            merge_top64(x0, x1, sm.tlist[warp + w][lane], sm.tlist[warp + w][lane + 32], lane);
            sm.tlist[warp][lane] = x0;
            sm.tlist[warp][lane + 32] = x1;
        }
        __syncthreads();
    }
    if (warp == 0) {
        const int nt = min(kTopMax, n);   // pool keys sort before every other position
        const unsigned long long f0 = lane < nt ? fixed48((uint32_t)(x0 >> 32)) : 0ull;
        const unsigned long long f1 = lane + 32 < nt ? fixed48((uint32_t)(x1 >> 32)) : 0ull;
        unsigned long long s0 = f0, s1 = f1;   // inclusive prefix sums over positions lane, lane + 32
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y0 = __shfl_up_sync(0xffffffffu, s0, o), y1 = __shfl_up_sync(0xffffffffu, s1, o);
            if (lane >= o) {
                s0 += y0;
                s1 += y1;
            }
        }
        s1 += __shfl_sync(0xffffffffu, s0, 31);
        const ThetaKey big{INT32_MAX, ~0ull};
        const ThetaKey t0 = lane < nt ? theta_key(R, s0, sm.tsps[lane + 1], status) : big;
        const ThetaKey t1 = lane + 32 < nt ? theta_key(R, s1, sm.tsps[lane + 33], status) : big;
        ThetaKey p0{__shfl_up_sync(0xffffffffu, t0.e, 1), __shfl_up_sync(0xffffffffu, t0.m, 1)};
        ThetaKey p1{__shfl_up_sync(0xffffffffu, t1.e, 1), __shfl_up_sync(0xffffffffu, t1.m, 1)};
        const ThetaKey t0_last{__shfl_sync(0xffffffffu, t0.e, 31), __shfl_sync(0xffffffffu, t0.m, 31)};
        if (lane == 0) {
            p0 = theta_key(R, 0ull, sm.tsps[0], status);
            p1 = t0_last;
        }
        const uint32_t b0 = __ballot_sync(0xffffffffu, lane < nt && !key_gt(t0, p0));
        const uint32_t b1 = __ballot_sync(0xffffffffu, lane + 32 < nt && !key_gt(t1, p1));
        // first position whose key does not raise Theta: m* keys come before it
        int m_star = b0 ? __ffs(b0) - 1 : b1 ? 32 + __ffs(b1) - 1 : (nt == n ? n : -1);
        unsigned long long s_star = 0ull;
        if (m_star >= 0) {
            // exclusive prefix at position m* (the sum of all nt keys when m* = nt)
            const unsigned long long e0 = __shfl_sync(0xffffffffu, s0 - f0, m_star & 31);
            const unsigned long long e1 = __shfl_sync(0xffffffffu, s1 - f1, m_star & 31);
            const unsigned long long tot = __shfl_sync(0xffffffffu, s1, 31);
            s_star = m_star == nt ? (nt > 32 ? tot : __shfl_sync(0xffffffffu, s0, 31)) : (m_star < 32 ? e0 : e1);
            if (lane < m_star) sm.val[0][sk(lane)] = (uint16_t)(x0 & 0xFFFFu);
            if (lane + 32 < m_star) sm.val[0][sk(lane + 32)] = (uint16_t)(x1 & 0xFFFFu);
        }
        if (lane == 0) {
            sm.first_bad = m_star;
            sm.s_star = s_star;
        }
    }
    __syncthreads();
    const int m = sm.first_bad;
    __syncthreads();
    return m;
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

// keep[r] = l_r from the admitted keys at sorted positions 0 .. m_star - 1 (val[0] holds their
// slots); no global write when keep is null (the code warm-up). Algorithm 1 sets l_r = j at each
// admission in sorted order, so in the sync and full-scan modes (last_wins) l_r is the position of
// r's last admitted key, packed behind its sorted index so that the largest index wins; the
// asynchronous mode fills its capacity with r's largest admitted position. With survivals
// non-increasing in j both are r's admitted count.
__device__ __noinline__ void write_keep(SchedSmem& sm, int m_star, int R, int G, bool last_wins, int32_t* keep)
{
    uint32_t* cnt = sm.hist;
    for (int q = threadIdx.x; q < R; q += kSchedThreads) cnt[q] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m_star; i += kSchedThreads) {
        const int slot = sm.val[0][sk(i)];
        const uint32_t j1 = (uint32_t)(slot % G + 1);   // <= 8192 < 2^14
        atomicMax(&cnt[slot / G], last_wins ? ((uint32_t)i << 14) | j1 : j1);
    }
    __syncthreads();
    if (keep)
        for (int q = threadIdx.x; q < R; q += kSchedThreads) keep[q] = (int32_t)(cnt[q] & 0x3FFFu);
}

// Code warm-up of the out-of-line phases. The draft steps before this kernel stream more than L2
// holds, so on its first run each phase's code comes from DRAM a few cache lines at a time, which
// measured slower than the phase's work (24 us against 11 us for the same sync-mode round run a
// second time). CTAs 1 .. kWarmCtas run one phase each on their own shared memory while CTA 0 waits
// for the sampler, and CTA 0 then fetches that code from L2. The warm-up reads only inputs (the
// throughput table), writes no global memory and raises no status.
constexpr int kWarmCtas = kScheduleCtas - 1;

__device__ void warm_phase(SchedSmem& sm, const ScheduleParams& p, int n_slots, int ni)
{
    if (blockIdx.x == 1) {
        // n_sps >= R (1 + G) > n_slots entries (checked by the host): keys from the table
        const int n = load_pool(sm, nullptr, p.G, nullptr, p.sps, n_slots, ni);
        write_keep(sm, n, p.R, p.G, true, nullptr);
        return;
    }
    for (int i = threadIdx.x; i <= kTopMax; i += kSchedThreads) sm.tsps[i] = 1.f;
    for (int i = threadIdx.x; i < n_slots; i += kSchedThreads) {   // ascending runs: the merge path
        sm.key[0][sk(i)] = (uint32_t)i;
        sm.val[0][sk(i)] = (uint16_t)i;
    }
    __syncthreads();
    if (blockIdx.x == 2)
        top_scan(sm, p.R, nullptr, n_slots, n_slots);
    else
        sort_pool(sm, n_slots, p.G, ni);
}

__global__ void __launch_bounds__(kSchedThreads, 1) schedule_kernel(ScheduleParams p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SchedSmem& sm = *reinterpret_cast<SchedSmem*>(smem_raw);
    const int n_slots = p.R * p.G;
    const int ni = (n_slots + kSchedThreads - 1) / kSchedThreads;   // keys per thread, 1..8
    if (blockIdx.x > 0) {
        pdl_trigger();
        if (p.mode != DSPARK_SCHED_THRESHOLD) warm_phase(sm, p, n_slots, ni);
        return;
    }
    // The throughput-table entries of this thread's scan positions, SPS(R + m) for
    // m = tid*ni .. tid*ni + ni (index R + m - 1; n_sps >= R (1 + G) covers every m <= R G). The
    // table is an input: it is read before the dependency wait, so the scans never wait on memory.
#pragma unroll
    for (int u = 0; u <= kMaxItems; ++u) {
        const int m = (int)threadIdx.x * ni + u;
        sm.sv[u][threadIdx.x] = (u <= ni && m <= n_slots && p.R + m >= 1) ? p.sps[p.R + m - 1] : 0.f;
    }
    // sync mode: the table's first forced decrease and its first entries (see top_scan); the table
    // is an input like the entries above
    const bool sync_mode = p.mode == DSPARK_SCHED_SYNC;
    if (sync_mode) {
        if (threadIdx.x == 0) sm.m_bound = INT32_MAX;
        __syncthreads();
        const int t = threadIdx.x, m = t + 1;
        if (t <= kTopMax && t <= n_slots) sm.tsps[t] = p.sps[p.R + t - 1];
        if (m <= kTopMax && m <= n_slots) {
            const double lo = p.sps[p.R + m - 2], hi = p.sps[p.R + m - 1];   // exact products in double
            if (hi > 0.0 && lo * p.R >= hi * (p.R + 1.0)) atomicMin(&sm.m_bound, m);
        }
    }
    pdl_enter();   // the survivals come from the sampler's last commit
    if (p.mode == DSPARK_SCHED_THRESHOLD) {
        threshold_admit(sm, p, n_slots);
        return;
    }

    unsigned long long S[kMaxItems], excl;
    int capacity = -1;
    if (p.mode == DSPARK_SCHED_ASYNC_CAPACITY) {
        const int n_old = load_pool(sm, p.gamma, p.G, p.status, p.surv_capacity, n_slots, ni);
        sort_pool(sm, n_slots, p.G, ni);
        prefix_sums(sm, n_old, ni, S, excl);
        capacity = full_scan(sm, p, n_old, ni, S);
    }
    const int n = load_pool(sm, p.gamma, p.G, p.status, p.surv, n_slots, ni);
    int m_star = -1;
    bool top = false;
    if (sync_mode && sm.m_bound <= kTopMax) {
        // the whole scan reads every table entry up to |pool|: flag a bad one the same way
#pragma unroll
        for (int u = 0; u <= kMaxItems; ++u) {
            const int m = (int)threadIdx.x * ni + u;
            const float v = sm.sv[u][threadIdx.x];
            if (u <= ni && m <= n && !(v > 0.f && v != INFINITY)) raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
        }
        m_star = top_scan(sm, p.R, p.status, n_slots, n);
        top = m_star >= 0;
    }
    if (m_star < 0) {
        sort_pool(sm, n_slots, p.G, ni);
        prefix_sums(sm, n, ni, S, excl);
        if (p.mode == DSPARK_SCHED_SYNC)
            m_star = sync_scan(sm, p, n, ni, S, excl);
        else if (p.mode == DSPARK_SCHED_FULL_SCAN)
            m_star = full_scan(sm, p, n, ni, S);
        else
            m_star = min(capacity, n);
    }

    write_keep(sm, m_star, p.R, p.G, p.mode == DSPARK_SCHED_SYNC || p.mode == DSPARK_SCHED_FULL_SCAN, p.keep);

    // Theta of the admitted set with the current survivals, from the prefix sums
    const int last = m_star - 1;
    if (top) {
        if (threadIdx.x == 0) p.stats->theta_best = theta_of(p.R, m_star, sm.s_star, p.sps);
    } else if (m_star == 0 && threadIdx.x == 0) {
        p.stats->theta_best = theta_of(p.R, 0, 0ull, p.sps);
    } else if (last >= 0 && last / ni == (int)threadIdx.x) {
        unsigned long long s_last = 0ull;   // S[last % ni], selected without a dynamic index (S stays in registers)
#pragma unroll
        for (int it = 0; it < kMaxItems; ++it)
            if (it == last % ni) s_last = S[it];
        p.stats->theta_best = theta_of(p.R, m_star, s_last, p.sps);
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
    const cudaError_t e = launch_pdl(schedule_kernel, 1 + kWarmCtas, kSchedThreads, smem, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
