// draft_loop.cu -- the whole serial draft loop of the Markov head in one persistent launch, with
// the vocabulary slice of W each SM owns held on chip between the steps.
//
// Method ("DSpark", zhongzhuzhou.org notes eq. 4-5 and 7; caijizhuo.github.io section 4
// dspark_cycle step 3): for k = 0 .. gamma_max - 1
//   B_k = W_1[x_{k-1}] W_2,  l_k = (U_k + B_k) / T,  x_k ~ softmax(l_k)  (two-level Gumbel-max),
//   c_k = sigmoid((w_h . h_k + w_e . W_1[x] + b) / t_k),  a_k = a_{k-1} c_k.
// The per-step kernels of sample_tc.cu / sample.cu stream all of W (r x V) from DRAM at every
// step: this GPU's L2 keeps none of it between steps. Here one cooperative CTA per SM owns a
// contiguous range of 128-wide vocabulary blocks for the whole call and keeps the first blocks of
// its range on chip: W^T tiles [128 vocabulary rows x r] in tensor memory (the MMA's A operand,
// up to 3 tiles) and one more in shared memory; the rest are streamed each step.
//
// One step, on every CTA (roles by warp):
//   warp 0      TMA producer: U tiles [64 requests x 128 columns] of the step, streamed W chunks
//   warp 1      TMEM owner and MMA issuer: D[v][q] = sum_i W[i][v] E[x_{k-1}(q)][i] per block and
//               request half (M = 128 vocabulary rows, N = 64 requests, K = 16 per instruction)
//   warp 2      grid barriers and the copy of the next step's conditioning rows (E tile)
//   warps 4-11  epilogue: lane quarter (warp % 4) = 32 vocabulary rows, column group = 32 requests.
//               y = (U + D) log2(e) / T; per (request, block) the block maximum and sum of
//               2^(y - max) by reduce-scatter over the lanes and a combine across the quarters;
//               the block key of the two-level draw; the CTA's running (max, sum) of each row;
//               the logits of each row's leading block are saved to a per-CTA slot.
//   then, after a grid barrier, the commit: per request (one warp), the winning block and CTA
//   from the packed 64-bit key, the log-normaliser from the CTAs' partials, the element-level
//   Gumbel-max over the saved logits, the confidence head and survival product, and the next
//   step's conditioning row W_1[x_k] in 8 copies; a second grid barrier, then the E tile.
// Every wait is bounded by the global timer. A wait that runs out records DSPARK_ERR_TIMEOUT and
// sets an abort flag every CTA polls; each role then stops issuing, lets its own copies and MMAs
// land, and the CTA frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace dspark {
namespace {

constexpr int LP_THREADS = 384;                 // 12 warps
constexpr int LP_EPI_WARP0 = 4;                 // warps 4-11: epilogue and commit
constexpr int LP_EPI_WARPS = 8;
constexpr int NHALF = 64;                       // requests per MMA (N)
constexpr int RMAX = 128;                       // requests handled by this path
constexpr int KR = 256;                         // Markov rank r
constexpr int KCH = 64;                         // K per chunk (128 bytes of bf16)
constexpr int NKC = KR / KCH;                   // 4 chunks
constexpr int TM_TILES = 3;                     // W tiles held in tensor memory
constexpr uint32_t TILE_COLS = KR / 2;          // TMEM columns of one W^T tile (bf16 pairs)
constexpr uint32_t ACC_COL = TM_TILES * TILE_COLS;   // 384: two accumulators of 64 columns
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t CHUNK_BYTES = KCH * 128 * 2;      // 16 KB: [64 K rows x 128 vocabulary] as 2 boxes
constexpr uint32_t BOX_BYTES = 8192;                 // [64 rows x 64 elements] bf16
constexpr int WR_ST = 2;                        // streamed W chunk stages
constexpr int U_ST = 3;                         // U half-tile stages [64 requests x 128 columns]
// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_E = 0;                                   // E tile: 4 chunks [128 rows x 64 K]
constexpr uint32_t OFF_S = OFF_E + NKC * RMAX * 128;           // 64 KB: the W tile kept in shared memory
constexpr uint32_t OFF_WR = OFF_S + NKC * CHUNK_BYTES;         // streamed W chunks
constexpr uint32_t OFF_U = OFF_WR + WR_ST * CHUNK_BYTES;       // U stages
constexpr uint32_t OFF_RED = OFF_U + U_ST * (NHALF * 128 * 2); // [2 cg][2 kinds][4 quarters][32] floats
constexpr uint32_t OFF_SCALE = OFF_RED + 2 * 2 * 4 * 32 * 4;   // [128] floats: log2(e) / T per request
constexpr uint32_t OFF_MISC = OFF_SCALE + RMAX * 4;            // lead masks, flags, TMEM base
constexpr uint32_t OFF_BAR = OFF_MISC + 64;
constexpr int N_BARS = 2 * WR_ST + 2 * U_ST + 4 + 5;
constexpr uint32_t SMEM_USED = OFF_BAR + N_BARS * 8;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;               // alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(OFF_S % 1024 == 0 && OFF_WR % 1024 == 0 && OFF_U % 1024 == 0, "swizzle atoms on 1 KB");
// the initial batch of TMEM-resident chunks is staged over E, S, W-ring and U regions
static_assert(TM_TILES * NKC * CHUNK_BYTES <= OFF_RED, "initial staging fits");

constexpr unsigned long long DRAIN_NS = 4000000000ull;

// instruction descriptors, kind::f16, D fp32, A = B = bf16, B K-major (request rows), N = 64,
// M = 128: A from tensor memory, or A from shared memory MN-major (vocabulary contiguous)
constexpr uint32_t IDESC_TA = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NHALF >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t IDESC_SA = IDESC_TA | (1u << 15);

struct LoopParams {
    DraftStep d;
    float* slots;            // [P][128][128] fp32: per CTA and request, the leading block's logits y
    float* hdot;             // [R][G] w_h . h_k
    unsigned int* gbar;      // grid barrier counter (zero at launch)
    int* gabort;             // grid-wide abort flag (zero at launch)
    int P;                   // CTAs
};

// ------------------------------------------------------------------ small PTX helpers

__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(IDESC_TA), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC_SA), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint16_t lds_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void bar_sync(int id, int count)
{
    asm volatile("barrier.cta.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}


// Reduce 32 values over the 32 lanes of the warp: value i of every lane belongs to column i; on
// return lane l holds op over all lanes of column l. Fixed pairing order: deterministic.
template <bool MAX>
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int j = 0; j < s; ++j) {
            const float send = up ? v[j] : v[j + s];
            const float keep = up ? v[j + s] : v[j];
            const float recv = __shfl_xor_sync(0xffffffffu, send, s);
            v[j] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
    }
    return v[0];
}

struct Lse2 {
    float m, s;   // sum of 2^x as s * 2^m
};

__device__ __forceinline__ Lse2 lse2_merge(Lse2 a, Lse2 b)
{
    if (!(b.s > 0.f)) return a;
    if (!(a.s > 0.f)) return b;
    return a.m >= b.m ? Lse2{a.m, a.s + b.s * ex2(b.m - a.m)} : Lse2{b.m, b.s + a.s * ex2(a.m - b.m)};
}

struct LoopCtl {
    volatile int* abort;   // this CTA gave up (shared memory)
    int* gabort;           // some CTA gave up (global)
    int* status;
    unsigned long long limit;
};

// Bounded wait on a shared-memory barrier phase; false when the CTA aborted or the wait ran out.
__device__ __noinline__ bool lp_wait(uint32_t bar, uint32_t parity, LoopCtl c)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort) return false;
        if (globaltimer() - t0 > c.limit) {
            *c.abort = 1;
            atomicExch(c.gabort, 1);
            raise_status(c.status, DSPARK_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __noinline__ void lp_drain(uint32_t bar, uint32_t parity)
{
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < DRAIN_NS) {
    }
}

// Grid barrier number n (1, 2, ...) over P CTAs, by one thread per CTA after the CTA's own
// threads have synchronised: its writes, ordered before by that synchronisation, are released
// with a fence; the others' are acquired after the count reaches n * P. Bounded; false (and the
// abort flags set) when it runs out or another CTA gave up.
__device__ __noinline__ bool grid_sync(unsigned int* gbar, unsigned int target, LoopCtl c)
{
    __threadfence();
    atomicAdd(gbar, 1u);
    const unsigned long long t0 = globaltimer();
    while (ld_acquire_u32(gbar) < target) {
        if (ld_relaxed_s32(c.gabort)) {
            *c.abort = 1;
            return false;
        }
        if (globaltimer() - t0 > c.limit) {
            *c.abort = 1;
            atomicExch(c.gabort, 1);
            raise_status(c.status, DSPARK_ERR_TIMEOUT);
            return false;
        }
    }
    __threadfence();
    return true;
}

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(LP_THREADS, 1)
    draft_loop_kernel(const LoopParams L, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmE)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const DraftStep& p = L.d;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x, P = L.P;
    const int R = p.R, G = p.G, V = p.V, nblk = p.nblk;
    const int NH = (R + NHALF - 1) / NHALF;
    // this CTA's vocabulary blocks [b0, b0 + nt): the first n_tm in tensor memory, then n_sm in
    // shared memory, the rest streamed every step
    const int b0 = (int)((long long)cta * nblk / P), b1 = (int)((long long)(cta + 1) * nblk / P);
    const int nt = b1 - b0;
    const int n_tm = nt < TM_TILES ? nt : TM_TILES;
    const int n_sm = nt > n_tm ? 1 : 0;

    float* s_red = reinterpret_cast<float*>(smem + OFF_RED);
    float* s_scale = reinterpret_cast<float*>(smem + OFF_SCALE);
    uint32_t* s_lead = reinterpret_cast<uint32_t*>(smem + OFF_MISC);        // [2] lead masks per column group
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 16);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 20);
    // written only by warp 2 lane 0 between two named barriers: a decision all its warps share
    volatile int* s_stop = reinterpret_cast<volatile int*>(smem + OFF_MISC + 24);
    const uint32_t bar0 = sbase + OFF_BAR;
    auto w_full = [&](int i) { return bar0 + 8u * i; };
    auto w_empty = [&](int i) { return bar0 + 8u * (WR_ST + i); };
    auto u_full = [&](int i) { return bar0 + 8u * (2 * WR_ST + i); };
    auto u_empty = [&](int i) { return bar0 + 8u * (2 * WR_ST + U_ST + i); };
    auto acc_full = [&](int h) { return bar0 + 8u * (2 * WR_ST + 2 * U_ST + h); };
    auto acc_empty = [&](int h) { return bar0 + 8u * (2 * WR_ST + 2 * U_ST + 2 + h); };
    const uint32_t e_full = bar0 + 8u * (2 * WR_ST + 2 * U_ST + 4);
    const uint32_t e_empty = e_full + 8u;
    const uint32_t s_full = e_full + 16u;
    const uint32_t init_full = e_full + 24u;
    const uint32_t mma_done = e_full + 32u;
    const LoopCtl ctl{s_abort, L.gabort, p.status, p.wait_ns};

    if (tid == 0) {
        for (int i = 0; i < WR_ST; ++i) {
            mbar_init(w_full(i), 1);
            mbar_init(w_empty(i), 1);
        }
        for (int i = 0; i < U_ST; ++i) {
            mbar_init(u_full(i), 1);
            mbar_init(u_empty(i), LP_EPI_WARPS);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(acc_full(h), 1);
            mbar_init(acc_empty(h), LP_EPI_WARPS);
        }
        mbar_init(e_full, 1);
        mbar_init(e_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(init_full, 1);
        mbar_init(mma_done, 1);
        *s_abort = 0;
        *s_stop = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (tid < RMAX) {
        float sc = kLog2e;   // padding rows: a finite scale
        if (tid < R) {
            const float T = p.temperature[tid];
            sc = T == 0.f ? kLog2e : kLog2e / T;
        }
        s_scale[tid] = sc;
    }
    if (warp == 1) tc5::alloc(s_tmem, TMEM_COLS);
    tc5::fence_before();
    __syncthreads();
    tc5::fence_after();
    const uint32_t tmem = *s_tmem;

    // ---------------- set-up 1: the tensor-memory tiles of W^T, staged through shared memory
    if (tid == 0 && n_tm > 0) {
        mbar_expect_tx(init_full, (uint32_t)(n_tm * NKC) * CHUNK_BYTES);
        const uint64_t pol = l2_policy_evict_first();
        for (int t = 0; t < n_tm; ++t)
            for (int kc = 0; kc < NKC; ++kc) {
                const uint32_t dst = sbase + (uint32_t)(t * NKC + kc) * CHUNK_BYTES;
                tma_load_2d(dst, &tmW, (b0 + t) * 128, kc * KCH, init_full, pol);
                tma_load_2d(dst + BOX_BYTES, &tmW, (b0 + t) * 128 + 64, kc * KCH, init_full, pol);
            }
    }
    // w_h . h_k of every position (inputs only), spread over all warps of the grid
    {
        const int gw = cta * (LP_THREADS / 32) + warp, nw = P * (LP_THREADS / 32);
        const __nv_bfloat16* H = static_cast<const __nv_bfloat16*>(p.h);
        const bool vec = p.d % 8 == 0 && (reinterpret_cast<uintptr_t>(p.h) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(p.w_h) & 15u) == 0;
        for (int pi = gw; pi < R * G; pi += nw) {
            const __nv_bfloat16* hr = H + (size_t)pi * p.d;
            float acc = 0.f;
            if (vec) {
                for (int c = lane * 8; c < p.d; c += 256) {
                    float x[8], w[8];
                    load8<__nv_bfloat16>(hr + c, x);
                    load8<float>(p.w_h + c, w);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc = fmaf(w[e], x[e], acc);
                }
            } else {
                for (int c = lane; c < p.d; c += 32) acc = fmaf(p.w_h[c], __bfloat162float(hr[c]), acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) L.hdot[pi] = acc;
        }
    }
    // the tiles' columns into TMEM: warp 4 + j holds vocabulary rows 32j .. 32j + 31 (its lane
    // quarter); K pair (2c, 2c + 1) in column c of the tile
    if (warp >= LP_EPI_WARP0 && warp < LP_EPI_WARP0 + 4 && n_tm > 0) {
        const bool ok = __all_sync(0xffffffffu, lp_wait(init_full, 0u, ctl));
        const int qw = warp & 3, vl = 32 * qw + lane;
        const uint32_t box = (uint32_t)(vl >> 6) * BOX_BYTES, vv = (uint32_t)(vl & 63);
        if (ok) {
            for (int t = 0; t < n_tm; ++t)
                for (int kc = 0; kc < NKC; ++kc) {
                    const uint32_t src = sbase + (uint32_t)(t * NKC + kc) * CHUNK_BYTES + box;
                    uint32_t a[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const uint32_t r0 = 2 * c, r1 = 2 * c + 1;
                        const uint16_t lo = lds_u16(src + r0 * 128 + ((((vv >> 3) ^ (r0 & 7)) << 4) | ((vv & 7) << 1)));
                        const uint16_t hi = lds_u16(src + r1 * 128 + ((((vv >> 3) ^ (r1 & 7)) << 4) | ((vv & 7) << 1)));
                        a[c] = (uint32_t)lo | ((uint32_t)hi << 16);
                    }
                    tmem_st32(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(t * TILE_COLS + kc * 32), a);
                }
        }
        tc5::fence_before();
    } else if (tid == 0 && n_tm > 0) {
        // thread 0 is not among the converting warps: nothing to do until the staging is consumed
    }
    __syncthreads();
    tc5::fence_after();
    if (tid == 0 && n_tm > 0 && *s_abort) lp_drain(init_full, 0u);   // copies land before the region is reused
    // the shared-memory tile (MN-major, 128-byte swizzle: chunk kc at OFF_S + kc * 16 KB)
    if (tid == 0 && n_sm && !*s_abort) {
        mbar_expect_tx(s_full, NKC * CHUNK_BYTES);
        const uint64_t pol = l2_policy_evict_first();
        for (int kc = 0; kc < NKC; ++kc) {
            const uint32_t dst = sbase + OFF_S + (uint32_t)kc * CHUNK_BYTES;
            tma_load_2d(dst, &tmW, (b0 + n_tm) * 128, kc * KCH, s_full, pol);
            tma_load_2d(dst + BOX_BYTES, &tmW, (b0 + n_tm) * 128 + 64, kc * KCH, s_full, pol);
        }
    }

    // ---------------- set-up 2 (the commit warps): conditioning rows of step 0 and cleared pick slots
    const __nv_bfloat16* E = static_cast<const __nv_bfloat16*>(p.E);
    __nv_bfloat16* an = static_cast<__nv_bfloat16*>(p.a_next);
    const size_t rep_stride = (size_t)R * KR;
    if (warp >= LP_EPI_WARP0) {
        const int ew = warp - LP_EPI_WARP0;
        for (int q = cta + P * ew; q < R; q += P * LP_EPI_WARPS) {
            for (int k = lane; k < G; k += 32) p.pick[(size_t)k * R + q] = 0ull;
            const int x0 = checked_index(p.anchor[q], V, p.status);
            uint4 row = make_uint4(0, 0, 0, 0);
            if (p.bias_first) row = *reinterpret_cast<const uint4*>(E + (size_t)x0 * KR + lane * 8);
            for (int rp = 0; rp < kAReplicas; ++rp)
                *reinterpret_cast<uint4*>(an + rp * rep_stride + (size_t)q * KR + lane * 8) = row;
        }
    }
    unsigned int n_grid = 0;   // grid barriers entered (warp 2 lane 0)
    int e_loads = 0;           // E tile copies issued (warp 2 lane 0)
    // warp 2 (all lanes take part in the named barriers; lane 0 does the grid work)
    const int BAR_STEP = 3, BAR_STEP_N = 32 * (1 + LP_EPI_WARPS);
    if (warp == 2 || warp >= LP_EPI_WARP0) {
        bar_sync(BAR_STEP, BAR_STEP_N);
        if (warp == 2 && lane == 0) {
            ++n_grid;
            if (grid_sync(L.gbar, n_grid * (unsigned)P, ctl)) {
                // E tile of step 0
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_expect_tx(e_full, NKC * RMAX * 128);
                for (int kc = 0; kc < NKC; ++kc)
                    tma_load_3d(sbase + OFF_E + (uint32_t)kc * (RMAX * 128), &tmE, kc * KCH, 0, cta % kAReplicas, e_full,
                                l2_policy_evict_last());
                ++e_loads;
            }
            *s_stop = *s_abort;
        }
        bar_sync(BAR_STEP, BAR_STEP_N);
    }

    // ======================================================================= the serial steps
    if (warp == 0 && lane == 0) {
        // ---------------- producer: per step, per tile, the streamed W chunks then the U halves
        const uint64_t pol_u = l2_policy_evict_first(), pol_w = l2_policy_evict_first();
        int us = 0, ws = 0;
        uint32_t uph = 0, wph = 0;
        int u_fills = 0, w_fills = 0;
        bool stop = false;
        for (int k = 0; k < G && !stop; ++k)
            for (int t = 0; t < nt && !stop; ++t) {
                const int b = b0 + t;
                if (t >= n_tm + n_sm) {
                    for (int kc = 0; kc < NKC && !stop; ++kc) {
                        if (!lp_wait(w_empty(ws), wph ^ 1u, ctl)) {
                            stop = true;
                            break;
                        }
                        const uint32_t dst = sbase + OFF_WR + (uint32_t)ws * CHUNK_BYTES;
                        mbar_expect_tx(w_full(ws), CHUNK_BYTES);
                        tma_load_2d(dst, &tmW, b * 128, kc * KCH, w_full(ws), pol_w);
                        tma_load_2d(dst + BOX_BYTES, &tmW, b * 128 + 64, kc * KCH, w_full(ws), pol_w);
                        ++w_fills;
                        if (++ws == WR_ST) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    }
                }
                for (int h = 0; h < NH && !stop; ++h) {
                    if (!lp_wait(u_empty(us), uph ^ 1u, ctl)) {
                        stop = true;
                        break;
                    }
                    const uint32_t dst = sbase + OFF_U + (uint32_t)us * (NHALF * 128 * 2);
                    mbar_expect_tx(u_full(us), NHALF * 128 * 2);
                    tma_load_3d(dst, &tmU, b * 128, k, h * NHALF, u_full(us), pol_u);
                    tma_load_3d(dst + BOX_BYTES, &tmU, b * 128 + 64, k, h * NHALF, u_full(us), pol_u);
                    ++u_fills;
                    if (++us == U_ST) {
                        us = 0;
                        uph ^= 1u;
                    }
                }
            }
        // copies in flight land before the CTA leaves (fill n of a stage completes phase n / ST)
        for (int n = (u_fills > U_ST ? u_fills - U_ST : 0); n < u_fills; ++n)
            lp_drain(u_full(n % U_ST), (uint32_t)(n / U_ST) & 1u);
        for (int n = (w_fills > WR_ST ? w_fills - WR_ST : 0); n < w_fills; ++n)
            lp_drain(w_full(n % WR_ST), (uint32_t)(n / WR_ST) & 1u);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        int ws = 0;
        uint32_t wph = 0;
        uint32_t n_tile = 0;   // tiles issued over the whole call (accumulator phases)
        bool ok = true;
        if (n_sm) ok = lp_wait(s_full, 0u, ctl);
        for (int k = 0; k < G && ok; ++k) {
            if (!lp_wait(e_full, (uint32_t)k & 1u, ctl)) break;
            tc5::fence_after();
            for (int t = 0; t < nt && ok; ++t) {
                for (int h = 0; h < NH && ok; ++h) ok = lp_wait(acc_empty(h), (n_tile & 1u) ^ 1u, ctl);
                if (!ok) break;
                tc5::fence_after();
                const bool in_tmem = t < n_tm, in_smem = !in_tmem && t < n_tm + n_sm;
                for (int kc = 0; kc < NKC; ++kc) {
                    uint32_t a_base = 0;
                    if (!in_tmem && !in_smem) {
                        if (!lp_wait(w_full(ws), wph, ctl)) {
                            ok = false;
                            break;
                        }
                        tc5::fence_after();
                        a_base = sbase + OFF_WR + (uint32_t)ws * CHUNK_BYTES;
                    } else if (in_smem) {
                        a_base = sbase + OFF_S + (uint32_t)kc * CHUNK_BYTES;
                    }
                    for (int h = 0; h < NH; ++h) {
                        const uint32_t d = tmem + ACC_COL + (uint32_t)(h * NHALF);
#pragma unroll
                        for (int kk = 0; kk < KCH / 16; ++kk) {
                            const uint64_t bd =
                                sw128_desc(sbase + OFF_E + (uint32_t)kc * (RMAX * 128) + (uint32_t)h * (NHALF * 128) + kk * 32, 16, 1024);
                            const uint32_t acc = (kc | kk) != 0;
                            if (in_tmem)
                                mma_ts(d, tmem + (uint32_t)(t * TILE_COLS + kc * 32 + kk * 8), bd, acc);
                            else
                                mma_ss(d, sw128_desc(a_base + kk * (16 * 128), BOX_BYTES, 1024), bd, acc);
                        }
                    }
                    if (!in_tmem && !in_smem) {
                        tc5::commit(w_empty(ws));
                        if (++ws == WR_ST) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                for (int h = 0; h < NH; ++h) tc5::commit(acc_full(h));
                ++n_tile;
            }
            if (ok) tc5::commit(e_empty);
        }
        // every MMA issued above completes before TMEM is freed (after an abort too)
        tc5::commit(mma_done);
        lp_drain(mma_done, 0u);
    } else if (warp == 2 || warp >= LP_EPI_WARP0) {
        // ---------------- epilogue (warps 4-11) and the grid work (warp 2)
        const bool epi = warp >= LP_EPI_WARP0;
        const int qw = warp & 3, cg = (warp - LP_EPI_WARP0) >> 2, ew = warp - LP_EPI_WARP0;
        const int vl = 32 * qw + lane;
        const uint32_t ubox = (uint32_t)(vl >> 6) * BOX_BYTES, uvv = (uint32_t)(vl & 63);
        const PhiloxKey key = make_key(p.seed);
        int us = 0;
        uint32_t uph = 0, n_tile = 0;
        // owner threads (quarter 0) of request 64 h + 32 cg + lane: draft length, greedy flag
        int o_gamma[2] = {0, 0};
        bool o_greedy[2] = {false, false};
        if (epi && qw == 0)
            for (int h = 0; h < 2; ++h) {
                const int q = h * NHALF + 32 * cg + lane;
                if (q < R) {
                    int g = p.gamma ? p.gamma[q] : G;
                    if (g < 0 || g > G) {
                        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                        g = g < 0 ? 0 : G;
                    }
                    o_gamma[h] = g;
                    o_greedy[h] = p.temperature[q] == 0.f;
                }
            }
        // commit warps keep, per assigned request, the previous token and survival
        int c_prev[2] = {0, 0};
        float c_surv[2] = {1.f, 1.f};
        bool dead = false;
        for (int k = 0; k < G && !dead; ++k) {
            if (epi) {
                Lse2 run[2] = {{-INFINITY, 0.f}, {-INFINITY, 0.f}};
                float best_z[2] = {-INFINITY, -INFINITY};
                int best_b[2] = {-1, -1};
                for (int t = 0; t < nt; ++t) {
                    const int b = b0 + t;
                    const bool vin = b * 128 + vl < V;
                    for (int h = 0; h < NH; ++h) {
                        uint32_t acc[32];
                        const bool a_ok = __all_sync(0xffffffffu, lp_wait(acc_full(h), n_tile & 1u, ctl));
                        if (a_ok) {
                            tc5::fence_after();
                            tmem_ld32(tmem + ((uint32_t)(qw * 32) << 16) + ACC_COL + (uint32_t)(h * NHALF + 32 * cg), acc);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) acc[i] = 0u;
                        }
                        tc5::fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_empty(h));
                        const bool u_ok = __all_sync(0xffffffffu, lp_wait(u_full(us), uph, ctl));
                        float y[32];
                        const uint32_t ust = sbase + OFF_U + (uint32_t)us * (NHALF * 128 * 2) + ubox;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const uint32_t rr = (uint32_t)(32 * cg + i);
                            float u = 0.f;
                            if (u_ok)
                                u = __uint_as_float((uint32_t)lds_u16(ust + rr * 128 + ((((uvv >> 3) ^ (rr & 7)) << 4) |
                                                                                         ((uvv & 7) << 1)))
                                                    << 16);
                            const float x = u + __uint_as_float(acc[i]);
                            y[i] = vin ? x * s_scale[h * NHALF + 32 * cg + i] : -INFINITY;
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(u_empty(us));
                        if (++us == U_ST) {
                            us = 0;
                            uph ^= 1u;
                        }
                        // block maximum per request: lanes, then the four quarters
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = y[i];
                        const float mq = reduce_scatter32<true>(v, lane);
                        float* red_m = s_red + (cg * 2 + 0) * 128;
                        float* red_s = s_red + (cg * 2 + 1) * 128;
                        red_m[qw * 32 + lane] = mq;
                        bar_sync(1 + cg, 128);
                        const float M = fmaxf(fmaxf(red_m[lane], red_m[32 + lane]), fmaxf(red_m[64 + lane], red_m[96 + lane]));
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float Mi = __shfl_sync(0xffffffffu, M, i);
                            v[i] = Mi == -INFINITY ? 0.f : ex2(y[i] - Mi);
                        }
                        const float sq = reduce_scatter32<false>(v, lane);
                        red_s[qw * 32 + lane] = sq;
                        bar_sync(1 + cg, 128);
                        const float S = (red_s[lane] + red_s[32 + lane]) + (red_s[64 + lane] + red_s[96 + lane]);
                        if (qw == 0) {
                            // owner of request q: block key, running log-normaliser, leading block
                            const int q = h * NHALF + 32 * cg + lane;
                            bool lead = false;
                            if (q < R && k < o_gamma[h] && a_ok && u_ok) {
                                if (!(S >= 0.f) || M == INFINITY || M != M) raise_status(p.status, DSPARK_ERR_NONFINITE_INPUT);
                                if (S > 0.f) {
                                    run[h] = lse2_merge(run[h], Lse2{M, S});
                                    const float z = o_greedy[h]
                                                        ? M
                                                        : (M + log2f(S)) * kLn2 -
                                                              logf(-logf(uniform_at(key, p.round, kDraftBlock, (uint32_t)q,
                                                                                    (uint32_t)k, (uint32_t)b)));
                                    if (z > best_z[h]) {
                                        best_z[h] = z;
                                        best_b[h] = b;
                                        lead = true;
                                    }
                                }
                            }
                            const uint32_t mask = __ballot_sync(0xffffffffu, lead);
                            if (lane == 0) s_lead[cg] = mask;
                        }
                        bar_sync(1 + cg, 128);
                        // the leading block's logits of these requests, for the commit's element draw
                        const uint32_t mask = s_lead[cg];
                        if (mask) {
                            float* slot = L.slots + ((size_t)cta * RMAX + h * NHALF + 32 * cg) * 128 + vl;
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if ((mask >> i) & 1u) slot[(size_t)i * 128] = y[i];
                        }
                    }
                    ++n_tile;
                }
                if (qw == 0)
                    for (int h = 0; h < NH; ++h) {
                        const int q = h * NHALF + 32 * cg + lane;
                        if (q < R && k < o_gamma[h]) {
                            p.stats[(size_t)q * P + cta] = make_float2(run[h].m, run[h].s);
                            if (best_b[h] >= 0)
                                atomicMax(p.pick + (size_t)k * R + q,
                                          pack_pick(best_z[h], (int)(((uint32_t)best_b[h] << 15) | (uint32_t)cta)));
                        }
                    }
            }
            // ---- grid barrier 1: every CTA's partials, block keys and slots are written
            bar_sync(BAR_STEP, BAR_STEP_N);
            if (warp == 2 && lane == 0) {
                ++n_grid;
                (void)grid_sync(L.gbar, n_grid * (unsigned)P, ctl);
                *s_stop = *s_abort;
            }
            bar_sync(BAR_STEP, BAR_STEP_N);
            if (*s_stop) {
                dead = true;
                break;
            }
            // ---- commit: one warp per request
            if (epi) {
                int j = 0;
                for (int q = cta + P * ew; q < R; q += P * LP_EPI_WARPS, ++j) {
                    const int jj = j < 2 ? j : 1;   // at most two requests per warp keep state (R <= 128)
                    const size_t o = (size_t)q * G + k;
                    int g = p.gamma ? p.gamma[q] : G;
                    g = g < 0 ? 0 : (g > G ? G : g);
                    if (k == 0) {
                        c_prev[jj] = checked_index(p.anchor[q], V, p.status);
                        c_surv[jj] = 1.f;
                    }
                    if (k >= g) {
                        if (lane == 0) {
                            p.tokens[o] = -1;
                            p.conf[o] = p.surv[o] = p.draft_lse[o] = p.draft_logit[o] = 0.f;
                        }
                        if (p.a_rows)
                            for (int i = lane; i < KR; i += 32) p.a_rows[o * KR + i] = 0.f;
                        continue;
                    }
                    const bool greedy = p.temperature[q] == 0.f;
                    const unsigned long long pk = *reinterpret_cast<volatile unsigned long long*>(p.pick + (size_t)k * R + q);
                    const uint32_t idx = ~(uint32_t)pk;
                    int bstar = (int)(idx >> 15), cstar = (int)(idx & 0x7FFFu);
                    if (pk == 0ull || bstar >= nblk || cstar >= P) {
                        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                        bstar = 0;
                        cstar = 0;
                    }
                    // log-normaliser from the CTAs' partials
                    Lse2 tot{-INFINITY, 0.f};
                    for (int c2 = lane; c2 < P; c2 += 32) {
                        // written by other CTAs before the grid barrier: load past L1 (not coherent)
                        const float2 st = __ldcg(p.stats + (size_t)q * P + c2);
                        tot = lse2_merge(tot, Lse2{st.x, st.y});
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const Lse2 o2{__shfl_xor_sync(0xffffffffu, tot.m, off), __shfl_xor_sync(0xffffffffu, tot.s, off)};
                        tot = lse2_merge(tot, o2);
                    }
                    // element-level draw over the winning block's saved logits (4 per lane)
                    const float4 y4 = __ldcg(reinterpret_cast<const float4*>(
                        L.slots + ((size_t)cstar * RMAX + q) * 128 + lane * 4));
                    const float yv[4] = {y4.x, y4.y, y4.z, y4.w};
                    const int vb = bstar * 128 + lane * 4;
                    uint4 w4 = make_uint4(0, 0, 0, 0);
                    if (!greedy)
                        w4 = philox4x32_10(make_uint4((uint32_t)(vb >> 2), (uint32_t)k, (uint32_t)q,
                                                      counter_word3(p.round, kDraftElem)),
                                           key);
                    const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
                    ArgMax best{-INFINITY, -1};
                    float lv_best = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int v = vb + i;
                        if (v < V) {
                            const float lv = yv[i] * kLn2;
                            const float c = greedy ? lv : lv - logf(-logf(bits_to_uniform(wv[i])));
                            if (best.i < 0 || c > best.v) {
                                best = ArgMax{c, v};
                                lv_best = lv;
                            }
                        }
                    }
                    const ArgMax win = warp_argmax(best);
                    int tok = win.i;
                    const int src = tok >= 0 ? ((tok - bstar * 128) >> 2) : 0;
                    const float logit = __shfl_sync(0xffffffffu, lv_best, src & 31);
                    if (tok < 0) {
                        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                        tok = min(bstar * 128, V - 1);
                    }
                    // confidence head (eq. 7) on W_1[x_{k-1}] (or W_1[x_k]), survival product
                    const int prev = c_prev[jj];
                    float ep[8], en[8], we[8];
                    load8<__nv_bfloat16>(E + (size_t)prev * KR + lane * 8, ep);
                    load8<__nv_bfloat16>(E + (size_t)tok * KR + lane * 8, en);
                    load8<float>(p.w_e + lane * 8, we);
                    float dot = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) dot = fmaf(we[i], p.conf_token ? en[i] : ep[i], dot);
                    dot = warp_sum(dot) + __ldcg(L.hdot + o);
                    const float lc = (dot + p.b) / (p.sts_temp ? p.sts_temp[k] : 1.f);
                    const float c = 1.f / (1.f + expf(-lc));
                    const float s = c_surv[jj] * c;
                    if (lane == 0) {
                        if (!isfinite(lc)) raise_status(p.status, DSPARK_ERR_NONFINITE_INPUT);
                        p.tokens[o] = tok;
                        p.conf[o] = c;
                        p.surv[o] = s;
                        p.draft_lse[o] = greedy ? logit : (tot.m + log2f(tot.s)) * kLn2;
                        p.draft_logit[o] = logit;
                    }
                    if (p.a_rows)   // the Markov operand row W_1[x_{k-1}] (reported even when no bias is added)
#pragma unroll
                        for (int i = 0; i < 8; ++i) p.a_rows[o * KR + lane * 8 + i] = ep[i];
                    // the next step's conditioning row, in every copy
                    const uint4 row = *reinterpret_cast<const uint4*>(E + (size_t)tok * KR + lane * 8);
                    for (int rp = 0; rp < kAReplicas; ++rp)
                        *reinterpret_cast<uint4*>(an + rp * rep_stride + (size_t)q * KR + lane * 8) = row;
                    c_prev[jj] = tok;
                    c_surv[jj] = s;
                }
            }
            if (k + 1 == G) break;
            // ---- grid barrier 2: every conditioning row of step k + 1 is written; then the E tile
            bar_sync(BAR_STEP, BAR_STEP_N);
            if (warp == 2 && lane == 0) {
                ++n_grid;
                if (grid_sync(L.gbar, n_grid * (unsigned)P, ctl) && lp_wait(e_empty, (uint32_t)k & 1u, ctl)) {
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    mbar_expect_tx(e_full, NKC * RMAX * 128);
                    for (int kc = 0; kc < NKC; ++kc)
                        tma_load_3d(sbase + OFF_E + (uint32_t)kc * (RMAX * 128), &tmE, kc * KCH, 0, cta % kAReplicas,
                                    e_full, l2_policy_evict_last());
                    ++e_loads;
                }
                *s_stop = *s_abort;
            }
            bar_sync(BAR_STEP, BAR_STEP_N);
            if (*s_stop) dead = true;
        }
        // the last E tile copy lands before exit (it may be unconsumed after an abort)
        if (warp == 2 && lane == 0 && e_loads > 0) lp_drain(e_full, (uint32_t)(e_loads - 1) & 1u);
    }
    __syncwarp();
    tc5::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc5::fence_after();
        tc5::dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 lp_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            (void)cudaGetLastError();
    }
    return fn;
}

// CTAs that can be co-resident: one per SM (the shared memory allows no more), if cooperative
// launches are available; 0 otherwise
int lp_max_ctas()
{
    static int n = -1;
    if (n < 0) {
        n = 0;
        int dev = 0, sms = 0, coop = 0, per_sm = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
            cudaFuncSetAttribute(draft_loop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) ==
                cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, draft_loop_kernel, LP_THREADS, SMEM_BYTES) ==
                cudaSuccess &&
            per_sm >= 1)
            n = sms;
        (void)cudaGetLastError();
    }
    return n;
}

bool a16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

cudaError_t enc(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                const cuuint32_t* box)
{
    const cuuint32_t es[3] = {1, 1, 1};
    return lp_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? cudaSuccess
               : cudaErrorInvalidValue;
}

}  // namespace

int loop_ctas(int R, int V)
{
    const int nblk = (V + 127) / 128;
    const int sms = lp_max_ctas();
    return sms < nblk ? sms : nblk;
}

bool loop_supported(int dtype, int head, int R, int V, int r, const void* U, const void* E, const void* W,
                    const void* h, const void* w_h, const void* w_e)
{
    if (dtype != DSPARK_BF16 || head != DSPARK_HEAD_MARKOV || R < 1 || R > RMAX || r != KR || V % 8 != 0) return false;
    // at least 8 CTAs, so that each commit warp keeps at most two requests
    if ((V + 127) / 128 < 8 || loop_ctas(R, V) < 8) return false;
    if (!a16(U) || !a16(E) || !a16(W) || !a16(h) || !a16(w_h) || !a16(w_e)) return false;
    return lp_encode_fn() != nullptr;
}

size_t loop_slot_bytes(int R, int V) { return (size_t)loop_ctas(R, V) * RMAX * 128 * sizeof(float); }

cudaError_t launch_draft_loop(const DraftStep& p, float* slots, float* hdot, unsigned int* gbar, int* gabort,
                              cudaStream_t s)
{
    const int P = loop_ctas(p.R, p.V);
    if (P < 8) return cudaErrorNotSupported;
    CUtensorMap tmW, tmU, tmE;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.V, (cuuint64_t)p.r};
        const cuuint64_t strides[1] = {(cuuint64_t)p.V * 2};
        const cuuint32_t box[2] = {64, KCH};
        const cudaError_t e = enc(&tmW, p.W, 2, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.V, (cuuint64_t)p.G, (cuuint64_t)p.R};
        const cuuint64_t strides[2] = {(cuuint64_t)p.V * 2, (cuuint64_t)p.G * p.V * 2};
        const cuuint32_t box[3] = {64, 1, NHALF};
        const cudaError_t e = enc(&tmU, p.U, 3, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.r, (cuuint64_t)p.R, (cuuint64_t)kAReplicas};
        const cuuint64_t strides[2] = {(cuuint64_t)p.r * 2, (cuuint64_t)p.R * p.r * 2};
        const cuuint32_t box[3] = {KCH, RMAX, 1};
        const cudaError_t e = enc(&tmE, p.a_next, 3, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    LoopParams L;
    memset(&L, 0, sizeof L);
    L.d = p;
    L.d.n_stats = P;
    L.slots = slots;
    L.hdot = hdot;
    L.gbar = gbar;
    L.gabort = gabort;
    L.P = P;
    cudaError_t e = cudaMemsetAsync(gbar, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(gabort, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P);
    cfg.blockDim = dim3(LP_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, draft_loop_kernel, L, tmW, tmU, tmE);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
