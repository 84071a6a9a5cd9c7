// sample_tc.cu -- the per-step bias contraction of the draft sampler, and the residual
// recompute of verification, on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// with the softmax statistics fused into the epilogue.
//
// Draft mode, for step k of "DSpark" (Markov head, zhongzhuzhou.org notes eq. 4-5;
// caijizhuo.github.io section 4 step 3), every request tile of 128 rows and every 128-wide
// vocabulary block b (one item):
//   D[m][n]  = sum_i A[m][i] * W_2[i][b*128 + n]      A = W_1[x_{k-1}(m)] (bf16 x bf16 -> fp32 in TMEM)
//   x[m][n]  = (U[m][k][b*128 + n] + D[m][n]) * log2(e) / T_m
//   block b: (max_n x, sum_n 2^(x - max)) (log2 units) -> the block key of the two-level draw
//            (packed 64-bit atomicMax per request) and the CTA's running (max, sum) of the row,
//            written once per CTA as its partial log-normaliser.
// Residual mode (verification, rejected requests packed into tiles): the same contraction at
// the rejected position and per block sum_n max(0, p_t(n) - p_d(n)).
// The V-wide bias lives only in TMEM; it never reaches global memory.
//
// Layout and roles (one persistent CTA per SM, 640 threads; items dealt round-robin in
// block-major order):
//   warp 0      TMA producer of W tiles: per item 4 K-chunks of [64 K x 128 N] bf16, two
//               64-column boxes each, 128-byte swizzle (MN-major B).
//   warp 1      TMEM allocator (512 columns: 3 accumulators of 128 x 128 fp32 and an A region)
//               and the single MMA-issuing thread (tcgen05.mma kind::f16, M=128, N=128, K=16
//               per instruction, cta_group::1).
//   warp 3      draft: TMA producer of U tiles [128 requests x 128 columns] via a 3-D map
//               (V, gamma, R), evict-first L2 policy.
//   warps 4-19  epilogue: four warpgroups, each owns 32 of the 128 accumulator columns; a
//               thread owns one request row (TMEM lane). Draft: the A tile arrives by TMA from
//               one of eight copies of the rows (K-major, 128-byte swizzle, shared memory).
//               Residual: the threads write A into TMEM and load their own U and target columns.
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records DSPARK_ERR_TIMEOUT,
// stops issuing work, waits (bounded) for its own TMA copies and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace dspark {
namespace {

constexpr int BM = 128;             // requests per tile = TMEM lanes
constexpr int BN = 128;             // vocabulary columns per item = one noise block
constexpr int BK = 64;              // K per shared-memory chunk (128 bytes of bf16)
constexpr int KMAX = 256;           // largest Markov rank held in the A tile
constexpr int TMEM_BUFS = 3;
constexpr int EPI_WARPS = 16;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int THREADS = 128 + EPI_THREADS;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_TMEM_COL = TMEM_BUFS * BN;      // A operand: 128 columns of packed bf16 pairs (K <= 256)
static_assert(A_TMEM_COL + KMAX / 2 <= TMEM_COLS, "accumulators and A must fit in TMEM");

constexpr uint32_t W_BOX_BYTES = BK * 64 * 2;        // 8 KB: [64 K x 64 N]
constexpr uint32_t W_STAGE_BYTES = 2 * W_BOX_BYTES;  // 16 KB
constexpr uint32_t U_BOX_BYTES = BM * 64 * 2;        // 16 KB: [128 rows x 64 N]

enum Mode { kDraftMode = 0, kResidualMode = 1 };

constexpr int A_REPLICAS = kAReplicas;   // copies of the draft A rows, so that ~19 CTAs share one

constexpr int MAX_TILES = 64;                                              // R <= 8192
constexpr uint32_t META_BYTES = BM * 40;
// Shared-memory layout of one mode. Draft mode: 5 W stages, U stages of two 128-byte-swizzled
// [128 x 64] boxes, and the A tile (the W_1 rows of the tile's previous tokens, K-major,
// 128-byte swizzle, r/64 boxes of [128 x 64]) loaded by TMA. Residual mode: 8 W stages and no U
// stages (each epilogue thread loads its own U and target columns); A lives in TMEM.
template <int MODE>
struct Lay {
    static constexpr int W_ST = MODE == kDraftMode ? 5 : 8;
    static constexpr int U_ST = 2;
    static constexpr uint32_t U_ST_BYTES = MODE == kDraftMode ? 2 * U_BOX_BYTES : 0;   // residual: no U stages
    static constexpr uint32_t A_BYTES = MODE == kDraftMode ? BM * KMAX * 2 : 0;   // draft: A tile in shared memory
    static constexpr uint32_t OFF_W = 0;
    static constexpr uint32_t OFF_U = OFF_W + W_ST * W_STAGE_BYTES;
    static constexpr uint32_t OFF_A = OFF_U + U_ST * U_ST_BYTES;           // 1024-byte aligned
    static constexpr uint32_t OFF_PART = OFF_A + A_BYTES;                   // [2][4][128] float2
    static constexpr uint32_t OFF_META = OFF_PART + 2 * 4 * BM * 8;        // per-row metadata, see RowMeta
    static constexpr uint32_t OFF_BAR = OFF_META + META_BYTES;
    static constexpr int N_BARS = 2 * W_ST + 2 * U_ST + 2 * TMEM_BUFS + 3;
    static constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;
    static constexpr uint32_t SMEM_USED = OFF_MISC + 16 + MAX_TILES * 4;
    static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;               // alignment slack
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
    static_assert(OFF_A % 1024 == 0, "A tile on a 1024-byte boundary (128-byte swizzle atoms)");
};

// A CTA's items it = i0, i0 + istep, ... in block-major order (block it / nt of tile it % nt),
// walked without a division per step; n counts the items visited
struct ItemIter {
    int it, tile, b, n, dq, dr, nt;
    __device__ ItemIter(int i0, int istep, int nt_)
        : it(i0), tile(i0 % nt_), b(i0 / nt_), n(0), dq(istep / nt_), dr(istep % nt_), nt(nt_) {}
    __device__ void next(int istep)
    {
        it += istep;
        ++n;
        b += dq;
        tile += dr;
        if (tile >= nt) {
            tile -= nt;
            ++b;
        }
    }
};

// Bound of the waits that drain this CTA's own copies and MMAs before it exits: these complete
// in microseconds once issued, whatever the limit of the other waits (a launch parameter).
constexpr unsigned long long DRAIN_LIMIT_NS = 4000000000ull;   // 4 s

// instruction descriptor, kind::f16: D fp32, A = B = bf16, A K-major (shared memory in draft mode,
// TMEM in residual mode), B MN-major, M = 128, N = 128
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                           ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

// ------------------------------------------------------------------ PTX wrappers

struct Ctl {
    volatile int* abort;
    int* status;
    unsigned long long limit_ns;   // bound of each wait (dspark_set_wait_limit)
};

// Wait for the phase of `bar` with the given parity; false if the CTA aborted or the wait ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, Ctl c)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort) return false;
        if (globaltimer() - t0 > c.limit_ns) {
            *c.abort = 1;
            raise_status(c.status, DSPARK_ERR_TIMEOUT);
            return false;
        }
    }
}

// Every lane waits; the result is uniform across the warp (false if any lane gave up), so that
// warp-collective instructions after it are never reached by part of a warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl c)
{
    const bool ok = mbar_wait(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag (used to drain our own copies before exit).
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity)
{
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < DRAIN_LIMIT_NS) {
    }
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory"); }

// shared-memory matrix descriptor, 128-byte swizzle (layout type 2), descriptor version 1
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

// D (TMEM) += A (TMEM: lane m = row m, column c = bf16 pair (2c, 2c+1)) x B (shared memory descriptor)
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(IDESC), "r"(accumulate)
        : "memory");
}

// D (TMEM) += A (shared memory descriptor) x B (shared memory descriptor)
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
        : "memory");
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

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// ------------------------------------------------------------------ kernel

// Per-row metadata of the current request tile (shared memory, 32 bytes per row).
struct RowMeta {
    int prev;         // token whose W_1 row forms this A row
    int active;       // row takes part (draft: k < gamma_q; residual: request rejected); draft: 2 = greedy
    int use_bias;     // A row is W_1[prev] (else zero)
    float scale;      // log2(e) / T
    float lse_d2;     // residual: draft log-normaliser of the rejected position, log2 units
    float lse_t2;     // residual: target log-normaliser of the same row, log2 units
    uint32_t u_row;   // residual: row index q*G + n of U (row of V elements)
    uint32_t t_row;   // residual: row index q*(G+1) + n of the target
    int q;            // the request of this row (residual rows are the rejected requests, packed)
    int pad;
};
static_assert(sizeof(RowMeta) == 40, "RowMeta is 40 bytes");

struct TcParams {
    DraftStep d;      // draft mode
    VerifyParams v;   // residual mode
    int R, G, V, r, nblk, k;
    int* status;
    unsigned long long wait_ns;   // bound of every wait that depends on another agent
};

// Does request q take part at this launch?
template <int MODE>
__device__ __forceinline__ bool row_takes_part(const TcParams& P, int q)
{
    if (q >= P.R) return false;
    if (MODE == kDraftMode) {
        const int g = P.d.gamma ? P.d.gamma[q] : P.G;
        return P.k < g;
    }
    return P.v.rej[q] >= 0;
}

// Request of row e of tile mt: the row itself in draft mode. In residual mode the n_act rejected
// requests are dealt over the ceil(n_act / 128) tiles round-robin, so the tiles fill evenly, and
// inside a tile the j-th row sits at e = (j % 4) * 32 + j / 4, so that a part-filled tile spreads
// its rows over the four TMEM lane quarters (the four epilogue warps of each column group); -1
// past the end of the list.
template <int MODE>
__device__ __forceinline__ int row_request(const TcParams& P, int mt, int e, int n_act)
{
    if (MODE == kDraftMode) return mt * BM + e;
    const int nt = (n_act + BM - 1) / BM;
    const int idx = ((e & 31) * 4 + (e >> 5)) * nt + mt;
    if (idx >= n_act) return -1;
    const int q = P.v.rej_list[idx];
    if (q < 0 || q >= P.R) {
        raise_status(P.status, DSPARK_ERR_DEVICE_INPUT);
        return -1;
    }
    return q;
}

template <int MODE>
__device__ __forceinline__ RowMeta row_meta(const TcParams& P, int q)
{
    RowMeta m{0, 0, 0, 0.f, 0.f, 0.f, 0u, 0u, q, 0};
    if (q < 0 || q >= P.R) return m;
    if (MODE == kDraftMode) {
        // inputs only (no output of the previous kernel): the A row itself comes from a_next
        const DraftStep& p = P.d;
        int g = p.gamma ? p.gamma[q] : p.G;
        if (g < 0 || g > p.G) {
            raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
            g = g < 0 ? 0 : p.G;
        }
        if (p.k >= g) return m;
        m.active = p.temperature[q] == 0.f ? 2 : 1;   // temperature 0: arg-max draft
        m.prev = q;   // row of a_next
        m.use_bias = (p.k > 0) || p.bias_first;
        m.scale = m.active == 2 ? kLog2e : kLog2e / p.temperature[q];
    } else {
        const VerifyParams& p = P.v;
        const int n = p.rej[q];
        if (n < 0) return m;
        m.active = 1;
        m.prev = checked_index(n == 0 ? p.anchor[q] : p.tokens[(size_t)q * p.G + n - 1], p.V, p.status);
        m.use_bias = (n > 0) || p.bias_first;
        m.scale = kLog2e / p.temperature[q];
        m.lse_d2 = p.draft_lse[(size_t)q * p.G + n] * kLog2e;
        m.lse_t2 = p.lse_t[(size_t)q * (p.G + 1) + n] * kLog2e;
        m.u_row = (uint32_t)(q * p.G + n);
        m.t_row = (uint32_t)(q * (p.G + 1) + n);
    }
    return m;
}

// Residual mode: this thread's 32 columns v0.. of its row of U and of the target, straight from
// global memory (8 x 16 bytes; V % 8 == 0 keeps every 8-column chunk wholly inside or outside).
__device__ __forceinline__ void load_res_cols(uint4 (&uv)[4], uint4 (&tv)[4], const VerifyParams& p, const RowMeta& rm,
                                              int v0, int V)
{
    const uint4* up = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.U) + (size_t)rm.u_row * V + v0);
    const uint4* tp =
        reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.target) + (size_t)rm.t_row * V + v0);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (v0 + 8 * c < V) {
            uv[c] = __ldg(up + c);
            tv[c] = __ldg(tp + c);
        }
    }
}

struct Ring {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int n)
    {
        if (++idx == n) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

// SPLIT (draft mode only): the A operand is a bf16 tile plus its bf16 remainder in TMEM (the RNN
// head's fp32 rows); a separate instance so that the Markov head's kernel carries none of it
template <int MODE, bool SPLIT = false>
__global__ void __launch_bounds__(THREADS, 1)
    stats_tc_kernel(const TcParams P, const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmU,
                    const __grid_constant__ CUtensorMap tmA)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    using L = Lay<MODE>;
    constexpr int W_STAGES = L::W_ST, U_STAGES = L::U_ST;
    constexpr uint32_t OFF_W = L::OFF_W, OFF_U = L::OFF_U, OFF_MISC = L::OFF_MISC;
    constexpr uint32_t U_STAGE_BYTES = L::U_ST_BYTES;
    float2* part = reinterpret_cast<float2*>(smem + L::OFF_PART);
    RowMeta* s_meta = reinterpret_cast<RowMeta*>(smem + L::OFF_META);
    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto w_full = [&](int i) { return bar0 + 8u * i; };
    auto w_empty = [&](int i) { return bar0 + 8u * (W_STAGES + i); };
    auto u_full = [&](int i) { return bar0 + 8u * (2 * W_STAGES + i); };
    auto u_empty = [&](int i) { return bar0 + 8u * (2 * W_STAGES + U_STAGES + i); };
    auto t_full = [&](int i) { return bar0 + 8u * (2 * W_STAGES + 2 * U_STAGES + i); };
    auto t_empty = [&](int i) { return bar0 + 8u * (2 * W_STAGES + 2 * U_STAGES + TMEM_BUFS + i); };
    const uint32_t a_full = bar0 + 8u * (2 * W_STAGES + 2 * U_STAGES + 2 * TMEM_BUFS);
    const uint32_t a_empty = a_full + 8u;
    const uint32_t mma_done = a_full + 16u;   // every MMA of this CTA has completed (before TMEM is freed)
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    int* s_ntiles = reinterpret_cast<int*>(smem + OFF_MISC + 8);
    int* s_tiles = reinterpret_cast<int*>(smem + OFF_MISC + 16);
    int* s_nact = reinterpret_cast<int*>(smem + OFF_MISC + 12);   // residual: rejected requests

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Ctl ctl{s_abort, P.status, P.wait_ns};
    const int n_mt = (P.R + BM - 1) / BM;

    // Tiles with at least one request taking part. Residual mode: the rows are the rejected
    // requests, packed in the order the previous kernel listed them, so ceil(n / 128) tiles.
    int n_act = 0;
    if (MODE == kResidualMode) {
        pdl_wait();
        n_act = min(max(*P.v.n_rej, 0), P.R);
    }
    if (tid == 0) {
        *s_ntiles = 0;
        *s_abort = 0;
        *s_nact = n_act;
    }
    __syncthreads();
    if (MODE == kResidualMode) {
        if (tid == 0) {
            for (int mt = 0; mt * BM < n_act; ++mt) s_tiles[mt] = mt;
            *s_ntiles = (n_act + BM - 1) / BM;
        }
        __syncthreads();
    } else {
        for (int mt = 0; mt < n_mt; ++mt) {
            const bool act = tid < BM && row_takes_part<MODE>(P, mt * BM + tid);
            if (__syncthreads_or(act) && tid == 0) s_tiles[(*s_ntiles)++] = mt;
        }
    }
    if (tid == 0) {
        for (int i = 0; i < W_STAGES; ++i) {
            mbar_init(w_full(i), 1);
            mbar_init(w_empty(i), 1);
        }
        for (int i = 0; i < U_STAGES; ++i) {
            mbar_init(u_full(i), 1);
            mbar_init(u_empty(i), EPI_WARPS);
        }
        for (int i = 0; i < TMEM_BUFS; ++i) {
            mbar_init(t_full(i), 1);
            mbar_init(t_empty(i), EPI_WARPS);
        }
        mbar_init(a_full, MODE == kDraftMode && SPLIT ? 2 : 1);   // split operand: the copy and the TMEM half
        mbar_init(a_empty, 1);
        mbar_init(mma_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_tmem)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    pdl_trigger();
    const int nblk = P.nblk;
    const int nt = *s_ntiles;
    const int n_items = nt * nblk;
    // items are dealt round-robin in block-major order (item it = block it / nt of tile it % nt):
    // at any moment the CTAs work on adjacent vocabulary blocks, so their U and W reads fall in the
    // same DRAM pages, and the nt tiles of one W block are read at the same time, by nt
    // neighbouring CTAs, so that W comes from DRAM once per step however many tiles there are.
    // The grid is a multiple of the tile count, so a CTA keeps one tile (one A load) throughout.
    // a CTA keeps one tile when the item stride is a multiple of the tile count: the CTAs past
    // the largest such stride (fewer than nt of them) sit this launch out
    const int i0 = blockIdx.x, istep = nt > 0 ? (int)gridDim.x - (int)gridDim.x % nt : (int)gridDim.x;
    const int n_items_cta = i0 < istep ? n_items : 0;
    const int nt_walk = nt > 0 ? nt : 1;   // no tiles: no items, and no division by zero in the walk
    const int KC = P.r / BK;

    if (warp == 0 && lane == 0) {
        // ---------------- W producer
        // W takes the default L2 policy: measured against evict-last and evict-first hints, it keeps
        // the most of the other kernels' working set (and of W) in L2 from one step to the next
        const uint64_t pol = l2_policy_evict_normal();
        Ring ws;
        uint32_t last_par[W_STAGES];
        bool filled[W_STAGES] = {};
        for (ItemIter I(i0, istep, nt_walk); I.it < n_items_cta && !*s_abort; I.next(istep)) {
            const int b = I.b;
            for (int kc = 0; kc < KC; ++kc) {
                if (!mbar_wait(w_empty(ws.idx), ws.phase ^ 1u, ctl)) break;
                const uint32_t dst = sbase + OFF_W + ws.idx * W_STAGE_BYTES;
                mbar_expect_tx(w_full(ws.idx), W_STAGE_BYTES);
                tma_load_2d(dst, &tmW, b * BN, kc * BK, w_full(ws.idx), pol);
                tma_load_2d(dst + W_BOX_BYTES, &tmW, b * BN + 64, kc * BK, w_full(ws.idx), pol);
                filled[ws.idx] = true;
                last_par[ws.idx] = ws.phase;
                ws.next(W_STAGES);
            }
        }
        if (*s_abort)
            for (int i = 0; i < W_STAGES; ++i)
                if (filled[i]) mbar_drain(w_full(i), last_par[i]);
    } else if (MODE == kDraftMode && warp == 3 && lane == 0) {
        // ---------------- U producer
        const uint64_t pol = l2_policy_evict_first();
        Ring us;
        uint32_t last_par[U_STAGES];
        bool filled[U_STAGES] = {false, false};
        for (ItemIter I(i0, istep, nt_walk); I.it < n_items_cta && !*s_abort; I.next(istep)) {
            const int mt = s_tiles[I.tile], b = I.b;
            if (!mbar_wait(u_empty(us.idx), us.phase ^ 1u, ctl)) break;
            const uint32_t dst = sbase + OFF_U + us.idx * U_STAGE_BYTES;
            mbar_expect_tx(u_full(us.idx), U_STAGE_BYTES);
            tma_load_3d(dst, &tmU, b * BN, P.k, mt * BM, u_full(us.idx), pol);
            tma_load_3d(dst + U_BOX_BYTES, &tmU, b * BN + 64, P.k, mt * BM, u_full(us.idx), pol);
            filled[us.idx] = true;
            last_par[us.idx] = us.phase;
            us.next(U_STAGES);
        }
        if (*s_abort)
            for (int i = 0; i < U_STAGES; ++i)
                if (filled[i]) mbar_drain(u_full(i), last_par[i]);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        Ring ws, tb;
        uint32_t a_par = 0;
        int cur_tile = -1;
        for (ItemIter I(i0, istep, nt_walk); I.it < n_items_cta; I.next(istep)) {
            const int tile = I.tile;
            if (tile != cur_tile) {
                if (cur_tile >= 0) mma_commit(a_empty);   // old A is free once its MMAs retire
                if (!mbar_wait(a_full, a_par, ctl)) break;
                a_par ^= 1u;
                cur_tile = tile;
                tc_fence_after();
            }
            if (!mbar_wait(t_empty(tb.idx), tb.phase ^ 1u, ctl)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(tb.idx * BN);
            bool ok = true;
            for (int kc = 0; kc < KC; ++kc) {
                if (!mbar_wait(w_full(ws.idx), ws.phase, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t b_addr = sbase + OFF_W + ws.idx * W_STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t bd = sw128_desc(b_addr + kk * 16 * 128, W_BOX_BYTES, 1024);
                    if (MODE == kDraftMode) {
                        // A: box kc of the tile in shared memory, K-major; 16 K elements = 32 bytes per step
                        const uint64_t ad = sw128_desc(sbase + L::OFF_A + kc * (BM * 128) + kk * 32, 16, 1024);
                        mma_bf16_ss(d_tmem, ad, bd, (kc | kk) != 0);
                        if (SPLIT)   // RNN head: + the operand's bf16 remainder, from TMEM
                            mma_bf16_ts(d_tmem, tmem_base + A_TMEM_COL + (uint32_t)(kc * (BK / 2) + kk * 8), bd, 1u);
                    } else {
                        const uint32_t a_tmem = tmem_base + A_TMEM_COL + (uint32_t)(kc * (BK / 2) + kk * 8);
                        mma_bf16_ts(d_tmem, a_tmem, bd, (kc | kk) != 0);
                    }
                }
                mma_commit(w_empty(ws.idx));
                ws.next(W_STAGES);
            }
            if (!ok) break;
            mma_commit(t_full(tb.idx));
            tb.next(TMEM_BUFS);
        }
        // every MMA issued above completes before the CTA frees its TMEM, after an abort too
        mma_commit(mma_done);
        mbar_drain(mma_done, 0u);
    } else if (warp >= 4) {
        // ---------------- epilogue (and A gather)
        // The A rows read the previous kernel's output and the block statistics overwrite what it
        // read: everything after the first tile's metadata waits for it (programmatic dependent
        // launch); residual-mode metadata itself reads the previous kernel's output.
        if (MODE == kResidualMode) pdl_wait();
        bool waited = MODE == kResidualMode;
        // Every epilogue warp runs the same sequence of named barriers whatever happens: after
        // an abort (a wait that gave up) a warp keeps iterating but skips its memory work, so no
        // warp is ever left alone in a barrier.
        const int e = tid - 128;
        const int q4 = warp & 3, g = (warp - 4) >> 2;
        const int m = q4 * 32 + lane;
        const __nv_bfloat16* E = static_cast<const __nv_bfloat16*>(MODE == kDraftMode ? P.d.E : P.v.E);
        Ring us, tb;
        uint32_t a_par = 0;
        int cur_tile = -1;
        bool live = true;
        int a_fills = 0;   // A-tile copies this thread issued (thread e == 0, draft mode)
        uint4 uv[4] = {}, tv[4] = {};
        RowMeta rm_reg{};
        bool have_next = false;   // residual: uv / tv already hold this item's columns
        // draft: this CTA's running (max, sum) of its row over the blocks it has processed, log2
        // units, written to stats[q][blockIdx.x] when the CTA leaves the tile (g == 0 threads)
        float run_m = -INFINITY, run_s = 0.f;
        uint64_t done_tiles = 0ull;   // request tiles whose rows this CTA has written
        const auto flush_run = [&](int mt_old) {
            const int q = mt_old * BM + m;
            if (MODE == kDraftMode && g == 0 && q < P.R) P.d.stats[(size_t)q * P.d.n_stats + blockIdx.x] = make_float2(run_m, run_s);
            done_tiles |= 1ull << mt_old;
            run_m = -INFINITY;
            run_s = 0.f;
        };
        for (ItemIter I(i0, istep, nt_walk); I.it < n_items_cta; I.next(istep)) {
            const int tile = I.tile, b = I.b;
            const int mt = s_tiles[tile];
            if (tile != cur_tile) {
                if (MODE == kDraftMode && cur_tile >= 0) flush_run(s_tiles[cur_tile]);
                if (cur_tile >= 0) {
                    live = live && warp_wait(a_empty, a_par, ctl);
                    a_par ^= 1u;
                }
                if (e < BM) s_meta[e] = row_meta<MODE>(P, row_request<MODE>(P, mt, e, *s_nact));
                if (!waited) {
                    pdl_wait();
                    waited = true;
                }
                epi_barrier();
                if (MODE == kDraftMode) {
                    // A = the tile's rows of a_next (W_1 of the previous tokens, written by the
                    // previous kernel) from this CTA's replica, one TMA tile per 64 columns
                    if (e == 0 && live) {
                        ++a_fills;
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        mbar_expect_tx(a_full, (uint32_t)(P.r / BK) * BM * 128u);
                        const uint64_t pol = l2_policy_evict_last();
                        for (int cb = 0; cb < P.r / BK; ++cb)
                            tma_load_3d(sbase + L::OFF_A + cb * (BM * 128), &tmA, cb * BK, mt * BM,
                                        (int)(blockIdx.x % P.d.a_replicas), a_full, pol);
                    }
                    // RNN head: the bf16 remainder of the operand rows goes to TMEM (the second A
                    // operand) while that copy flies, warpgroup g covering K elements [64g, 64g + 64)
                    // of its lanes' rows; a_full then takes a second arrival, so that the MMAs wait
                    // for both halves of the operand
                    if (SPLIT) {
                        if (live && g * BK < P.r) {
                            uint32_t a[32];
                            const int q = mt * BM + m;
                            if (q < P.R) {
                                const uint4* src = reinterpret_cast<const uint4*>(
                                    static_cast<const __nv_bfloat16*>(P.d.a_lo) + (size_t)q * P.r + g * BK);
                                uint4 c8[8];
#pragma unroll
                                for (int c = 0; c < 8; ++c) c8[c] = src[c];
#pragma unroll
                                for (int c = 0; c < 8; ++c) {
                                    a[4 * c] = c8[c].x;
                                    a[4 * c + 1] = c8[c].y;
                                    a[4 * c + 2] = c8[c].z;
                                    a[4 * c + 3] = c8[c].w;
                                }
                            } else {
#pragma unroll
                                for (int c = 0; c < 32; ++c) a[c] = 0u;
                            }
                            tmem_st32(tmem_base + ((uint32_t)(q4 * 32) << 16) + A_TMEM_COL + (uint32_t)(g * 32), a);
                            tc_fence_before();
                        }
                        epi_barrier();
                        if (e == 0 && live) mbar_arrive(a_full);
                    }
                } else {
                    // A = W_1[prev] rows into TMEM: warpgroup g writes K elements [64g, 64g + 64) of
                    // its four warps' lanes (32 columns of bf16 pairs), loaded with 8 independent
                    // 16-byte reads per thread
                    if (live && g * BK < P.r) {
                        const RowMeta& mr = s_meta[m];
                        uint32_t a[32];
                        if (mr.active && mr.use_bias) {
                            const __nv_bfloat16* rows = E;
                            const uint4* src = reinterpret_cast<const uint4*>(rows + (size_t)mr.prev * P.r + g * BK);
                            uint4 c8[8];
    #pragma unroll
                            for (int c = 0; c < 8; ++c) c8[c] = __ldg(src + c);
    #pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                a[4 * c] = c8[c].x;
                                a[4 * c + 1] = c8[c].y;
                                a[4 * c + 2] = c8[c].z;
                                a[4 * c + 3] = c8[c].w;
                            }
                        } else {
    #pragma unroll
                            for (int c = 0; c < 32; ++c) a[c] = 0u;
                        }
                        tmem_st32(tmem_base + ((uint32_t)(q4 * 32) << 16) + A_TMEM_COL + (uint32_t)(g * 32), a);
                        tc_fence_before();
                    }
                    epi_barrier();
                    if (e == 0 && live) mbar_arrive(a_full);
                }
                if (MODE == kDraftMode) rm_reg = s_meta[m];
                cur_tile = tile;
            }
            // this row's metadata for the current tile: a register copy in draft mode, read from shared
            // memory in residual mode (whose epilogue has no registers to spare)
            const RowMeta& rm = MODE == kDraftMode ? rm_reg : s_meta[m];
            const int v0 = b * BN + g * 32;
            // this thread's 32 columns of the row's input logits: U (draft) or U and target (residual)
            bool u_ok = live;
            if (MODE == kDraftMode) {
                u_ok = live && warp_wait(u_full(us.idx), us.phase, ctl);
                if (u_ok) {
                    const uint32_t ubox = sbase + OFF_U + us.idx * U_STAGE_BYTES + (g >> 1) * U_BOX_BYTES + m * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        uv[c] = ld_shared_v4(ubox + ((uint32_t)((((g & 1) << 2) + c) ^ (m & 7)) << 4));
                    __syncwarp();
                    if (lane == 0) mbar_arrive(u_empty(us.idx));
                }
                us.next(U_STAGES);
            } else {
                // rows of U and the target at the rejected positions: scattered 64-byte pieces, loaded by
                // the thread that uses them (one TMA copy per row and item was issue-bound in the copy
                // engine); the next item's are requested before this item's combine
                if (!have_next && live && rm.active) load_res_cols(uv, tv, P.v, rm, v0, P.V);
                have_next = false;
            }
            // accumulator columns 32g .. 32g+31 of this row
            uint32_t acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0u;
            const bool t_ok = u_ok && warp_wait(t_full(tb.idx), tb.phase, ctl);
            if (t_ok) {
                tc_fence_after();
                tmem_ld32(tmem_base + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(tb.idx * BN + g * 32), acc);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(t_empty(tb.idx));
            }
            tb.next(TMEM_BUFS);
            live = t_ok;
            // x = U + B (unscaled logits of the draft)
            float x[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t w4[4] = {uv[c].x, uv[c].y, uv[c].z, uv[c].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int j = c * 8 + h * 2;
                    x[j] = __uint_as_float(w4[h] << 16) + (rm.use_bias ? __uint_as_float(acc[j]) : 0.f);
                    x[j + 1] = __uint_as_float(w4[h] & 0xFFFF0000u) + (rm.use_bias ? __uint_as_float(acc[j + 1]) : 0.f);
                }
            }
            const bool tail = v0 + 32 > P.V;
            float2 partial;
            if (MODE == kDraftMode) {
                // block softmax statistics: max, then sum of 2^((x - max) * scale)
                if (tail) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (v0 + j >= P.V) x[j] = -INFINITY;
                }
                float mx = x[0];
#pragma unroll
                for (int j = 1; j < 32; ++j) mx = fmaxf(mx, x[j]);
                float pm = -INFINITY, ps = 0.f;
                if (mx > -INFINITY) {
                    const float nb = -mx * rm.scale;
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        s0 += ex2(fmaf(x[j], rm.scale, nb));
                        s1 += ex2(fmaf(x[j + 1], rm.scale, nb));
                    }
                    pm = mx * rm.scale;
                    ps = s0 + s1;
                }
                // a NaN logit leaves a NaN sum, a +inf one an infinite maximum (-inf is a zero weight)
                if (rm.active && (!(ps >= 0.f) || mx == INFINITY || mx != mx))
                    raise_status(P.status, DSPARK_ERR_NONFINITE_INPUT);
                partial = make_float2(pm, ps);
            } else {
                // residual mass: sum of max(0, p_t - p_d), both from log2-unit logits
                float rs = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t w4[4] = {tv[c].x, tv[c].y, tv[c].z, tv[c].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2) {
                            const int j = c * 8 + h * 2 + s2;
                            const float zt = __uint_as_float(s2 ? (w4[h] & 0xFFFF0000u) : (w4[h] << 16));
                            const float pt = ex2(fmaf(zt, rm.scale, -rm.lse_t2));
                            const float pd = ex2(fmaf(x[j], rm.scale, -rm.lse_d2));
                            const float d = pt - pd;
                            if (!(tail && v0 + j >= P.V) && d > 0.f) rs += d;
                        }
                    }
                }
                partial = make_float2(rs, 0.f);
            }
            float2* pp = part + (I.n & 1) * 4 * BM;
            pp[g * BM + m] = partial;
            if (MODE == kResidualMode && live && rm.active) {
                ItemIter J = I;
                J.next(istep);
                if (J.it < n_items && J.tile == I.tile) {
                    load_res_cols(uv, tv, P.v, rm, J.b * BN + g * 32, P.V);
                    have_next = true;
                }
            }
            epi_barrier();
            if (g == 0 && rm.active && live) {
                const size_t o = (size_t)(MODE == kDraftMode ? mt * BM + m : rm.q) * nblk + b;
                if (MODE == kDraftMode) {
                    float M = pp[m].x;
#pragma unroll
                    for (int gg = 1; gg < 4; ++gg) M = fmaxf(M, pp[gg * BM + m].x);
                    float S = 0.f;
#pragma unroll
                    for (int gg = 0; gg < 4; ++gg) {
                        const float2 t = pp[gg * BM + m];
                        if (t.y > 0.f) S += t.y * ex2(t.x - M);
                    }
                    // merge the block into this CTA's running log-normaliser of the row
                    if (M > run_m) {
                        run_s = run_s * ex2(run_m - M) + S;
                        run_m = M;
                    } else {
                        run_s += S * ex2(M - run_m);
                    }
                    // block-level Gumbel-max of the two-level draw, folded into a packed key
                    const int q = mt * BM + m;
                    // greedy requests take the block holding the maximum
                    const float z = rm.active == 2 ? M
                                                   : (M + log2f(S)) * kLn2 -
                                                         logf(-logf(uniform_at(make_key(P.d.seed), P.d.round, kDraftBlock,
                                                                               (uint32_t)q, (uint32_t)P.k, (uint32_t)b)));
                    atomicMax(P.d.pick + (size_t)P.k * P.R + q, pack_pick(z, b));
                } else {
                    P.v.res_stats[o] = pp[m].x + pp[BM + m].x + pp[2 * BM + m].x + pp[3 * BM + m].x;
                }
            }
        }
        if (MODE == kDraftMode) {
            // the last tile's partials, then empty ones for every other tile's rows: the commit
            // merges all n_stats entries of a row
            if (cur_tile >= 0) flush_run(s_tiles[cur_tile]);
            for (int mt2 = 0; mt2 * BM < P.R; ++mt2)
                if (!((done_tiles >> mt2) & 1ull)) flush_run(mt2);
            // the last A copy lands before the CTA exits (it may be unconsumed after an abort)
            if (e == 0 && a_fills > 0) mbar_drain(a_full, (uint32_t)(a_fills - 1) & 1u);
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            (void)cudaGetLastError();
    }
    return fn;
}


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int num_sms()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    }
    return n;
}

bool tc_supported(int dtype, int R, int V, int r, const void* U, const void* E, const void* W)
{
    if (dtype != DSPARK_BF16) return false;
    if (r % BK != 0 || r > KMAX || V % 8 != 0 || V < BN || R > MAX_TILES * BM) return false;
    if (!aligned16(U) || !aligned16(E) || !aligned16(W)) return false;
    return encode_fn() != nullptr;
}

bool tc_residual_supported(int dtype, int R, int V, int r, const void* U, const void* E, const void* W)
{
    return tc_supported(dtype, R, V, r, U, E, W);
}

size_t tc_stats_rows(int R) { return (size_t)R; }

// a multiple of the tile count (when every tile takes part, each CTA keeps one tile), at most
// one CTA per SM
int tc_grid(int R, int nblk)
{
    const int n_mt = (R + BM - 1) / BM, items = n_mt * nblk;
    int grid = num_sms();
    if (n_mt <= grid) grid -= grid % n_mt;
    if (items < grid) grid = items;
    return grid;
}

namespace {

cudaError_t encode_w(CUtensorMap* m, const void* W, int V, int r)
{
    const cuuint64_t dims[2] = {(cuuint64_t)V, (cuuint64_t)r};
    const cuuint64_t strides[1] = {(cuuint64_t)V * 2};
    const cuuint32_t box[2] = {64, BK};
    const cuuint32_t es[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? cudaSuccess
               : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t encode_w_block_map(CUtensorMap* m, const void* W, int V, int r)
{
    if (!encode_fn() || r < 1 || r > 256 || V % 8 != 0 || !aligned16(W)) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)V, (cuuint64_t)r};
    const cuuint64_t strides[1] = {(cuuint64_t)V * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BN, (cuuint32_t)r};
    const cuuint32_t es[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? cudaSuccess
               : cudaErrorInvalidValue;
}

namespace {

cudaError_t encode_u(CUtensorMap* m, const void* U, int V, int G, int R)
{
    const cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)G, (cuuint64_t)R};
    const cuuint64_t strides[2] = {(cuuint64_t)V * 2, (cuuint64_t)G * V * 2};
    const cuuint32_t box[3] = {64, 1, BM};
    const cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? cudaSuccess
               : cudaErrorInvalidValue;
}

// the draft A rows a_next, A_REPLICAS copies of [R][r]: boxes of 64 columns x 128 rows
cudaError_t encode_a(CUtensorMap* m, const void* A, int R, int r)
{
    const cuuint64_t dims[3] = {(cuuint64_t)r, (cuuint64_t)R, (cuuint64_t)A_REPLICAS};
    const cuuint64_t strides[2] = {(cuuint64_t)r * 2, (cuuint64_t)R * r * 2};
    const cuuint32_t box[3] = {BK, BM, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(A), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? cudaSuccess
               : cudaErrorInvalidValue;
}

template <int MODE, bool SPLIT = false>
cudaError_t launch_tc(const TcParams& P, const CUtensorMap& tmW, const CUtensorMap& tmU, const CUtensorMap& tmA,
                      cudaStream_t s)
{
    constexpr uint32_t SMEM_BYTES = Lay<MODE>::SMEM_BYTES;
    static bool smem_set = false;
    if (!smem_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(stats_tc_kernel<MODE, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        smem_set = true;
    }
    const int grid = tc_grid(P.R, P.nblk);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, stats_tc_kernel<MODE, SPLIT>, P, tmW, tmU, tmA);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_draft_stats_tc(const DraftStep& p, cudaStream_t s)
{
    if (!encode_fn()) return cudaErrorNotSupported;
    CUtensorMap tmW, tmU, tmA;
    cudaError_t e = encode_w(&tmW, p.W, p.V, p.r);
    if (e == cudaSuccess) e = encode_u(&tmU, p.U, p.V, p.G, p.R);
    if (e == cudaSuccess) e = encode_a(&tmA, p.a_next, p.R, p.r);
    if (e != cudaSuccess) return e;
    TcParams P;
    memset(&P, 0, sizeof P);
    P.d = p;
    P.R = p.R;
    P.G = p.G;
    P.V = p.V;
    P.r = p.r;
    P.nblk = p.nblk;
    P.k = p.k;
    P.status = p.status;
    P.wait_ns = p.wait_ns;
    return p.a_lo ? launch_tc<kDraftMode, true>(P, tmW, tmU, tmA, s) : launch_tc<kDraftMode>(P, tmW, tmU, tmA, s);
}

cudaError_t launch_residual_stats_tc(const VerifyParams& p, cudaStream_t s)
{
    if (!encode_fn()) return cudaErrorNotSupported;
    CUtensorMap tmW;
    const cudaError_t e = encode_w(&tmW, p.W, p.V, p.r);
    if (e != cudaSuccess) return e;
    TcParams P;
    memset(&P, 0, sizeof P);
    P.v = p;
    P.R = p.R;
    P.G = p.G;
    P.V = p.V;
    P.r = p.r;
    P.nblk = p.nblk;
    P.k = 0;
    P.status = p.status;
    P.wait_ns = p.wait_ns;
    return launch_tc<kResidualMode>(P, tmW, tmW, tmW, s);
}

}  // namespace dspark
