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
//   warp 0      TMA producer: U tiles [64 requests x 128 columns] of the step, streamed W chunks;
//               it runs ahead into the next step as far as its rings allow (neither depends on
//               the draws)
//   warp 1      TMEM owner and MMA issuer: D[v][q] = sum_i W[i][v] E[x_{k-1}(q)][i] per block and
//               request half (M = 128 vocabulary rows, N = 64 requests, K = 16 per instruction)
//   warp 2      the grid barrier; then waits for the step's tokens and loads the next step's E
//               tile (their W_1 rows) from one of 8 replicas with 4 TMA copies
//   warp 3      the outputs of this CTA's requests (q = cta mod P): log-normaliser, confidence
//               head and survival product; off the serial path
//   warps 4-19  epilogue, two sets of eight warps, one set per request half. A warp holds lane
//               quarter (warp % 4) = 32 vocabulary rows and a column group of 32 requests. With the
//               16x256b TMEM load each thread holds 4 vocabulary rows x 8 requests, so the
//               per-request block maximum and sum of 2^(y - max) cost 3 in-thread steps per 4 rows
//               and a reduce-scatter over 8 threads (3 shuffle levels); the four quarters' partials
//               meet in shared memory behind one named barrier, and every thread then merges the
//               partials of one request (the four warps hold identical copies of each request's
//               running state, so each decides alone whether the block leads, and writes its own
//               rows of the leading block's logits to the CTA's slot).
//   After its last block every CTA posts, per request, its leading block's key in a packed
//   64-bit atomicMax (key, block, CTA). One grid barrier; then the CTA that holds the winning
//   block draws the element from its slot (Gumbel-max over 128 logits, one Philox call per lane)
//   and writes the token's W_1 row into the 8 replicas, then publishes the token with a release
//   store tagged with the step. Every CTA waits for the tags and loads the next E tile; the draw
//   costs one request per winner, not one per CTA.
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

constexpr int LP_THREADS = 640;                 // 20 warps
constexpr int LP_EPI_WARP0 = 4;                 // warps 4-19: epilogue
constexpr int LP_EPI_WARPS = 16;
constexpr int SET_WARPS = 8;                    // epilogue warps per request half
constexpr int NHALF = 64;                       // requests per MMA (N)
constexpr int RMAX = 128;                       // requests handled by this path
constexpr int KR = 256;                         // Markov rank r
constexpr int KCH = 64;                         // K per chunk (128 bytes of bf16)
constexpr int NKC = KR / KCH;                   // 4 chunks
constexpr int TM_TILES = 3;                     // W tiles held in tensor memory
constexpr int NT_MAX = 8;                       // vocabulary blocks per CTA
constexpr int MAX_P = 256;                      // CTAs (one per SM)
constexpr uint32_t TILE_COLS = KR / 2;          // TMEM columns of one W^T tile (bf16 pairs)
constexpr uint32_t ACC_COL = TM_TILES * TILE_COLS;   // 384: two accumulators of 64 columns
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t CHUNK_BYTES = KCH * 128 * 2;      // 16 KB: [64 K rows x 128 vocabulary] as 2 boxes
constexpr uint32_t BOX_BYTES = 8192;                 // [64 rows x 64 elements] bf16
constexpr uint32_t U_BYTES = NHALF * 128 * 2;        // one U stage [64 requests x 128 columns]
constexpr int WR_ST = 2;                        // streamed W chunk stages
constexpr int U_ST = 3;                         // U stages
constexpr int PF_TILES = 2;                     // tiles requested into L2 ahead of the rings
// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_E = 0;                                   // E tile: 4 chunks [128 rows x 64 K]
constexpr uint32_t OFF_S = OFF_E + NKC * RMAX * 128;           // 64 KB: the W tile kept in shared memory
constexpr uint32_t OFF_WR = OFF_S + NKC * CHUNK_BYTES;         // streamed W chunks
constexpr uint32_t OFF_U = OFF_WR + WR_ST * CHUNK_BYTES;       // U stages
constexpr uint32_t OFF_RED = OFF_U + U_ST * U_BYTES;           // [2 parity][2 set][2 cg][4 quarter][32] float2
constexpr uint32_t RED_BYTES = 2 * 2 * 2 * 4 * 32 * 8;
constexpr uint32_t OFF_GUM = OFF_RED + RED_BYTES;              // [NT_MAX][RMAX] block Gumbels of the step
constexpr uint32_t OFF_SCALE = OFF_GUM + NT_MAX * RMAX * 4;    // [RMAX] log2(e) / T per request
constexpr uint32_t OFF_TOK = OFF_SCALE + RMAX * 4;             // [RMAX] the step's tokens (warp 2 -> warp 3)
constexpr uint32_t OFF_PREV = OFF_TOK + RMAX * 4;              // [RMAX] x_{k-1} of the CTA's own requests
constexpr uint32_t OFF_SURV = OFF_PREV + RMAX * 4;             // [RMAX] survival of the CTA's own requests
constexpr uint32_t OFF_MISC = OFF_SURV + RMAX * 4;             // flags, TMEM base
constexpr uint32_t OFF_BAR = OFF_MISC + 64;
constexpr int N_BARS = 2 * WR_ST + 2 * U_ST + 4 + 5;
constexpr uint32_t SMEM_USED = OFF_BAR + N_BARS * 8;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;               // alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(OFF_S % 1024 == 0 && OFF_WR % 1024 == 0 && OFF_U % 1024 == 0, "swizzle atoms on 1 KB");
// the initial batch of TMEM-resident chunks is staged over E, S, W-ring and U regions
static_assert(TM_TILES * NKC * CHUNK_BYTES <= OFF_RED, "initial staging fits");

// named barriers: 1-4 the quarters of one (set, column group); the step barrier (warps 2-19);
// the epilogue warps; warps 2 and 3
constexpr int BAR_STEP = 5, BAR_STEP_N = 32 * (LP_THREADS / 32 - 2);
constexpr int BAR_EPI = 6, BAR_EPI_N = 32 * LP_EPI_WARPS;
constexpr int BAR_TOK = 7, BAR_TOK_N = 64;

constexpr unsigned long long DRAIN_NS = 4000000000ull;
constexpr uint32_t WAIT_HINT_NS = 100000;            // suspend hint of one mbarrier try_wait
constexpr uint32_t TAG_SHIFT = 18;                   // token tag: (step + 1) << 18 | token
constexpr uint32_t TOK_MASK = (1u << TAG_SHIFT) - 1u;

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

// The MMA warp runs its loop converged, with warp-uniform operands; one lane, elected inside the
// instruction sequence, issues each MMA and commit.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(IDESC_TA), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC_SA), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void commit_elect(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// try_wait that lets the hardware suspend the thread (up to the hint) until the phase completes,
// so that waiting warps leave the issue slots to the working ones
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(WAIT_HINT_NS)
        : "memory");
    return ok != 0;
}

// 16 lanes x 8 columns, four times along the columns (+8 each): thread t receives, in register
// 4j + {0, 1, 2, 3}, (lane t/4, column 2(t%4) + 8j), (t/4, 2(t%4) + 1 + 8j), (t/4 + 8, 2(t%4) + 8j),
// (t/4 + 8, 2(t%4) + 1 + 8j) relative to the address. Completion: tmem_wait_ld.
__device__ __forceinline__ void tmem_ld16x256(uint32_t taddr, uint32_t* v)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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

__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int* p)
{
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned int* p, unsigned int v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// four rows (r0..r3) of a 2-D map, columns [col, col + box width), into consecutive rows at dst
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int col, int r0, int r1, int r2,
                                            int r3, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar), "l"(policy)
        : "memory");
}

// L2 prefetch of one box of a 2-D / 3-D map (no shared memory, no completion)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// Reduce 8 values over the 8 lanes that share lane % 4 (lane bits 2-4): value c of every lane
// belongs to column c; on return lane l holds op over those lanes of column l / 4. Fixed pairing
// order: deterministic, and the same in every warp.
template <bool MAX>
__device__ __forceinline__ float reduce_scatter8(float (&v)[8], int lane)
{
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) {
        const bool up = ((lane >> 2) & s) != 0;
#pragma unroll
        for (int j = 0; j < s; ++j) {
            const float send = up ? v[j] : v[j + s];
            const float keep = up ? v[j + s] : v[j];
            const float recv = __shfl_xor_sync(0xffffffffu, send, s << 2);
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

__device__ __forceinline__ void give_up(LoopCtl c)
{
    *c.abort = 1;
    atomicExch(c.gabort, 1);
    raise_status(c.status, DSPARK_ERR_TIMEOUT);
}

// Bounded wait on a shared-memory barrier phase; false when the CTA aborted or the wait ran out.
// Inline: a call in the MMA and epilogue loops makes the compiler keep values live across it in
// the stack, and with the shared memory this kernel takes, L1 holds little of that stack (the MMA
// issue measured 3-4x slower with the call).
__device__ __forceinline__ bool lp_wait(uint32_t bar, uint32_t parity, LoopCtl c)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*c.abort) return false;
        if (globaltimer() - t0 > c.limit) {
            give_up(c);
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
    while (ld_relaxed_u32(gbar) < target) {
        if (ld_relaxed_s32(c.gabort)) {
            *c.abort = 1;
            return false;
        }
        if (globaltimer() - t0 > c.limit) {
            give_up(c);
            return false;
        }
    }
    __threadfence();
    return true;
}

// Bounded wait for the tokens of four requests (q0 .. q0 + 3, those with need[r]) at step k,
// each published by the CTA that drew it with a release store of ((k + 1) << 18) | token. The
// four tags are polled together with relaxed loads (an acquire load per tag serialises the
// polls); one acquire fence after the last one orders what the publishers wrote before their
// tags. false when the wait ran out or another CTA gave up.
__device__ __noinline__ bool wait_tokens(const unsigned int* tags, int q0, const bool (&need)[4], int k, int (&tok)[4],
                                         LoopCtl c)
{
    const unsigned int want = (unsigned int)(k + 1);
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (globaltimer() - t0 > c.limit) {
            give_up(c);
            return false;
        }
        bool all = true;
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (need[r] && tok[r] < 0) {
                const unsigned int v = ld_relaxed_u32(tags + q0 + r);
                if ((v >> TAG_SHIFT) == want)
                    tok[r] = (int)(v & TOK_MASK);
                else
                    all = false;
            }
        if (all) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            return true;
        }
        if (*c.abort || ld_relaxed_s32(c.gabort)) {
            *c.abort = 1;
            return false;
        }
    }
}

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(LP_THREADS, 1)
    draft_loop_kernel(const LoopParams L, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmG,
                      const __grid_constant__ CUtensorMap tmE)
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

    float* s_scale = reinterpret_cast<float*>(smem + OFF_SCALE);
    float* s_gum = reinterpret_cast<float*>(smem + OFF_GUM);
    int* s_tok = reinterpret_cast<int*>(smem + OFF_TOK);
    int* s_prev = reinterpret_cast<int*>(smem + OFF_PREV);
    float* s_surv = reinterpret_cast<float*>(smem + OFF_SURV);
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
    const PhiloxKey key = make_key(p.seed);
    unsigned int* tags = reinterpret_cast<unsigned int*>(p.x_cur);

    if (tid == 0) {
        for (int i = 0; i < WR_ST; ++i) {
            mbar_init(w_full(i), 1);
            mbar_init(w_empty(i), 1);
        }
        for (int i = 0; i < U_ST; ++i) {
            mbar_init(u_full(i), 1);
            mbar_init(u_empty(i), SET_WARPS);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(acc_full(h), 1);
            mbar_init(acc_empty(h), SET_WARPS);
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

    // w_h . h_k of every position (inputs only), spread over warps 2-19 of the grid: they enter the
    // step barrier before the first grid barrier, which publishes these writes
    if (warp >= 2) {
        const int gw = cta * (LP_THREADS / 32 - 2) + (warp - 2), nw = P * (LP_THREADS / 32 - 2);
        const __nv_bfloat16* H = static_cast<const __nv_bfloat16*>(p.h);
        const bool vec = p.d % 8 == 0 && (reinterpret_cast<uintptr_t>(p.h) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(p.w_h) & 15u) == 0;
        for (int pi = gw; pi < R * G; pi += nw) {
            const __nv_bfloat16* hr = H + (size_t)pi * p.d;
            float acc = 0.f;
            if (vec) {
#pragma unroll 4
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

    // ======================================================================= the serial steps
    if (warp == 0 && lane == 0) {
        // ---------------- producer: per step, per tile, the streamed W chunks then the U halves
        const uint64_t pol_u = l2_policy_evict_first(), pol_w = l2_policy_evict_first();
        int us = 0, ws = 0;
        uint32_t uph = 0, wph = 0;
        int u_fills = 0, w_fills = 0;
        bool stop = false;
        // tiles are taken in order n = k nt + t; the W chunks and U halves of tile n + PF_TILES are
        // requested into L2 when tile n is loaded, so that more bytes are in flight than the rings hold
        const int n_all = G * nt;
        int n_pf = 0;
        auto prefetch_upto = [&](int n_end) {
            for (; n_pf < n_end && n_pf < n_all; ++n_pf) {
                const int pk = n_pf / nt, pt = n_pf - pk * nt, pb = b0 + pt;
                if (pt >= n_tm + n_sm)
                    for (int kc = 0; kc < NKC; ++kc) {
                        tma_prefetch_2d(&tmW, pb * 128, kc * KCH);
                        tma_prefetch_2d(&tmW, pb * 128 + 64, kc * KCH);
                    }
                for (int h = 0; h < NH; ++h) {
                    tma_prefetch_3d(&tmU, pb * 128, pk, h * NHALF);
                    tma_prefetch_3d(&tmU, pb * 128 + 64, pk, h * NHALF);
                }
            }
        };
        for (int k = 0; k < G && !stop; ++k)
            for (int t = 0; t < nt && !stop; ++t) {
                const int b = b0 + t;
                prefetch_upto(k * nt + t + 1 + PF_TILES);
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
                    const uint32_t dst = sbase + OFF_U + (uint32_t)us * U_BYTES;
                    mbar_expect_tx(u_full(us), U_BYTES);
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
    } else if (warp == 1) {
        // ---------------- MMA issuer: the warp runs converged (uniform operands, descriptors as a
        // base plus constant offsets); lane 0 waits, one elected lane issues
        int ws = 0;
        uint32_t wph = 0;
        uint32_t n_tile = 0;   // tiles issued over the whole call (accumulator phases)
        auto wait_w = [&](uint32_t bar, uint32_t parity) {
            bool r = true;
            if (lane == 0) r = lp_wait(bar, parity, ctl);
            return __shfl_sync(0xffffffffu, (int)r, 0) != 0;
        };
        // descriptor address fields are 16-byte units: + (bytes >> 4) moves a descriptor
        const uint64_t dE = sw128_desc(sbase + OFF_E, 16, 1024);
        const uint64_t dS = sw128_desc(sbase + OFF_S, BOX_BYTES, 1024);
        const uint64_t dR = sw128_desc(sbase + OFF_WR, BOX_BYTES, 1024);
        bool ok = true;
        if (n_sm) ok = wait_w(s_full, 0u);
        for (int k = 0; k < G && ok; ++k) {
            if (!wait_w(e_full, (uint32_t)k & 1u)) break;
            tc5::fence_after();
            for (int t = 0; t < nt && ok; ++t) {
                for (int h = 0; h < NH && ok; ++h) ok = wait_w(acc_empty(h), (n_tile & 1u) ^ 1u);
                if (!ok) break;
                tc5::fence_after();
                const bool in_tmem = t < n_tm, in_smem = !in_tmem && t < n_tm + n_sm;
                const uint32_t a_tm = tmem + (uint32_t)(t * TILE_COLS);
                for (int kc = 0; kc < NKC; ++kc) {
                    uint64_t dA = dS + (uint64_t)((kc * CHUNK_BYTES) >> 4);
                    if (!in_tmem && !in_smem) {
                        if (!wait_w(w_full(ws), wph)) {
                            ok = false;
                            break;
                        }
                        tc5::fence_after();
                        dA = dR + (uint64_t)((ws * CHUNK_BYTES) >> 4);
                    }
                    const uint64_t dB = dE + (uint64_t)((kc * (RMAX * 128)) >> 4);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (h < NH) {
                            const uint32_t d = tmem + ACC_COL + (uint32_t)(h * NHALF);
#pragma unroll
                            for (int kk = 0; kk < KCH / 16; ++kk) {
                                const uint64_t bd = dB + (uint64_t)((h * (NHALF * 128) + kk * 32) >> 4);
                                const uint32_t acc = (kc | kk) != 0;
                                if (in_tmem)
                                    mma_ts(d, a_tm + (uint32_t)(kc * 32 + kk * 8), bd, acc);
                                else
                                    mma_ss(d, dA + (uint64_t)((kk * 16 * 128) >> 4), bd, acc);
                            }
                        }
                    if (!in_tmem && !in_smem) {
                        commit_elect(w_empty(ws));
                        if (++ws == WR_ST) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                for (int h = 0; h < NH; ++h) commit_elect(acc_full(h));
                ++n_tile;
            }
            if (ok) commit_elect(e_empty);
        }
        // every MMA issued above completes before TMEM is freed (after an abort too)
        commit_elect(mma_done);
        if (lane == 0) lp_drain(mma_done, 0u);
    } else if (warp == 2) {
        // ---------------- grid barrier, the step's tokens, the next E tile
        int gam[4];
        int rows[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int q = 4 * lane + r;
            int g = 0;
            rows[r] = 0;
            if (q < R) {
                g = p.gamma ? p.gamma[q] : G;
                g = g < 0 ? 0 : (g > G ? G : g);   // out-of-range lengths are flagged by the epilogue
                rows[r] = checked_index(p.anchor[q], V, p.status);
            }
            gam[r] = g;
        }
        unsigned int n_grid = 0;
        int e_loads = 0;
        // E tile of step 0: W_1 rows of the anchors, or zeros when the first step has no bias
        if (!*s_abort) {
            if (p.bias_first) {
                if (lane == 0) mbar_expect_tx(e_full, NKC * RMAX * 128);
                __syncwarp();
                const uint64_t pol = l2_policy_evict_last();
                for (int kc = 0; kc < NKC; ++kc)
                    tma_gather4(sbase + OFF_E + (uint32_t)kc * (RMAX * 128) + (uint32_t)lane * 512, &tmG, kc * KCH,
                                rows[0], rows[1], rows[2], rows[3], e_full, pol);
            } else {
                uint4* e4 = reinterpret_cast<uint4*>(smem + OFF_E);
                for (int i = lane; i < NKC * RMAX * 128 / 16; i += 32) e4[i] = make_uint4(0, 0, 0, 0);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(e_full);
            }
            e_loads = 1;
        }
        for (int k = 0; k < G; ++k) {
            bar_sync(BAR_STEP, BAR_STEP_N);
            if (lane == 0) {
                ++n_grid;
                (void)grid_sync(L.gbar, n_grid * (unsigned)P, ctl);
                *s_stop = *s_abort;
            }
            bar_sync(BAR_STEP, BAR_STEP_N);
            if (*s_stop) break;
            // the tokens of step k, as their winners publish them (with the W_1 rows in the replicas)
            bool need[4];
            int tok[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                need[r] = 4 * lane + r < R && k < gam[r];
                tok[r] = -1;
            }
            const bool got = __all_sync(0xffffffffu, wait_tokens(tags, 4 * lane, need, k, tok, ctl));
#pragma unroll
            for (int r = 0; r < 4; ++r) s_tok[4 * lane + r] = tok[r];
            bar_sync(BAR_TOK, BAR_TOK_N);
            if (k + 1 < G && got && lane == 0 && lp_wait(e_empty, (uint32_t)k & 1u, ctl)) {
                // the replicas were written with generic stores before each tag's release
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_expect_tx(e_full, NKC * RMAX * 128);
                const uint64_t pol = l2_policy_evict_last();
                for (int kc = 0; kc < NKC; ++kc)
                    tma_load_3d(sbase + OFF_E + (uint32_t)kc * (RMAX * 128), &tmE, kc * KCH, 0, cta % kAReplicas, e_full,
                                pol);
                ++e_loads;
            }
            e_loads = __shfl_sync(0xffffffffu, e_loads, 0);
        }
        // the last E tile copy lands before exit (it may be unconsumed after an abort)
        if (lane == 0 && e_loads > 0) lp_drain(e_full, (uint32_t)(e_loads - 1) & 1u);
    } else if (warp == 3) {
        // ---------------- outputs of this CTA's requests (q = cta + P j), one step behind the draw
        const __nv_bfloat16* E = static_cast<const __nv_bfloat16*>(p.E);
        if (lane == 0)
            for (int q = cta; q < R; q += P) {
                s_prev[q] = checked_index(p.anchor[q], V, p.status);
                s_surv[q] = 1.f;
            }
        __syncwarp();
        for (int k = 0; k < G; ++k) {
            bar_sync(BAR_STEP, BAR_STEP_N);
            bar_sync(BAR_STEP, BAR_STEP_N);
            if (*s_stop) break;
            bar_sync(BAR_TOK, BAR_TOK_N);
            for (int q = cta; q < R; q += P) {
                const size_t o = (size_t)q * G + k;
                int g = p.gamma ? p.gamma[q] : G;
                g = g < 0 ? 0 : (g > G ? G : g);
                if (k >= g) {
                    if (lane == 0) {
                        p.tokens[o] = -1;
                        p.conf[o] = p.surv[o] = p.draft_lse[o] = p.draft_logit[o] = 0.f;
                    }
                    if (p.a_rows)
                        for (int i = lane; i < KR; i += 32) p.a_rows[o * KR + i] = 0.f;
                    continue;
                }
                const int tok = s_tok[q];
                if (tok < 0) continue;   // the wait for it ran out: the call has failed
                const bool greedy = p.temperature[q] == 0.f;
                if (!greedy) {
                    // log-normaliser from the CTAs' partials of this step (written before the grid barrier)
                    const float2* st = p.stats + ((size_t)(k & 1) * R + q) * P;
                    float2 v[MAX_P / 32];
#pragma unroll
                    for (int i = 0; i < MAX_P / 32; ++i)
                        v[i] = lane + 32 * i < P ? __ldcg(st + lane + 32 * i) : make_float2(-INFINITY, 0.f);
                    Lse2 tot{-INFINITY, 0.f};
#pragma unroll
                    for (int i = 0; i < MAX_P / 32; ++i) tot = lse2_merge(tot, Lse2{v[i].x, v[i].y});
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const Lse2 o2{__shfl_xor_sync(0xffffffffu, tot.m, off),
                                      __shfl_xor_sync(0xffffffffu, tot.s, off)};
                        tot = lse2_merge(tot, o2);
                    }
                    if (lane == 0) p.draft_lse[o] = (tot.m + log2f(tot.s)) * kLn2;
                }
                // confidence head (eq. 7) on W_1[x_{k-1}] (or W_1[x_k]) and the hidden state h_k
                const int prev = s_prev[q];
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
                const float s = s_surv[q] * c;
                if (p.a_rows)   // the Markov operand row W_1[x_{k-1}] (reported even when no bias is added)
#pragma unroll
                    for (int i = 0; i < 8; ++i) p.a_rows[o * KR + lane * 8 + i] = ep[i];
                __syncwarp();
                if (lane == 0) {
                    if (!isfinite(lc)) raise_status(p.status, DSPARK_ERR_NONFINITE_INPUT);
                    p.conf[o] = c;
                    p.surv[o] = s;
                    s_prev[q] = tok;
                    s_surv[q] = s;
                }
                __syncwarp();
            }
        }
    } else if (warp >= LP_EPI_WARP0) {
        // ---------------- epilogue
        const int ew = warp - LP_EPI_WARP0, set = ew >> 3, cg = (ew >> 2) & 1, qw = warp & 3;
        const int t4 = lane & 3, tq = lane >> 2;
        const bool live = set < NH;
        // this thread's 8 requests: local column c = 2j + e is request colbase + e + 8j
        const int colbase = NHALF * set + 32 * cg + 2 * t4;
        float sc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) sc[c] = s_scale[colbase + (c & 1) + 8 * (c >> 1)];
        // the request whose block statistics this thread holds after the reductions (column tq)
        const int q_own = colbase + (tq & 1) + 8 * (tq >> 1);
        const int loc_own = q_own - NHALF * set - 32 * cg;
        const float sc_own = s_scale[q_own];
        int g_own = 0;
        bool greedy_own = false;
        if (q_own < R) {
            int g = p.gamma ? p.gamma[q_own] : G;
            if (g < 0 || g > G) {
                if (live && qw == 0) raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                g = g < 0 ? 0 : G;
            }
            g_own = g;
            greedy_own = p.temperature[q_own] == 0.f;
        }
        // U element (row e + 8j of this thread's column group, vocabulary row 32 qw + tq + 8i of
        // the block) in a stage: two boxes of [64 rows x 64 columns], 128-byte swizzle
        uint32_t uoff[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                uoff[i][e] = (uint32_t)(qw >> 1) * BOX_BYTES + (uint32_t)(32 * cg + 2 * t4 + e) * 128u +
                             ((((uint32_t)(4 * (qw & 1) + i)) ^ (uint32_t)(2 * t4 + e)) << 4) + (uint32_t)tq * 2u;
        const uint32_t t_acc = tmem + ((uint32_t)(32 * qw) << 16) + ACC_COL + (uint32_t)(set * NHALF + 32 * cg);
        float2* s_red = reinterpret_cast<float2*>(smem + OFF_RED);
        uint32_t n_tile = 0;
        // the block Gumbels of step k: one Philox call per request and group of 4 blocks
        auto block_gumbels = [&](int k) {
            const int e = ew * 32 + lane, q = e >> 2, grp = (b0 >> 2) + (e & 3);
            if (q < R && 4 * grp < b0 + nt) {
                const uint4 w = philox4x32_10(
                    make_uint4((uint32_t)grp, (uint32_t)k, (uint32_t)q, counter_word3(p.round, kDraftBlock)), key);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const int b = 4 * grp + s;
                    if (b >= b0 && b < b0 + nt) s_gum[(b - b0) * RMAX + q] = -logf(-logf(bits_to_uniform(ww[s])));
                }
            }
        };
        // the draw's requests of this warp (q = ew + 16 jj, held by lane jj): length, greedy flag
        const __nv_bfloat16* E = static_cast<const __nv_bfloat16*>(p.E);
        __nv_bfloat16* an = static_cast<__nv_bfloat16*>(p.a_next);
        int d_gam = 0, d_greedy = 0;
        if (lane < 8 && ew + 16 * lane < R) {
            const int q = ew + 16 * lane;
            const int g = p.gamma ? p.gamma[q] : G;
            d_gam = g < 0 ? 0 : (g > G ? G : g);
            d_greedy = p.temperature[q] == 0.f;
        }
        block_gumbels(0);
        bar_sync(BAR_EPI, BAR_EPI_N);
        for (int k = 0; k < G; ++k) {
            const bool act = q_own < R && k < g_own;
            Lse2 run{-INFINITY, 0.f};
            float best_z = -INFINITY;
            int best_b = -1;
            if (live)
                for (int t = 0; t < nt; ++t) {
                    const int b = b0 + t;
                    const uint32_t par = n_tile & 1u;
                    uint32_t a[32];
                    const bool a_ok = __all_sync(0xffffffffu, lp_wait(acc_full(set), par, ctl));
                    if (a_ok) {
                        tc5::fence_after();
                        tmem_ld16x256(t_acc, a);
                        tmem_ld16x256(t_acc + (16u << 16), a + 16);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) a[i] = 0u;
                    }
                    tc5::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty(set));
                    const uint32_t pos = n_tile * (uint32_t)NH + (uint32_t)set;
                    const int us = (int)(pos % U_ST);
                    const bool u_ok = __all_sync(0xffffffffu, lp_wait(u_full(us), (pos / U_ST) & 1u, ctl));
                    const uint32_t ust = sbase + OFF_U + (uint32_t)us * U_BYTES;
                    // y = U + D (unscaled) for vocabulary rows i, local columns c: y[4c + i]
                    float y[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const bool vin = b * 128 + 32 * qw + tq + 8 * i < V;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                float u = 0.f;
                                if (u_ok) u = __uint_as_float((uint32_t)lds_u16(ust + uoff[i][e] + j * 1024) << 16);
                                const float x = u + __uint_as_float(a[16 * (i >> 1) + 4 * j + 2 * (i & 1) + e]);
                                y[4 * (2 * j + e) + i] = vin ? x : -INFINITY;
                            }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(u_empty(us));
                    // per-request maximum over the quarter's 32 rows: 4 in-thread, then 8 threads
                    float v[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = fmaxf(fmaxf(y[4 * c], y[4 * c + 1]), fmaxf(y[4 * c + 2], y[4 * c + 3]));
                    const float m_q = reduce_scatter8<true>(v, lane);
                    float off[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float mc = __shfl_sync(0xffffffffu, m_q, (c << 2) | t4);
                        off[c] = mc == -INFINITY ? 0.f : mc * sc[c];
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = (ex2(fmaf(y[4 * c], sc[c], -off[c])) + ex2(fmaf(y[4 * c + 1], sc[c], -off[c]))) +
                               (ex2(fmaf(y[4 * c + 2], sc[c], -off[c])) + ex2(fmaf(y[4 * c + 3], sc[c], -off[c])));
                    const float s_q = reduce_scatter8<false>(v, lane);
                    if (act && a_ok && u_ok && (!(s_q >= 0.f) || m_q == INFINITY || m_q != m_q))
                        raise_status(p.status, DSPARK_ERR_NONFINITE_INPUT);
                    // the four quarters' partials of each request; every thread merges its request's
                    float2* red = s_red + (size_t)((par * 2 + set) * 2 + cg) * 4 * 32;
                    red[qw * 32 + loc_own] = make_float2(m_q == -INFINITY ? -INFINITY : m_q * sc_own, s_q);
                    bar_sync(1 + 2 * set + cg, 128);
                    float2 pq[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) pq[j] = red[j * 32 + loc_own];
                    const float mb = fmaxf(fmaxf(pq[0].x, pq[1].x), fmaxf(pq[2].x, pq[3].x));
                    float sb = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (pq[j].y > 0.f) sb += pq[j].y * ex2(pq[j].x - mb);
                    bool lead = false;
                    if (act && a_ok && u_ok && sb > 0.f) {
                        run = lse2_merge(run, Lse2{mb, sb});
                        const float z = greedy_own ? mb : (mb + log2f(sb)) * kLn2 + s_gum[t * RMAX + q_own];
                        if (z > best_z) {
                            best_z = z;
                            best_b = b;
                            lead = true;
                        }
                    }
                    // the leading block's logits of these requests, for the element draw
                    const uint32_t mask = __ballot_sync(0xffffffffu, lead);
                    if (mask) {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            if ((mask >> ((c << 2) | t4)) & 1u) {
                                float* slot = L.slots + ((size_t)cta * RMAX + colbase + (c & 1) + 8 * (c >> 1)) * 128 +
                                              32 * qw + tq;
#pragma unroll
                                for (int i = 0; i < 4; ++i) slot[8 * i] = y[4 * c + i] * sc[c];
                            }
                    }
                    ++n_tile;
                }
            // the CTA's partial log-normaliser and leading block key of each request
            if (live && qw == 0 && act) {
                p.stats[((size_t)(k & 1) * R + q_own) * P + cta] = make_float2(run.m, run.s);
                if (best_b >= 0)
                    atomicMax(p.pick + (size_t)k * R + q_own,
                              pack_pick(best_z, (int)(((uint32_t)best_b << 15) | (uint32_t)cta)));
            }
            bar_sync(BAR_EPI, BAR_EPI_N);   // every slot of the step is written
            // this warp's requests for the draw (q = ew + 16 jj): the CTA's own slots, in case it won
            float4 pre[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int q = ew + 16 * jj;
                pre[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q < R)
                    pre[jj] = __ldcg(reinterpret_cast<const float4*>(L.slots + ((size_t)cta * RMAX + q) * 128 + lane * 4));
            }
            bar_sync(BAR_STEP, BAR_STEP_N);
            bar_sync(BAR_STEP, BAR_STEP_N);   // warp 2 has passed the grid barrier
            if (*s_stop) break;
            // the draw of every request whose winning block this CTA holds
            unsigned long long pk_l = 0ull;
            if (lane < 8 && ew + 16 * lane < R)
                pk_l = *reinterpret_cast<volatile unsigned long long*>(p.pick + (size_t)k * R + ew + 16 * lane);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int q = ew + 16 * jj;
                if (q >= R) break;
                const unsigned long long pk = __shfl_sync(0xffffffffu, pk_l, jj);
                const int g = __shfl_sync(0xffffffffu, d_gam, jj);
                if (k >= g) continue;
                const uint32_t idx = ~(uint32_t)pk;
                const int bstar = (int)(idx >> 15), cstar = (int)(idx & 0x7FFFu);
                const bool valid = pk != 0ull && bstar < nblk && cstar < P;
                if (valid ? cstar != cta : q % P != cta) continue;
                const bool greedy = __shfl_sync(0xffffffffu, d_greedy, jj) != 0;
                int tok = 0;
                float logit = 0.f;
                if (valid) {
                    // element-level Gumbel-max over the winning block's saved logits (4 per lane)
                    const float yv[4] = {pre[jj].x, pre[jj].y, pre[jj].z, pre[jj].w};
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
                        const int vv = vb + i;
                        if (vv < V) {
                            const float lv = yv[i] * kLn2;
                            const float cand = greedy ? lv : lv - logf(-logf(bits_to_uniform(wv[i])));
                            if (best.i < 0 || cand > best.v) {
                                best = ArgMax{cand, vv};
                                lv_best = lv;
                            }
                        }
                    }
                    const ArgMax win = warp_argmax(best);
                    tok = win.i;
                    const int src = tok >= 0 ? ((tok - bstar * 128) >> 2) : 0;
                    logit = __shfl_sync(0xffffffffu, lv_best, src & 31);
                    if (tok < 0) {
                        raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                        tok = min(bstar * 128, V - 1);
                    }
                } else {
                    raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                }
                // the next step's conditioning row W_1[x_k], in every replica, before the tag
                if (k + 1 < g) {
                    const uint4 row = *reinterpret_cast<const uint4*>(E + (size_t)tok * KR + lane * 8);
#pragma unroll
                    for (int rp = 0; rp < kAReplicas; ++rp)
                        *reinterpret_cast<uint4*>(an + ((size_t)rp * R + q) * KR + lane * 8) = row;
                }
                // the lanes' stores are ordered before lane 0's release by the warp barrier
                __syncwarp();
                if (lane == 0) {
                    const size_t o = (size_t)q * G + k;
                    p.tokens[o] = tok;
                    p.draft_logit[o] = logit;
                    if (greedy) p.draft_lse[o] = logit;
                    st_release_u32(tags + q, ((uint32_t)(k + 1) << TAG_SHIFT) | (uint32_t)tok);
                }
            }
            if (k + 1 < G) {
                block_gumbels(k + 1);
                bar_sync(BAR_EPI, BAR_EPI_N);
            }
        }
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
    // tokens fit the step tag; at least 8 CTAs, each with at most NT_MAX vocabulary blocks
    if (V > (int)TOK_MASK + 1) return false;
    const int nblk = (V + 127) / 128, P = loop_ctas(R, V);
    if (nblk < 8 || P < 8 || P > MAX_P || (nblk + P - 1) / P > NT_MAX) return false;
    if (!a16(U) || !a16(E) || !a16(W) || !a16(h) || !a16(w_h) || !a16(w_e)) return false;
    return lp_encode_fn() != nullptr;
}

size_t loop_slot_bytes(int R, int V) { return (size_t)loop_ctas(R, V) * RMAX * 128 * sizeof(float); }

cudaError_t launch_draft_loop(const DraftStep& p, float* slots, float* hdot, unsigned int* gbar, int* gabort,
                              cudaStream_t s)
{
    const int P = loop_ctas(p.R, p.V);
    if (P < 8) return cudaErrorNotSupported;
    CUtensorMap tmW, tmU, tmG, tmE;
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
        // W_1 [V][r] for the row gathers: boxes of one row x 64 columns (tile::gather4 takes 4 rows)
        const cuuint64_t dims[2] = {(cuuint64_t)p.r, (cuuint64_t)p.V};
        const cuuint64_t strides[1] = {(cuuint64_t)p.r * 2};
        const cuuint32_t box[2] = {KCH, 1};
        const cudaError_t e = enc(&tmG, p.E, 2, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    {
        // the replicas [kAReplicas][R][r] of the next step's W_1 rows: boxes of 64 columns x 128 rows
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
    // cleared per call: the grid barrier, the abort flag, and the step tags (x_cur) through the
    // pick slots (the partial statistics between them are rewritten before they are read)
    cudaError_t e = cudaMemsetAsync(gbar, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(gabort, 0, sizeof(int), s);
    if (e == cudaSuccess) {
        const char* lo = reinterpret_cast<const char*>(p.x_cur);
        const char* hi = reinterpret_cast<const char*>(p.pick + (size_t)p.G * p.R);
        e = cudaMemsetAsync(p.x_cur, 0, (size_t)(hi - lo), s);
    }
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
    e = cudaLaunchKernelEx(&cfg, draft_loop_kernel, L, tmW, tmU, tmG, tmE);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
