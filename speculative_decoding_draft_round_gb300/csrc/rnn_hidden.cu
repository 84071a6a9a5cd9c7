// rnn_hidden.cu -- the h part of the RNN sequential head's projection (zhongzhuzhou.org notes,
// eq. 6), for every (request, position) before the serial loop:
//   yh[p][n] = sum_i W_rnn[n][2r + i] h[p][i],   p = q * gamma_max + k,  n < 3r,  i < d,
// with fp32 accumulation. It does not depend on the draws, so it is one dense GEMM
// [R*gamma_max x d] x [d x 3r] per call.
//
// Tensor-core path (bf16, shapes the copy engine takes): tcgen05 MMAs with M = 128 positions and
// N = 96 outputs, fp32 accumulators in TMEM, both operands K-major with the 128-byte swizzle,
// K streamed in 64-column chunks by TMA through a 6-stage ring. Warp 0 issues the copies, warp 1
// the MMAs, warps 2-5 read the accumulators (one TMEM lane quarter each) and store fp32 rows.
// Every wait is bounded by the global timer; a wait that runs out records DSPARK_ERR_TIMEOUT, the
// CTA stops issuing, lets its copies and MMAs land, frees its TMEM and returns.
// CUDA-core path (fp32, or shapes the copy engine does not take): 64 x 64 output tiles, K in
// slices of 16 staged in shared memory, fp32 fused multiply-adds.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace dspark {

namespace {

constexpr int kHM = 128;                                    // positions per tile (TMEM lanes)
constexpr int kHN = 96;                                     // outputs per tile (MMA N)
constexpr int kHK = 64;                                     // K per chunk: 128 bytes of bf16
constexpr int kHStages = 6;
constexpr uint32_t kHABytes = kHM * kHK * 2;                // 16 KB
constexpr uint32_t kHBBytes = kHN * kHK * 2;                // 12 KB
constexpr uint32_t kHStageBytes = kHABytes + kHBBytes;      // 28 KB, a multiple of 1024
constexpr uint32_t kHTmemCols = 128;
constexpr int kHThreads = 64 + 128;                         // warp 0 TMA, warp 1 MMA, 4 epilogue warps
constexpr uint32_t kHSmem = kHStages * kHStageBytes + 1024 + 256;
constexpr unsigned long long kHDrainNs = 4000000000ull;     // own copies and MMAs land long before
// instruction descriptor, kind::f16: D fp32, A = B = bf16, both K-major, N = 96, M = 128
constexpr uint32_t kHIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kHN >> 3) << 17) | ((uint32_t)(kHM >> 4) << 24);
static_assert(kHStageBytes % 1024 == 0 && kHABytes % 1024 == 0, "stages and operands on 1024-byte boundaries");

__device__ __forceinline__ bool h_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status,
                                    unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (globaltimer() - t0 > limit_ns) {
            *abort = 1;
            raise_status(status, DSPARK_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __noinline__ void h_drain(uint32_t bar, uint32_t parity)
{
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < kHDrainNs) {
    }
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp-wide)
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&v)[32])
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

// grid (ceil(P / 128) position tiles, 3r / 96 output tiles)
__global__ void __launch_bounds__(kHThreads, 1)
    rnn_hidden_tc_kernel(DraftStep p, const __grid_constant__ CUtensorMap hmap, const __grid_constant__ CUtensorMap wmap)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + kHStages * kHStageBytes;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kHStages + i); };
    const uint32_t done = bar0 + 8u * (2 * kHStages);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kHStages * kHStageBytes + 8 * (2 * kHStages + 1));
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = p.R * p.G, N3 = 3 * p.r;
    const int m0 = blockIdx.x * kHM, n0 = blockIdx.y * kHN;
    const int n_chunks = (p.d + kHK - 1) / kHK;
    if (tid == 0) {
        for (int i = 0; i < kHStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        mbar_init(done, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 1) tc5::alloc(s_tmem, kHTmemCols);
    tc5::fence_before();
    __syncthreads();
    tc5::fence_after();
    const uint32_t tmem = *s_tmem;
    // the previous call's steps read yh: wait for them before it is overwritten
    pdl_wait();
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: chunk c = columns [64c, 64c + 64) of the tile's h rows and of
        // its 96 W_rnn rows (from column 2r on)
        const uint64_t pol_a = l2_policy_evict_first();
        const uint64_t pol_b = l2_policy_evict_last();   // W_rnn is read by every position tile
        int issued = 0;
        for (int c = 0; c < n_chunks && !*s_abort; ++c) {
            const int st = c % kHStages;
            if (c >= kHStages && !h_wait(empty(st), ((c / kHStages) - 1) & 1u, s_abort, p.status, p.wait_ns)) break;
            const uint32_t dst = sbase + st * kHStageBytes;
            mbar_expect_tx(full(st), kHStageBytes);
            tma_load_2d(dst, &hmap, c * kHK, m0, full(st), pol_a);
            tma_load_2d(dst + kHABytes, &wmap, 2 * p.r + c * kHK, n0, full(st), pol_b);
            issued = c + 1;
        }
        if (*s_abort)   // copies still in flight land before the CTA leaves
            for (int c = (issued > kHStages ? issued - kHStages : 0); c < issued; ++c)
                h_drain(full(c % kHStages), (c / kHStages) & 1u);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        for (int c = 0; c < n_chunks; ++c) {
            const int st = c % kHStages;
            if (!h_wait(full(st), (c / kHStages) & 1u, s_abort, p.status, p.wait_ns)) break;
            tc5::fence_after();
            const uint32_t a = sbase + st * kHStageBytes, b = a + kHABytes;
#pragma unroll
            for (int kk = 0; kk < kHK / 16; ++kk)
                tc5::mma_ss(tmem, tc5::desc_sw128(a + kk * 32), tc5::desc_sw128(b + kk * 32), kHIdesc, (c | kk) != 0);
            tc5::commit(empty(st));
        }
        // completion of every MMA issued above (also after an abort, before TMEM is freed)
        tc5::commit(done);
        h_drain(done, 0u);
    } else if (warp >= 2) {
        // ---------------- epilogue: TMEM lane quarter warp % 4 = rows m0 + 32 (warp % 4) ..
        const bool ok = h_wait(done, 0u, s_abort, p.status, p.wait_ns);
        const bool all_ok = __all_sync(0xffffffffu, ok);
        const int row = (warp & 3) * 32 + lane, pos = m0 + row;
        if (all_ok) {
            tc5::fence_after();
            const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
#pragma unroll 1
            for (int cb = 0; cb < kHN / 32; ++cb) {
                uint32_t v[32];
                ld32(lane_base + (uint32_t)(cb * 32), v);
                if (pos < P) {
                    float4* dst = reinterpret_cast<float4*>(p.yh + (size_t)pos * N3 + n0 + cb * 32);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                             __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                }
            }
        }
    }
    tc5::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc5::fence_after();
        tc5::dealloc(tmem, kHTmemCols);
    }
}

// ---------------------------------------------------------------- CUDA-core path

constexpr int kSimtTile = 64;
constexpr int kSimtK = 16;

// grid (ceil(P / 64), ceil(3r / 64)), 256 threads: each thread 4 positions x 4 outputs
template <typename T>
__global__ void __launch_bounds__(256) rnn_hidden_simt_kernel(DraftStep p)
{
    __shared__ float hs[kSimtK][kSimtTile + 1];
    __shared__ float ws[kSimtK][kSimtTile + 1];
    pdl_wait();
    pdl_trigger();
    const int P = p.R * p.G, N3 = 3 * p.r, Z = 2 * p.r + p.d;
    const int m0 = blockIdx.x * kSimtTile, n0 = blockIdx.y * kSimtTile;
    const int t = threadIdx.x, tm = t / 16, tn = t % 16;
    const T* H = static_cast<const T*>(p.h);
    const T* Wr = static_cast<const T*>(p.W_rnn);
    float acc[4][4] = {};
    for (int k0 = 0; k0 < p.d; k0 += kSimtK) {
        for (int i = t; i < kSimtK * kSimtTile; i += 256) {
            const int kk = i % kSimtK, mm = i / kSimtK;
            const int pos = m0 + mm, n = n0 + mm, kx = k0 + kk;
            hs[kk][mm] = (pos < P && kx < p.d) ? ld(H, (size_t)pos * p.d + kx) : 0.f;
            ws[kk][mm] = (n < N3 && kx < p.d) ? ld(Wr, (size_t)n * Z + 2 * p.r + kx) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kSimtK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = hs[kk][tm * 4 + u];
                b[u] = ws[kk][tn * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int pos = m0 + tm * 4 + u;
        if (pos >= P) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int n = n0 + tn * 4 + v;
            if (n < N3) p.yh[(size_t)pos * N3 + n] = acc[u][v];
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 h_encode_fn()
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

bool hidden_tc_supported(const DraftStep& p)
{
    const int Z = 2 * p.r + p.d;
    // 16-byte row pitches and copy origins for the copy engine; 96-wide output tiles; 16-byte stores
    return p.dtype == DSPARK_BF16 && p.d % 8 == 0 && Z % 8 == 0 && p.r % 32 == 0 &&
           (reinterpret_cast<uintptr_t>(p.h) & 15u) == 0 && (reinterpret_cast<uintptr_t>(p.W_rnn) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(p.yh) & 15u) == 0 && h_encode_fn() != nullptr;
}

cudaError_t hidden_maps(const DraftStep& p, CUtensorMap* hmap, CUtensorMap* wmap)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = h_encode_fn();
    const cuuint32_t es2[2] = {1, 1};
    // h: [R*G][d] bf16, boxes of 64 columns x 128 rows
    const cuuint64_t hd[2] = {(cuuint64_t)p.d, (cuuint64_t)p.R * p.G};
    const cuuint64_t hs[1] = {(cuuint64_t)p.d * 2};
    const cuuint32_t hb[2] = {(cuuint32_t)kHK, (cuuint32_t)kHM};
    if (enc(hmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.h), hd, hs, hb, es2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // W_rnn: [3r][2r + d] bf16, boxes of 64 columns x 96 rows (columns past 2r + d read as zero)
    const int Z = 2 * p.r + p.d;
    const cuuint64_t wd[2] = {(cuuint64_t)Z, (cuuint64_t)3 * p.r};
    const cuuint64_t ws[1] = {(cuuint64_t)Z * 2};
    const cuuint32_t wb[2] = {(cuuint32_t)kHK, (cuuint32_t)kHN};
    if (enc(wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.W_rnn), wd, ws, wb, es2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_rnn_hidden(const DraftStep& p, cudaStream_t s)
{
    // s_0 = 0
    cudaError_t e = cudaMemsetAsync(p.state, 0, sizeof(float) * (size_t)p.R * p.r, s);
    if (e != cudaSuccess) return e;
    const int P = p.R * p.G;
    if (hidden_tc_supported(p)) {
        CUtensorMap hmap, wmap;
        e = hidden_maps(p, &hmap, &wmap);
        if (e != cudaSuccess) return e;
        static bool smem_set = false;
        if (!smem_set) {
            e = cudaFuncSetAttribute(rnn_hidden_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kHSmem);
            if (e != cudaSuccess) return e;
            smem_set = true;
        }
        const dim3 grid(cdiv(P, kHM), 3 * p.r / kHN);
        e = launch_pdl(rnn_hidden_tc_kernel, grid, dim3(kHThreads), kHSmem, s, p, hmap, wmap);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const dim3 grid(cdiv(P, kSimtTile), cdiv(3 * p.r, kSimtTile));
    e = p.dtype == DSPARK_BF16 ? launch_pdl(rnn_hidden_simt_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, p)
                               : launch_pdl(rnn_hidden_simt_kernel<float>, grid, dim3(256), 0, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
