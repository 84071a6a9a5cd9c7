// rnn_tc.cu -- one serial step of the RNN sequential head on the tensor cores (zhongzhuzhou.org
// notes, eq. 6):
//   [y_g; y_c; y_o] = W_rnn[:, :2r] [s_{k-1}; W_1[x_{k-1}]] + yh_k   (yh_k: the h part, one GEMM
//                                                                   before the serial loop)
//   s_k = sigmoid(y_g) s_{k-1} + (1 - sigmoid(y_g)) tanh(y_c),   bias operand tanh(y_o).
// The contraction is [R x 2r] x [2r x 3r] per step, a dense GEMM: tcgen05 MMAs, M = 128 requests,
// N = 48 outputs (gates g, c, o of 16 state elements, so that a CTA's epilogue holds all three
// gates of its elements), K streamed in 64-column chunks by TMA. The operand rows live in a bf16
// buffer z[parity][R][3r] = [hi(s); lo(s); W_1[x]]: the fp32 state enters as its bf16 rounding plus
// the bf16 rounding of the remainder (two chunks against the same W columns, about 16 significant
// bits), W_1 rows are bf16 already. This kernel writes the next step's state halves; the commit
// writes the drawn token's W_1 row.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace dspark {

namespace {

constexpr int kRtM = 128;                                   // requests per tile (TMEM lanes)
constexpr int kRtEl = 16;                                   // state elements per CTA
constexpr int kRtN = 3 * kRtEl;                             // MMA N: gates g, c, o
constexpr int kRtK = 64;                                    // K per chunk: 128 bytes of bf16
constexpr int kRtStages = 6;
constexpr uint32_t kRtABytes = kRtM * kRtK * 2;             // 16 KB
constexpr uint32_t kRtBBox = kRtEl * kRtK * 2;              // 2 KB: one gate's 16 rows
constexpr uint32_t kRtStageBytes = kRtABytes + 3 * kRtBBox;   // 22 KB, a multiple of 1024
constexpr uint32_t kRtTmemCols = 64;
constexpr int kRtEpiGroups = 4;                            // epilogue warps per TMEM lane quarter
constexpr int kRtElT = kRtEl / kRtEpiGroups;                // state elements per epilogue thread
constexpr int kRtThreads = 64 + 128 * kRtEpiGroups;         // warp 0 TMA, warp 1 MMA, 16 epilogue warps
constexpr uint32_t kRtSmem = kRtStages * kRtStageBytes + 1024 + 256;
constexpr unsigned long long kRtWaitNs = 4000000000ull;     // 4 s
constexpr int kRtStF = 20;                                  // staged fp32 row stride (16 + 4 of padding)
constexpr int kRtStB = 24;                                  // staged bf16 row stride (16 + 8 of padding)
static_assert(2 * kRtM * kRtStF * 4 + 4 * kRtM * kRtStB * 2 <= kRtStages * kRtStageBytes, "staging fits the stages");
// instruction descriptor, kind::f16: D fp32, A = B = bf16, both K-major, N = 48, M = 128
constexpr uint32_t kRtIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRtN >> 3) << 17) | ((uint32_t)(kRtM >> 4) << 24);

// bounded wait for a barrier phase; false (status raised, abort flag set) when it runs out or the
// CTA already gave up
__device__ __forceinline__ bool rt_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (globaltimer() - t0 > kRtWaitNs) {
            *abort = 1;
            raise_status(status, DSPARK_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __noinline__ void rt_drain(uint32_t bar, uint32_t parity)
{
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < kRtWaitNs) {
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo_elem)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi_elem)) << 16);
}

// grid (r / 16 element blocks, ceil(R / 128) request tiles)
__global__ void __launch_bounds__(kRtThreads, 1)
    rnn_tc_kernel(DraftStep p, const __grid_constant__ CUtensorMap zmap, const __grid_constant__ CUtensorMap wmap)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + kRtStages * kRtStageBytes;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kRtStages + i); };
    const uint32_t done = bar0 + 8u * (2 * kRtStages);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kRtStages * kRtStageBytes + 8 * (2 * kRtStages + 1));
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e0 = blockIdx.x * kRtEl, mt = blockIdx.y;
    const int r = p.r, R = p.R, k = p.k, G = p.G;
    const int kc_r = r / kRtK;          // chunks per r columns
    const int n_chunks = 3 * kc_r;      // hi(s), lo(s), W_1[x]
    if (tid == 0) {
        for (int i = 0; i < kRtStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        mbar_init(done, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 1) tc5::alloc(s_tmem, kRtTmemCols);
    tc5::fence_before();
    __syncthreads();
    tc5::fence_after();
    const uint32_t tmem = *s_tmem;

    // epilogue: warp w >= 2 takes TMEM lane quarter w % 4 (row q) and elements e0 + 4 ge .. + 3,
    // ge = (w - 2) / 4. Inputs that no earlier kernel of this call writes, loaded first: the h part
    // of the projection (the GEMM before the serial loop) and the request's draft length.
    const int row = (warp & 3) * 32 + lane, q = mt * kRtM + row;
    const bool epi = warp >= 2;
    const int ge = epi ? (warp - 2) / 4 : 0, el = e0 + kRtElT * ge;
    bool active = false;
    float4 yh[3] = {};
    if (epi && q < R) {
        int g = p.gamma ? p.gamma[q] : G;
        g = g < 0 ? 0 : (g > G ? G : g);
        active = k < g;
        const float* yrow = p.yh + ((size_t)q * G + k) * 3 * r;
#pragma unroll
        for (int u = 0; u < 3; ++u) yh[u] = *reinterpret_cast<const float4*>(yrow + u * r + el);
    }
    // The operand rows z[parity] = [hi(s_{k-1}); lo(s_{k-1}); W_1[x_{k-1}]]: the state halves were written by
    // the previous step's kernel, which completed before the kernel this one follows (the commit) started; only
    // W_1[x_{k-1}] comes from that commit. So the state chunks and every W_rnn chunk are copied before the
    // dependency wait, and only the last r columns after it. Step 0 waits first: its seed kernel (zero state,
    // the anchor's row) is the one it follows.
    if (k == 0 || !(warp == 0 && lane == 0)) {
        if (k == 0) pdl_wait();
    }

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: chunk c of A = z[parity] columns [64c, 64c + 64) of the tile's
        // rows; of B = the 16 rows of each gate over the W_rnn columns that chunk multiplies
        const uint64_t pol = l2_policy_evict_last();
        const int par = k & 1;
        int issued = 0;
        bool waited = k == 0;
        for (int c = 0; c < n_chunks && !*s_abort; ++c) {
            const int st = c % kRtStages;
            if (c >= kRtStages && !rt_wait(empty(st), ((c / kRtStages) - 1) & 1u, s_abort, p.status)) break;
            if (!waited && c >= 2 * kc_r) {
                pdl_wait();      // W_1[x_{k-1}] comes from the commit this kernel follows
                waited = true;
            }
            if (c == 2 * kc_r || (k == 0 && c == 0))
                pdl_trigger();   // the statistics kernel may start its prologue
            const uint32_t dst = sbase + st * kRtStageBytes;
            mbar_expect_tx(full(st), kRtStageBytes);
            tma_load_3d(dst, &zmap, c * kRtK, mt * kRtM, par, full(st), pol);
            const int wcol = c < 2 * kc_r ? (c % kc_r) * kRtK : r + (c - 2 * kc_r) * kRtK;
#pragma unroll
            for (int u = 0; u < 3; ++u)
                tma_load_2d(dst + kRtABytes + u * kRtBBox, &wmap, wcol, u * r + e0, full(st), pol);
            issued = c + 1;
        }
        if (*s_abort)   // copies still in flight land before the CTA leaves
            for (int c = (issued > kRtStages ? issued - kRtStages : 0); c < issued; ++c)
                rt_drain(full(c % kRtStages), (c / kRtStages) & 1u);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        bool ok = true;
        for (int c = 0; c < n_chunks; ++c) {
            const int st = c % kRtStages;
            if (!rt_wait(full(st), (c / kRtStages) & 1u, s_abort, p.status)) {
                ok = false;
                break;
            }
            tc5::fence_after();
            const uint32_t a = sbase + st * kRtStageBytes, b = a + kRtABytes;
#pragma unroll
            for (int kk = 0; kk < kRtK / 16; ++kk)
                tc5::mma_ss(tmem, tc5::desc_sw128(a + kk * 32), tc5::desc_sw128(b + kk * 32), kRtIdesc, (c | kk) != 0);
            tc5::commit(empty(st));
        }
        if (ok) tc5::commit(done);
    } else if (epi) {
        // ---------------- epilogue: row q, elements el .. el + 3
        const float* s_prev = p.state + (size_t)(k & 1) * R * r;
        float4 sp4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q < R) sp4 = *reinterpret_cast<const float4*>(s_prev + (size_t)q * r + el);
        const bool ok = rt_wait(done, 0u, s_abort, p.status);
        const bool all_ok = __all_sync(0xffffffffu, ok);
        uint32_t acc[3][kRtElT];
        if (all_ok) {
            tc5::fence_after();
            const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(kRtElT * ge);
            tc5::ld4(lane_base + 0, acc[0]);
            tc5::ld4(lane_base + kRtEl, acc[1]);
            tc5::ld4(lane_base + 2 * kRtEl, acc[2]);
        }
        // The results go out through shared memory (the stage buffers, free once the MMAs have
        // completed): written row by row here, then stored with 2-4 lanes per row segment, so that
        // every 32-byte sector is written whole (a lane per row would write each sector in pieces,
        // and the 8 operand copies made that the longest part of the step).
        float* st_sn = reinterpret_cast<float*>(smem);            // [128][kRtStF] state
        float* st_op = st_sn + kRtM * kRtStF;                     // [128][kRtStF] bias operand
        __nv_bfloat16* st_b = reinterpret_cast<__nv_bfloat16*>(st_op + kRtM * kRtStF);   // [4][128][kRtStB]
        const int cl = kRtElT * ge;   // this thread's first element within the CTA's 16
        if (all_ok && q < R) {
            const float sp[kRtElT] = {sp4.x, sp4.y, sp4.z, sp4.w};
            const float yg0[kRtElT] = {yh[0].x, yh[0].y, yh[0].z, yh[0].w};
            const float yc0[kRtElT] = {yh[1].x, yh[1].y, yh[1].z, yh[1].w};
            const float yo0[kRtElT] = {yh[2].x, yh[2].y, yh[2].z, yh[2].w};
            float sn[kRtElT], op[kRtElT];
#pragma unroll
            for (int j = 0; j < kRtElT; ++j) {
                sn[j] = sp[j];
                op[j] = 0.f;
                if (active) {
                    const float yg = __uint_as_float(acc[0][j]) + yg0[j];
                    const float yc = __uint_as_float(acc[1][j]) + yc0[j];
                    const float yo = __uint_as_float(acc[2][j]) + yo0[j];
                    const float gate = 1.f / (1.f + expf(-yg));
                    sn[j] = gate * sp[j] + (1.f - gate) * tanhf(yc);
                    op[j] = tanhf(yo);
                }
            }
            // the state in fp32 and, for the next step's operand, its bf16 rounding and remainder
            uint32_t hi2[kRtElT / 2], lo2[kRtElT / 2], ohi2[kRtElT / 2], olo2[kRtElT / 2];
#pragma unroll
            for (int j = 0; j < kRtElT; j += 2) {
                const float h0 = __bfloat162float(__float2bfloat16_rn(sn[j]));
                const float h1 = __bfloat162float(__float2bfloat16_rn(sn[j + 1]));
                hi2[j / 2] = pack_bf16x2(h0, h1);
                lo2[j / 2] = pack_bf16x2(sn[j] - h0, sn[j + 1] - h1);
                const float g0 = __bfloat162float(__float2bfloat16_rn(op[j]));
                const float g1 = __bfloat162float(__float2bfloat16_rn(op[j + 1]));
                ohi2[j / 2] = pack_bf16x2(g0, g1);
                olo2[j / 2] = pack_bf16x2(op[j] - g0, op[j + 1] - g1);
            }
            fence_proxy_async();   // the stage buffers were last read by the MMAs (async proxy)
            *reinterpret_cast<float4*>(st_sn + row * kRtStF + cl) = make_float4(sn[0], sn[1], sn[2], sn[3]);
            *reinterpret_cast<float4*>(st_op + row * kRtStF + cl) = make_float4(op[0], op[1], op[2], op[3]);
            *reinterpret_cast<uint2*>(st_b + (0 * kRtM + row) * kRtStB + cl) = make_uint2(hi2[0], hi2[1]);
            *reinterpret_cast<uint2*>(st_b + (1 * kRtM + row) * kRtStB + cl) = make_uint2(lo2[0], lo2[1]);
            *reinterpret_cast<uint2*>(st_b + (2 * kRtM + row) * kRtStB + cl) = make_uint2(olo2[0], olo2[1]);
            *reinterpret_cast<uint2*>(st_b + (3 * kRtM + row) * kRtStB + cl) = make_uint2(ohi2[0], ohi2[1]);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(128 * kRtEpiGroups) : "memory");   // the epilogue warps
        if (all_ok) {
            const int e = threadIdx.x - 64;   // 0 .. 511
            // fp32 rows: 16 elements = 4 lanes x 16 bytes per row, 128 rows
            {
                const int rr = e >> 2, part = e & 3, qq = mt * kRtM + rr;
                if (qq < R) {
                    const size_t o = (size_t)qq * G + k;
                    float* s_next = p.state + (size_t)((k + 1) & 1) * R * r;
                    *reinterpret_cast<float4*>(s_next + (size_t)qq * r + e0 + 4 * part) =
                        *reinterpret_cast<const float4*>(st_sn + rr * kRtStF + 4 * part);
                    *reinterpret_cast<float4*>(p.a_rows + o * r + e0 + 4 * part) =
                        *reinterpret_cast<const float4*>(st_op + rr * kRtStF + 4 * part);
                }
            }
            // bf16 rows: 16 elements = 2 lanes x 16 bytes; state hi and lo (z, next parity),
            // operand remainder (a_lo) and the a_replicas copies of the operand's rounding (a_next)
            const int n_dst = 3 + p.a_replicas;
            __nv_bfloat16* zn = static_cast<__nv_bfloat16*>(p.zbuf) + (size_t)((k + 1) & 1) * R * 3 * r;
            for (int u = e; u < n_dst * 2 * kRtM; u += 128 * kRtEpiGroups) {
                const int dst = u / (2 * kRtM), rr = (u >> 1) % kRtM, half = u & 1, qq = mt * kRtM + rr;
                if (qq >= R) continue;
                const int src = dst < 3 ? dst : 3;
                const uint4 v = *reinterpret_cast<const uint4*>(st_b + (src * kRtM + rr) * kRtStB + 8 * half);
                __nv_bfloat16* out;
                if (dst == 0)
                    out = zn + (size_t)qq * 3 * r;                       // hi(s_k)
                else if (dst == 1)
                    out = zn + (size_t)qq * 3 * r + r;                   // lo(s_k)
                else if (dst == 2)
                    out = static_cast<__nv_bfloat16*>(p.a_lo) + (size_t)qq * r;
                else
                    out = static_cast<__nv_bfloat16*>(p.a_next) + ((size_t)(dst - 3) * R + qq) * r;
                *reinterpret_cast<uint4*>(out + e0 + 8 * half) = v;
            }
        }
    }
    tc5::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc5::fence_after();
        tc5::dealloc(tmem, kRtTmemCols);
    }
}

// z[0] for step 0: zero state halves, W_1 of the anchor
__global__ void __launch_bounds__(128) rnn_z0_kernel(DraftStep p)
{
    pdl_enter();
    const int q = blockIdx.x, r = p.r;
    const __nv_bfloat16* E = static_cast<const __nv_bfloat16*>(p.E);
    __nv_bfloat16* z = static_cast<__nv_bfloat16*>(p.zbuf) + (size_t)q * 3 * r;
    const int x0 = checked_index(p.anchor[q], p.V, p.status);
    for (int i = threadIdx.x; i < r; i += blockDim.x) {
        z[i] = __float2bfloat16_rn(0.f);
        z[r + i] = __float2bfloat16_rn(0.f);
        z[2 * r + i] = E[(size_t)x0 * r + i];
    }
}

PFN_cuTensorMapEncodeTiled_v12000 rt_encode_fn()
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

}  // namespace

bool rnn_tc_supported(const DraftStep& p)
{
    const int Z = 2 * p.r + p.d;
    return p.dtype == DSPARK_BF16 && p.a_lo != nullptr && p.zbuf != nullptr && p.r % kRtK == 0 && (Z % 8) == 0 &&
           (reinterpret_cast<uintptr_t>(p.W_rnn) & 15u) == 0 && (reinterpret_cast<uintptr_t>(p.zbuf) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(p.a_rows) & 15u) == 0 &&   // the epilogue's 16-byte stores
           rt_encode_fn() != nullptr;
}

cudaError_t rnn_tc_maps(const DraftStep& p, CUtensorMap* zmap, CUtensorMap* wmap)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = rt_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint32_t es3[3] = {1, 1, 1}, es2[2] = {1, 1};
    // z: [2][R][3r] bf16, boxes of 64 columns x 128 rows of one parity
    const cuuint64_t zd[3] = {(cuuint64_t)3 * p.r, (cuuint64_t)p.R, 2};
    const cuuint64_t zs[2] = {(cuuint64_t)3 * p.r * 2, (cuuint64_t)3 * p.r * p.R * 2};
    const cuuint32_t zb[3] = {(cuuint32_t)kRtK, (cuuint32_t)kRtM, 1};
    if (enc(zmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.zbuf, zd, zs, zb, es3, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // W_rnn: [3r][2r + d] bf16, boxes of 64 columns x 16 rows
    const int Z = 2 * p.r + p.d;
    const cuuint64_t wd[2] = {(cuuint64_t)Z, (cuuint64_t)3 * p.r};
    const cuuint64_t ws[1] = {(cuuint64_t)Z * 2};
    const cuuint32_t wb[2] = {(cuuint32_t)kRtK, (cuuint32_t)kRtEl};
    if (enc(wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.W_rnn), wd, ws, wb, es2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t launch_rnn_z0(const DraftStep& p, cudaStream_t s)
{
    const cudaError_t e = launch_pdl(rnn_z0_kernel, dim3(p.R), dim3(128), 0, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rnn_step_tc(const DraftStep& p, const CUtensorMap& zmap, const CUtensorMap& wmap, cudaStream_t s)
{
    static bool smem_set = false;
    if (!smem_set) {
        const cudaError_t e = cudaFuncSetAttribute(rnn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRtSmem);
        if (e != cudaSuccess) return e;
        smem_set = true;
    }
    const dim3 grid(p.r / kRtEl, cdiv(p.R, kRtM));
    const cudaError_t e = launch_pdl(rnn_tc_kernel, grid, dim3(kRtThreads), kRtSmem, s, p, zmap, wmap);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
