// rnn.cu -- the RNN sequential head (zhongzhuzhou.org notes, eq. 6).
//
//   z_k = [s_{k-1}; W_1[x_{k-1}]; h_k],  [y_g; y_c; y_o] = W_rnn z_k  (W_rnn: [3r][2r+d]),
//   s_k = sigmoid(y_g) * s_{k-1} + (1 - sigmoid(y_g)) * tanh(y_c),  s_0 = 0,
//   B_k = tanh(y_o) W_2  -- the bias contraction of the Markov head with A = tanh(y_o).
// The h part of W_rnn z_k does not depend on the draws: one GEMM over every (request, position)
// before the serial loop (cuBLAS, bf16 or fp32 inputs, fp32 accumulation). Each step then adds
// the [s_{k-1}; W_1[x_{k-1}]] part in fp32 (rnn_step_kernel), updates the state and writes the
// bias operand: fp32 rows for the CUDA-core path and the commit, and for the tensor-core path
// its bf16 rounding (the A tile copies) plus the bf16 rounding of the remainder (a second A
// operand in TMEM), so the contraction keeps about 16 significant bits of the operand.
#include <cublas_v2.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dspark {

namespace {

constexpr int kRnnReq = 8;        // requests per CTA
constexpr int kRnnElems = 32;     // state elements per CTA (4 per warp)
constexpr int kRnnThreads = 256;

std::mutex g_blas_mutex;
cublasHandle_t g_blas[64] = {};

// one cuBLAS handle per device, created on the first RNN-head call on that device
cublasHandle_t blas_handle()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!g_blas[dev] && cublasCreate(&g_blas[dev]) != CUBLAS_STATUS_SUCCESS) g_blas[dev] = nullptr;
    return g_blas[dev];
}

template <typename T>
__global__ void __launch_bounds__(kRnnThreads) rnn_step_kernel(DraftStep p)
{
    extern __shared__ float zs[];   // [kRnnReq][2r]: s_{k-1}, then W_1[x_{k-1}]
    __shared__ int s_active[kRnnReq];
    const int q0 = blockIdx.x * kRnnReq, i0 = blockIdx.y * kRnnElems;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int r = p.r, K2 = 2 * r, Z = 2 * r + p.d, k = p.k;
    const float* s_prev = p.state + (size_t)(k & 1) * p.R * r;
    float* s_next = p.state + (size_t)((k + 1) & 1) * p.R * r;
    const T* E = static_cast<const T*>(p.E);
    const T* Wr = static_cast<const T*>(p.W_rnn);
    if (t < kRnnReq) {
        const int q = q0 + t;
        int act = 0;
        if (q < p.R) {
            int g = p.gamma ? p.gamma[q] : p.G;
            g = g < 0 ? 0 : (g > p.G ? p.G : g);
            act = k < g;
        }
        s_active[t] = act;
    }
    __syncthreads();
    // a finished request (k >= gamma) has no operand: its x_cur may never have been written
    for (int idx = t; idx < kRnnReq * K2; idx += kRnnThreads) {
        const int j = idx / K2, c = idx % K2, q = q0 + j;
        float v = 0.f;
        if (s_active[j]) {
            if (c < r) {
                v = s_prev[(size_t)q * r + c];
            } else {
                const int prev = checked_index(k == 0 ? p.anchor[q] : p.x_cur[q], p.V, p.status);
                v = ld(E, (size_t)prev * r + (c - r));
            }
        }
        zs[idx] = v;
    }
    __syncthreads();
    for (int e = 0; e < kRnnElems / 8; ++e) {
        const int i = i0 + warp * (kRnnElems / 8) + e;
        if (i >= r) break;   // uniform per warp
        float acc[3][kRnnReq];
#pragma unroll
        for (int u = 0; u < 3; ++u)
#pragma unroll
            for (int j = 0; j < kRnnReq; ++j) acc[u][j] = 0.f;
        for (int c = lane; c < K2; c += 32) {
            const float wg = ld(Wr, (size_t)i * Z + c);
            const float wc = ld(Wr, (size_t)(r + i) * Z + c);
            const float wo = ld(Wr, (size_t)(2 * r + i) * Z + c);
#pragma unroll
            for (int j = 0; j < kRnnReq; ++j) {
                const float zj = zs[j * K2 + c];
                acc[0][j] = fmaf(wg, zj, acc[0][j]);
                acc[1][j] = fmaf(wc, zj, acc[1][j]);
                acc[2][j] = fmaf(wo, zj, acc[2][j]);
            }
        }
#pragma unroll
        for (int u = 0; u < 3; ++u)
#pragma unroll
            for (int j = 0; j < kRnnReq; ++j) acc[u][j] = warp_sum(acc[u][j]);
        if (lane < kRnnReq) {
            const int j = lane, q = q0 + j;
            float yg = 0.f, yc = 0.f, yo = 0.f;
#pragma unroll
            for (int jj = 0; jj < kRnnReq; ++jj)
                if (jj == j) {
                    yg = acc[0][jj];
                    yc = acc[1][jj];
                    yo = acc[2][jj];
                }
            if (q < p.R) {
                const size_t o = (size_t)q * p.G + k;
                float op = 0.f;
                if (s_active[j]) {
                    const float* yrow = p.yh + o * 3 * r;
                    yg += yrow[i];
                    yc += yrow[r + i];
                    yo += yrow[2 * r + i];
                    const float gate = 1.f / (1.f + expf(-yg));
                    s_next[(size_t)q * r + i] = gate * zs[j * K2 + i] + (1.f - gate) * tanhf(yc);
                    op = tanhf(yo);
                }
                p.a_rows[o * r + i] = op;
                if (p.a_lo) {   // tensor-core path: bf16 operand copies and the remainder
                    const __nv_bfloat16 hi = __float2bfloat16_rn(op);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(op - __bfloat162float(hi));
                    __nv_bfloat16* an = static_cast<__nv_bfloat16*>(p.a_next);
                    for (int rp = 0; rp < p.a_replicas; ++rp) an[((size_t)rp * p.R + q) * r + i] = hi;
                    static_cast<__nv_bfloat16*>(p.a_lo)[(size_t)q * r + i] = lo;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_rnn_hidden(const DraftStep& p, cudaStream_t s)
{
    // s_0 = 0
    cudaError_t e = cudaMemsetAsync(p.state, 0, sizeof(float) * (size_t)p.R * p.r, s);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_blas_mutex);
    cublasHandle_t h = blas_handle();
    if (!h) return cudaErrorNotSupported;
    if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    // yh [R*G][3r] = h [R*G][d] x W_rnn[:, 2r:2r+d]^T, in column-major terms
    // C (3r x RG, ld 3r) = A^T (A: the d x 3r column-major view of W_rnn from column 2r, ld 2r+d) x B (d x RG)
    const float one = 1.f, zero = 0.f;
    const int Z = 2 * p.r + p.d;
    const cudaDataType_t dt = p.dtype == DSPARK_BF16 ? CUDA_R_16BF : CUDA_R_32F;
    const size_t es = p.dtype == DSPARK_BF16 ? 2 : 4;
    const void* A = static_cast<const char*>(p.W_rnn) + 2 * (size_t)p.r * es;
    const cublasStatus_t st =
        cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, 3 * p.r, p.R * p.G, p.d, &one, A, dt, Z, p.h, dt, p.d, &zero, p.yh,
                     CUDA_R_32F, 3 * p.r, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    return st == CUBLAS_STATUS_SUCCESS ? cudaGetLastError() : cudaErrorUnknown;
}

cudaError_t launch_rnn_step(const DraftStep& p, cudaStream_t s)
{
    const dim3 grid(cdiv(p.R, kRnnReq), cdiv(p.r, kRnnElems));
    const size_t smem = sizeof(float) * kRnnReq * 2 * (size_t)p.r;
    if (p.dtype == DSPARK_BF16) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(rnn_step_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        rnn_step_kernel<__nv_bfloat16><<<grid, kRnnThreads, smem, s>>>(p);
    } else {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(rnn_step_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        rnn_step_kernel<float><<<grid, kRnnThreads, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace dspark
