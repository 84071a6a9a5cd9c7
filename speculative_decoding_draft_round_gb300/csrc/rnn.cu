// rnn.cu -- the RNN sequential head (zhongzhuzhou.org notes, eq. 6).
//
//   z_k = [s_{k-1}; W_1[x_{k-1}]; h_k],  [y_g; y_c; y_o] = W_rnn z_k  (W_rnn: [3r][2r+d]),
//   s_k = sigmoid(y_g) * s_{k-1} + (1 - sigmoid(y_g)) * tanh(y_c),  s_0 = 0,
//   B_k = tanh(y_o) W_2  -- the bias contraction of the Markov head with A = tanh(y_o).
// The h part of W_rnn z_k does not depend on the draws: one GEMM over every (request, position)
// before the serial loop (rnn_hidden.cu, fp32 accumulation). Each step then adds
// the [s_{k-1}; W_1[x_{k-1}]] part in fp32 (rnn_step_kernel), updates the state and writes the
// bias operand: fp32 rows for the CUDA-core path and the commit, and for the tensor-core path
// its bf16 rounding (the A tile copies) plus the bf16 rounding of the remainder (a second A
// operand in TMEM), so the contraction keeps about 16 significant bits of the operand.
#include "common.cuh"
#include "internal.h"

namespace dspark {

namespace {

constexpr int kRnnReq = 16;       // requests per CTA
constexpr int kRnnWarps = 8;      // one state element per warp
constexpr int kRnnThreads = 32 * kRnnWarps;
constexpr int kRnnSpan = 256;     // K elements a warp covers per pass: lane l takes 4l.. and 128+4l..
constexpr int kRnnPre = 2;        // passes of W_rnn fetched before the dependency wait (2r <= 512)
constexpr int kRnnVals = 3 * kRnnReq;   // per-lane partial sums: gates g, c, o of each request

// Four consecutive elements of a row, kept in the row's own type until used: one 16-byte (fp32)
// or 8-byte (bf16) load when the row is aligned for it, else element by element (zero at and
// past n).
template <typename T>
struct Raw4;
template <>
struct Raw4<float> {
    float4 v;
};
template <>
struct Raw4<__nv_bfloat16> {
    uint2 v;
};

__device__ __forceinline__ Raw4<float> load_raw4(const float* row, int c0, int n, bool vec)
{
    Raw4<float> o;
    if (vec && c0 + 4 <= n) {
        o.v = *reinterpret_cast<const float4*>(row + c0);
    } else {
        o.v.x = c0 < n ? row[c0] : 0.f;
        o.v.y = c0 + 1 < n ? row[c0 + 1] : 0.f;
        o.v.z = c0 + 2 < n ? row[c0 + 2] : 0.f;
        o.v.w = c0 + 3 < n ? row[c0 + 3] : 0.f;
    }
    return o;
}

__device__ __forceinline__ Raw4<__nv_bfloat16> load_raw4(const __nv_bfloat16* row, int c0, int n, bool vec)
{
    Raw4<__nv_bfloat16> o;
    if (vec && c0 + 4 <= n) {
        o.v = *reinterpret_cast<const uint2*>(row + c0);
    } else {
        uint32_t h[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) h[u] = c0 + u < n ? (uint32_t)__bfloat16_as_ushort(row[c0 + u]) : 0u;
        o.v = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    }
    return o;
}

__device__ __forceinline__ float4 to_f4(Raw4<float> a) { return a.v; }

__device__ __forceinline__ float4 to_f4(Raw4<__nv_bfloat16> a)
{
    return make_float4(__uint_as_float(a.v.x << 16), __uint_as_float(a.v.x & 0xffff0000u),
                       __uint_as_float(a.v.y << 16), __uint_as_float(a.v.y & 0xffff0000u));
}

// This lane's W elements of one pass: rows u = g, c, o; halves m = 0, 1 (K elements
// base + 128 m + 4 lane .. +3)
template <typename T>
struct RnnSlice {
    Raw4<T> w[3][2];
};

template <typename T>
__device__ __forceinline__ void load_slice(RnnSlice<T>& sl, const T* const (&rows)[3], int base, int lane, int K2,
                                           bool vec, bool has)
{
#pragma unroll
    for (int u = 0; u < 3; ++u)
#pragma unroll
        for (int m = 0; m < 2; ++m)
            sl.w[u][m] = load_raw4(rows[u], base + 128 * m + 4 * lane, has ? K2 : 0, vec);
}

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc)
{
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

// acc[3j + u] += the dot of this lane's K elements of pass `base` in row u with request j's z row;
// consecutive lanes read consecutive 16 bytes of z (no bank conflicts)
template <typename T>
__device__ __forceinline__ void rnn_accumulate(const RnnSlice<T>& sl, const float* zs, int base, int lane, int K2,
                                               float (&acc)[kRnnVals])
{
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int c0 = base + 128 * m + 4 * lane;
        if (c0 >= K2) continue;   // the slice holds zeros there
        float4 w[3];
#pragma unroll
        for (int u = 0; u < 3; ++u) w[u] = to_f4(sl.w[u][m]);
#pragma unroll
        for (int j = 0; j < kRnnReq; ++j) {
            float4 z;
            if ((K2 & 3) == 0 && c0 + 4 <= K2) {   // 16-byte aligned: every z row starts on a multiple of 4
                z = *reinterpret_cast<const float4*>(zs + j * K2 + c0);
            } else {
                z.x = zs[j * K2 + c0];
                z.y = c0 + 1 < K2 ? zs[j * K2 + c0 + 1] : 0.f;
                z.z = c0 + 2 < K2 ? zs[j * K2 + c0 + 2] : 0.f;
                z.w = c0 + 3 < K2 ? zs[j * K2 + c0 + 3] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 3; ++u) acc[3 * j + u] = dot4(w[u], z, acc[3 * j + u]);
        }
    }
}

// Sum the kRnnVals per-lane values over the warp by halving: at strides 16, 8, 4, 2 a lane keeps
// half of its values and adds its partner's copy of that half (24 + 12 + 6 + 3 shuffles), then the
// last three are summed over stride 1. Afterwards lanes 2j and 2j+1 hold the totals of values
// 3j, 3j+1, 3j+2 in v[0..2].
__device__ __forceinline__ void transpose_reduce(float (&v)[kRnnVals], int lane)
{
    static_assert(kRnnVals == 48, "the halving schedule below is for 16 requests");
#pragma unroll
    for (int half = kRnnVals / 2, bit = 16; half >= 3; half >>= 1, bit >>= 1) {
        const bool upper = (lane & bit) != 0;
#pragma unroll
        for (int x = 0; x < half; ++x) {
            const float send = upper ? v[x] : v[x + half];
            const float keep = upper ? v[x + half] : v[x];
            v[x] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
#pragma unroll
    for (int x = 0; x < 3; ++x) v[x] += __shfl_xor_sync(0xffffffffu, v[x], 1);
}

// One step of the recurrence for kRnnReq requests and kRnnWarps state elements: warp w owns
// element i of the state and dots its three rows W_g[i], W_c[i], W_o[i] (first 2r columns) with
// the requests' [s_{k-1}; W_1[x_{k-1}]] rows staged in shared memory. The rows' first 512
// columns are loaded before the dependency wait, overlapping the end of the previous commit;
// the grid (R/16 x r/8 CTAs of 8 warps, two per SM) fits one wave for R = 128 and r = 256.
template <typename T>
__global__ void __launch_bounds__(kRnnThreads, 2) rnn_step_kernel(DraftStep p)
{
    extern __shared__ float4 zs4[];   // [kRnnReq][2r] floats: s_{k-1}, then W_1[x_{k-1}]
    float* zs = reinterpret_cast<float*>(zs4);
    __shared__ int s_active[kRnnReq], s_tok[kRnnReq];
    const int q0 = blockIdx.x * kRnnReq;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int r = p.r, K2 = 2 * r, Z = 2 * r + p.d, k = p.k;
    const int i = blockIdx.y * kRnnWarps + warp;   // this warp's state element
    const bool has_i = i < r;
    const T* Wr = static_cast<const T*>(p.W_rnn);
    const bool vec = (Z * sizeof(T)) % 16 == 0 && (reinterpret_cast<uintptr_t>(Wr) & 15u) == 0;
    const int ii = has_i ? i : 0;
    const T* const rows[3] = {Wr + (size_t)ii * Z, Wr + (size_t)(r + ii) * Z, Wr + (size_t)(2 * r + ii) * Z};
    RnnSlice<T> pre[kRnnPre];
#pragma unroll
    for (int sp = 0; sp < kRnnPre; ++sp) load_slice(pre[sp], rows, sp * kRnnSpan, lane, K2, vec, has_i);
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
    pdl_wait();      // x_cur, the state and the operand buffers belong to the kernels before this one
    pdl_trigger();   // the statistics kernel may start its prologue
    const float* s_prev = p.state + (size_t)(k & 1) * p.R * r;
    float* s_next = p.state + (size_t)((k + 1) & 1) * p.R * r;
    const T* E = static_cast<const T*>(p.E);
    // a finished request (k >= gamma) has no operand: its x_cur may never have been written
    if (t < kRnnReq)
        s_tok[t] = s_active[t] ? checked_index(k == 0 ? p.anchor[q0 + t] : p.x_cur[q0 + t], p.V, p.status) : 0;
    // the h part of this warp's element for the request its lane pair finishes (loaded early)
    const int jr = lane >> 1, qr = q0 + jr;
    const bool fin = has_i && (lane & 1) == 0 && qr < p.R;
    float yh[3] = {0.f, 0.f, 0.f};
    if (fin) {
        const float* yrow = p.yh + ((size_t)qr * p.G + k) * 3 * r;
        yh[0] = yrow[i];
        yh[1] = yrow[r + i];
        yh[2] = yrow[2 * r + i];
    }
    __syncthreads();
    // stage the z rows 4 elements at a time, four chunks per thread in flight (r a multiple of 4
    // keeps a chunk on one side of the [s; W_1[x]] boundary; consecutive threads write
    // consecutive 16 bytes)
    const bool zvec = r % 4 == 0 && (reinterpret_cast<uintptr_t>(E) & (sizeof(T) * 4 - 1)) == 0;
    if (zvec) {
        const int cpr = K2 / 4, n = kRnnReq * cpr;
        for (int c00 = t; c00 < n; c00 += 4 * kRnnThreads) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int ci = c00 + u * kRnnThreads, j = ci / cpr, c0 = (ci - j * cpr) * 4;
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ci < n && s_active[j])
                    v[u] = c0 < r ? to_f4(load_raw4(s_prev + (size_t)(q0 + j) * r, c0, r, true))
                                  : to_f4(load_raw4(E + (size_t)s_tok[j] * r, c0 - r, r, true));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int ci = c00 + u * kRnnThreads;
                if (ci < n) zs4[ci] = v[u];   // chunk ci of row j sits at float offset j*K2 + 4*(ci - j*cpr) = 4 ci
            }
        }
    } else {
        for (int ci = t; ci < kRnnReq * K2; ci += kRnnThreads) {
            const int j = ci / K2, c = ci - j * K2;
            float v = 0.f;
            if (s_active[j]) v = c < r ? s_prev[(size_t)(q0 + j) * r + c] : ld(E, (size_t)s_tok[j] * r + (c - r));
            zs[ci] = v;
        }
    }
    __syncthreads();
    if (!has_i) return;   // warp-uniform, after the last block barrier
    float acc[kRnnVals];
#pragma unroll
    for (int x = 0; x < kRnnVals; ++x) acc[x] = 0.f;
#pragma unroll
    for (int sp = 0; sp < kRnnPre; ++sp) rnn_accumulate(pre[sp], zs, sp * kRnnSpan, lane, K2, acc);
    for (int base = kRnnPre * kRnnSpan; base < K2; base += kRnnSpan) {   // 2r > 512: the rest now
        RnnSlice<T> sl;
        load_slice(sl, rows, base, lane, K2, vec, true);
        rnn_accumulate(sl, zs, base, lane, K2, acc);
    }
    transpose_reduce(acc, lane);
    if (fin) {
        const size_t o = (size_t)qr * p.G + k;
        float op = 0.f;
        if (s_active[jr]) {
            const float yg = acc[0] + yh[0], yc = acc[1] + yh[1], yo = acc[2] + yh[2];
            const float gate = 1.f / (1.f + expf(-yg));
            s_next[(size_t)qr * r + i] = gate * zs[jr * K2 + i] + (1.f - gate) * tanhf(yc);
            op = tanhf(yo);
        }
        p.a_rows[o * r + i] = op;
        if (p.a_lo) {   // tensor-core path: bf16 operand copies and the remainder
            const __nv_bfloat16 hi = __float2bfloat16_rn(op);
            const __nv_bfloat16 lo = __float2bfloat16_rn(op - __bfloat162float(hi));
            __nv_bfloat16* an = static_cast<__nv_bfloat16*>(p.a_next);
            for (int rp = 0; rp < p.a_replicas; ++rp) an[((size_t)rp * p.R + qr) * r + i] = hi;
            static_cast<__nv_bfloat16*>(p.a_lo)[(size_t)qr * r + i] = lo;
        }
    }
}

}  // namespace

cudaError_t launch_rnn_step(const DraftStep& p, cudaStream_t s)
{
    const size_t smem = sizeof(float) * kRnnReq * 2 * (size_t)p.r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cdiv(p.R, kRnnReq), cdiv(p.r, kRnnWarps));
    cfg.blockDim = dim3(kRnnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.dtype == DSPARK_BF16) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(rnn_step_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return cudaLaunchKernelEx(&cfg, rnn_step_kernel<__nv_bfloat16>, p);
    }
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(rnn_step_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return cudaLaunchKernelEx(&cfg, rnn_step_kernel<float>, p);
}

}  // namespace dspark
