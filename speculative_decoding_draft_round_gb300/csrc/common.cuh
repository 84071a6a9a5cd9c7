// common.cuh -- device helpers shared by the libdspark kernels.
//
// Random numbers follow the counter-based generator stated in dspark.h:
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11), key = (seed lo, seed hi), counter =
// (e>>2, position, request, (round<<3)|purpose), word e&3,
// u = (2*(x>>9)+1) * 2^-24, Gumbel noise -log(-log u).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

constexpr int kNoiseBlock = DSPARK_NOISE_BLOCK;   // vocabulary block of the two-level Gumbel-max
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// random purposes (low 3 bits of counter word 3)
enum Purpose : uint32_t {
    kDraftElem = 0,    // element-level Gumbel of a draft draw
    kAccept = 1,       // acceptance uniform
    kFinalElem = 2,    // element-level Gumbel of the residual / bonus draw
    kDraftBlock = 3,   // block-level Gumbel of a draft draw
    kFinalBlock = 4    // block-level Gumbel of the residual / bonus draw
};

struct PhiloxKey {
    uint32_t k0, k1;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key)
{
    uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

__device__ __forceinline__ float bits_to_uniform(uint32_t x)
{
    // (x>>9) + 1/2 in units of 2^-23: exact in binary32 (24 significant bits)
    return __fmaf_rn((float)(x >> 9), 0x1.0p-23f, 0x1.0p-24f);
}

__device__ __forceinline__ uint32_t counter_word3(uint64_t round, uint32_t purpose)
{
    return (uint32_t)(round << 3) | purpose;
}

// one uniform for element e of (purpose, request, position)
__device__ __forceinline__ float uniform_at(PhiloxKey key, uint64_t round, uint32_t purpose, uint32_t req,
                                            uint32_t pos, uint32_t e)
{
    const uint4 w = philox4x32_10(make_uint4(e >> 2, pos, req, counter_word3(round, purpose)), key);
    const uint32_t sel = e & 3u;
    const uint32_t x = sel == 0 ? w.x : sel == 1 ? w.y : sel == 2 ? w.z : w.w;
    return bits_to_uniform(x);
}

__device__ __forceinline__ float gumbel_at(PhiloxKey key, uint64_t round, uint32_t purpose, uint32_t req,
                                           uint32_t pos, uint32_t e)
{
    return -logf(-logf(uniform_at(key, round, purpose, req, pos, e)));
}

__host__ __device__ inline PhiloxKey make_key(uint64_t seed)
{
    return PhiloxKey{(uint32_t)seed, (uint32_t)(seed >> 32)};
}

// ------------------------------------------------------------------ programmatic dependent launch
//
// A kernel launched with the programmatic-serialization attribute may start while the previous
// kernel on the stream is still running; it must call pdl_wait() before it reads anything that
// kernel writes or writes anything that kernel reads. pdl_trigger() lets the next such kernel start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Kernels that do nothing before the dependency: wait for the previous kernel, then let the next
// one be scheduled, so that its launch overlaps this kernel's work.
__device__ __forceinline__ void pdl_enter()
{
    pdl_wait();
    pdl_trigger();
}

// Launch with the programmatic-serialization attribute (the kernel calls pdl_wait / pdl_enter).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// 2^x by the hardware approximation (the SFU's ex2, flushing subnormal results to zero)
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------ element loads

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ float ld(const T* p, size_t i) { return to_f32<T>(p[i]); }

// ------------------------------------------------------------------ packed arg-max key
//
// (value, index) packed into 64 bits so that unsigned atomicMax keeps the larger value and, on
// equal values, the lower index: high word = value bits made order-preserving, low = ~index.
// NaN values are packed as -infinity; 0 means "no candidate".
__device__ __forceinline__ unsigned long long pack_pick(float z, int idx)
{
    if (z != z) z = -INFINITY;
    const uint32_t b = __float_as_uint(z);
    const uint32_t key = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)idx;
}

__device__ __forceinline__ int unpack_pick_index(unsigned long long k) { return (int)~(uint32_t)k; }

// ------------------------------------------------------------------ status word

__device__ __forceinline__ void raise_status(int* status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// clamp a device-supplied index into [0, n) and flag an out-of-range value
__device__ __forceinline__ int checked_index(int x, int n, int* status)
{
    if (x < 0 || x >= n) {
        raise_status(status, DSPARK_ERR_DEVICE_INPUT);
        return x < 0 ? 0 : n - 1;
    }
    return x;
}

// ------------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_min_int(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// (value, index) arg-max: larger value wins, lower index on ties; NaN never wins
struct ArgMax {
    float v;
    int i;
};

__device__ __forceinline__ ArgMax argmax_better(ArgMax a, ArgMax b)
{
    if (b.i < 0) return a;
    if (a.i < 0) return b;
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax b{__shfl_xor_sync(0xffffffffu, a.v, o), __shfl_xor_sync(0xffffffffu, a.i, o)};
        a = argmax_better(a, b);
    }
    return a;
}

// block-wide reductions for a block of NT threads (NT multiple of 32, <= 1024)
template <int NT>
__device__ __forceinline__ float block_max(float v, float* scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = -INFINITY;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) r = fmaxf(r, scratch[w]);
    return r;
}

template <int NT>
__device__ __forceinline__ float block_sum(float v, float* scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) r += scratch[w];
    return r;
}

template <int NT>
__device__ __forceinline__ ArgMax block_argmax(ArgMax a, float* sv, int* si)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    a = warp_argmax(a);
    __syncthreads();
    if (lane == 0) {
        sv[warp] = a.v;
        si[warp] = a.i;
    }
    __syncthreads();
    ArgMax r{-INFINITY, -1};
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) r = argmax_better(r, ArgMax{sv[w], si[w]});
    return r;
}

template <int NT>
__device__ __forceinline__ int block_min_int(int v, int* scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_min_int(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    int r = INT32_MAX;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) r = min(r, scratch[w]);
    return r;
}

}  // namespace dspark

namespace dspark {

// ------------------------------------------------------------------ one block of the Markov bias
//
// bias[n] = sum_i e[i] * W[i][v0 + n] for the kNoiseBlock columns n of one vocabulary block,
// computed by a CTA of kBlockGemvThreads threads: thread t owns 8 consecutive columns
// (t % 16) and a K-slice (t / 16) of the rows, reads W with 16-byte vector loads that are all
// independent, and the 16 K-slice partials are added in a fixed order. `e` (length r) and
// `part` ([16][kNoiseBlock] floats) live in shared memory. Columns at or beyond V give 0.
constexpr int kBlockGemvThreads = 256;

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&w)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&w)[8])
{
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        w[2 * h] = __uint_as_float(u[h] << 16);
        w[2 * h + 1] = __uint_as_float(u[h] & 0xFFFF0000u);
    }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&w)[8])
{
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// Returns, in thread t < kNoiseBlock, the bias of column v0 + t. Contains __syncthreads().
template <typename T>
__device__ float block_bias(const float* e, const T* W, int V, int r, int v0, float* part)
{
    const int t = threadIdx.x;
    const bool vec = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(W) & 15u) == 0);
    if (vec) {
        const int cg = t & 15, ks = t >> 4;
        const int c0 = v0 + cg * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (c0 < V) {   // V % 8 == 0: the 8 columns are all in range or all out
            // rows in batches of 8 so that eight independent 16-byte loads are in flight
            int i = ks;
            for (; i + 7 * 16 < r; i += 8 * 16) {
                float w[8][8];
#pragma unroll
                for (int u = 0; u < 8; ++u) load8<T>(W + (size_t)(i + u * 16) * V + c0, w[u]);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float ei = e[i + u * 16];
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = fmaf(ei, w[u][j], acc[j]);
                }
            }
            for (; i < r; i += 16) {
                float w[8];
                load8<T>(W + (size_t)i * V + c0, w);
                const float ei = e[i];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(ei, w[j], acc[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) part[ks * kNoiseBlock + cg * 8 + j] = acc[j];
    } else {
        // scalar fallback: thread t < kNoiseBlock handles column v0 + t alone
        float acc = 0.f;
        if (t < kNoiseBlock && v0 + t < V)
            for (int i = 0; i < r; ++i) acc = fmaf(e[i], ld(W, (size_t)i * V + v0 + t), acc);
        if (t < kNoiseBlock) {
            part[t] = acc;
            for (int s = 1; s < 16; ++s) part[s * kNoiseBlock + t] = 0.f;
        }
    }
    __syncthreads();
    float bias = 0.f;
    if (t < kNoiseBlock)
        for (int s = 0; s < 16; ++s) bias += part[s * kNoiseBlock + t];
    return bias;
}

}  // namespace dspark
