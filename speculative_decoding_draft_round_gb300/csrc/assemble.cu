// assemble.cu -- the verify batch as one flat token stream.
//
// After the scheduler, the admitted prefixes of all requests are laid end to end (each
// request: its anchor, then its admitted draft tokens) with a request id and a causal
// position per token, so that a target forward can treat every token alike and read the
// sequence structure from the side tensors ("DSpark" zhongzhuzhou.org notes, physical
// execution of variable-length batches without padding).
//
// One CTA: the R run lengths keep[r] + 1 are scanned in shared memory, then every
// (request, position) slot writes its flat entry and the tail is filled with -1. The work is
// a few tens of KB of index traffic, so one SM suffices.
#include "common.cuh"
#include "internal.h"

namespace dspark {

constexpr int kAsmThreads = 1024;
constexpr int kAsmPer = DSPARK_MAX_SLOTS / kAsmThreads;   // requests per thread in the scan, at most 8

__global__ void __launch_bounds__(kAsmThreads) assemble_kernel(AssembleParams p)
{
    pdl_enter();   // keep comes from the scheduler
    __shared__ int32_t s_off[DSPARK_MAX_SLOTS + 1];
    __shared__ int32_t s_warp[kAsmThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (p.R + kAsmThreads - 1) / kAsmThreads;
    // run lengths of this thread's consecutive requests, clamped into [0, G]
    int32_t len[kAsmPer];
    int32_t run = 0;
#pragma unroll
    for (int i = 0; i < kAsmPer; ++i) {
        const int q = tid * per + i;
        int32_t k = 0;
        if (i < per && q < p.R) {
            k = p.keep[q];
            if (k < 0 || k > p.G) {
                raise_status(p.status, DSPARK_ERR_DEVICE_INPUT);
                k = k < 0 ? 0 : p.G;
            }
            k += 1;
        }
        len[i] = k;
        run += k;
    }
    // exclusive scan of the per-thread totals
    int32_t inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int32_t w = s_warp[lane];
        int32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        s_warp[lane] = wi - w;
    }
    __syncthreads();
    int32_t off = s_warp[warp] + inc - run;
#pragma unroll
    for (int i = 0; i < kAsmPer; ++i) {
        const int q = tid * per + i;
        if (i < per && q < p.R) {
            s_off[q] = off;
            p.offsets[q] = off;
            off += len[i];
        }
    }
    if (tid == kAsmThreads - 1) {
        s_off[p.R] = off;   // the last thread's running offset is the total
        p.offsets[p.R] = off;
    }
    __syncthreads();
    const int total = s_off[p.R];
    // every (request, position) slot, request-major: consecutive threads write consecutive
    // flat entries of a run
    const int G1 = p.G + 1;
    const int n = p.R * G1;
    for (int s = tid; s < n; s += kAsmThreads) {
        const int q = s / G1, j = s % G1;
        const int f = s_off[q] + j;
        if (f < s_off[q + 1]) {
            p.flat_tokens[f] = j == 0 ? p.anchor[q] : p.tokens[(size_t)q * p.G + j - 1];
            p.flat_request[f] = q;
            p.flat_position[f] = j;
        }
    }
    for (int f = total + tid; f < n; f += kAsmThreads) {
        p.flat_tokens[f] = -1;
        p.flat_request[f] = -1;
        p.flat_position[f] = -1;
    }
}

cudaError_t launch_assemble(const AssembleParams& p, cudaStream_t s)
{
    const cudaError_t e = launch_pdl(assemble_kernel, 1, kAsmThreads, 0, s, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dspark
