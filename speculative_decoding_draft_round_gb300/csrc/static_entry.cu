// static_entry.cu -- dspark_sample_block_static: the draft sampler with its scratch memory in a
// fixed device array of this library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run a round: code that
// runs inside another framework's memory pool without access to its allocator, code that must
// not grow the process's device footprint after start-up, or embedded runtimes that hand the
// library only the input and output buffers. For them this entry point keeps the sampler's
// scratch (per-step block statistics, the pick slots of the block-level draw, the conditioning
// rows, w_h . h and the status word) in one file-scope device array of
// DSPARK_STATIC_WORKSPACE_BYTES, which every GPU that loads the library holds until the process
// exits. It calls no cudaMalloc, cudaFree or allocating library routine.
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[DSPARK_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
// device address of g_static_workspace, per device; host threads may call concurrently, and
// each stores the same value, so a relaxed atomic slot is enough
std::atomic<void*> g_static_ptr[kMaxDevices] = {};

// Device address of the static array on the current device. The host-side name of a
// __device__ array is only a stand-in, so the address is looked up once per device, with that
// device current, through cudaGetSymbolAddress.
dspark_status static_workspace(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSPARK_ERR_CUDA;
    void* p = g_static_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return DSPARK_ERR_CUDA;
        g_static_ptr[dev].store(p, std::memory_order_relaxed);
    }
    *out = p;
    return DSPARK_OK;
}

}  // namespace

extern "C" dspark_status dspark_sample_block_static(const dspark_sample_args* args, void* stream)
{
    size_t need = 0;
    const dspark_status st = dspark_sample_workspace_size(args, &need);
    if (st != DSPARK_OK) return st;
    if (need > (size_t)DSPARK_STATIC_WORKSPACE_BYTES) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    void* ws = nullptr;
    const dspark_status sw = static_workspace(&ws);
    if (sw != DSPARK_OK) return sw;
    // the array keeps the previous call's contents: the status word must start at zero (the
    // other scratch regions are written before they are read within a call)
    if (cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DSPARK_ERR_CUDA;
    return dspark_sample_block(args, ws, (size_t)DSPARK_STATIC_WORKSPACE_BYTES, stream);
}

// The status word of the static array: clamped device inputs and bounded waits that ran out in
// the calls since the last check. Synchronises the stream, returns the word and clears it.
extern "C" dspark_status dspark_check_static(void* stream)
{
    void* ws = nullptr;
    const dspark_status sw = static_workspace(&ws);
    if (sw != DSPARK_OK) return sw;
    return dspark_check(ws, stream);
}
