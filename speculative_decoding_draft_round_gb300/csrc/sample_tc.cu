// sample_tc.cu -- tensor-core (tcgen05) bias contraction for the draft sampler.
#include "common.cuh"
#include "internal.h"

namespace dspark {

bool tc_supported(int, int, int, int, const void*, const void*, const void*) { return false; }
size_t tc_stats_rows(int R) { return (size_t)R; }
cudaError_t launch_draft_stats_tc(const DraftStep&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_residual_stats_tc(const VerifyParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace dspark
