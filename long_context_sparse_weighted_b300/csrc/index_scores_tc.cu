// Indexer scores for chunked prefill as a tcgen05 GEMM (not yet enabled).
#include "common.cuh"
#include "kernels.cuh"

namespace lcsw {

bool index_scores_tc_supported(int, int, int, int, int64_t) { return false; }
cudaError_t launch_index_scores_tc(const uint16_t *, const float *, const uint16_t *, int64_t,
                                   const int32_t *, const int32_t *, int, int, int, int, int,
                                   float *, int *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace lcsw
