// Persistent fused decode step with FP8 (E4M3) pooled indexer keys: the host
// side of the kernel in decode_fused_kernel.cuh instantiated for the tile-major
// FP8 cache (e4m3_core.cuh).
#include "decode_fused_kernel.cuh"

namespace lcsw {

cudaError_t launch_fused_decode_e4m3(const lcsw_decode_args *a, uint8_t *kq, int64_t sq_b,
                                     void *ws, int *status, cudaStream_t st) {
    Params prm = make_params(a, ws, status);
    prm.kq = kq;
    prm.sq_b = sq_b;
    return launch_shape<true>(prm, a, st);
}

}  // namespace lcsw
