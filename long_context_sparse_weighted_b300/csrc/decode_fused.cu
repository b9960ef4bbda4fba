// Persistent fused decode step.  (The multi-kernel sequence in lcsw_api.cu is
// used until the persistent kernel is enabled.)
#include "fused.cuh"

namespace lcsw {

bool fused_decode_supported(int, int, int, int, int, int, int, int) { return false; }
size_t fused_decode_ws_bytes(int, int, int, int, int, int) { return 0; }
cudaError_t launch_fused_decode(const lcsw_decode_args *, void *, int *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace lcsw
