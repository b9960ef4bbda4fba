// Host side of TMA: the driver's tensor-map encoder, fetched once through the
// runtime (no link against libcuda).  nullptr when the driver lacks it.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

namespace lcsw {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
}  // namespace lcsw
