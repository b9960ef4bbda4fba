// Persistent fused decode step (append -> score -> top-k -> attention).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/lcsw.h"

namespace lcsw {

bool fused_decode_supported(int B, int G_max, int H_i, int H_q, int d_qk, int d_v, int k, int P);
size_t fused_decode_ws_bytes(int B, int G_max, int H_q, int d_v, int k, int P);
cudaError_t launch_fused_decode(const lcsw_decode_args *a, void *ws, int *status,
                                cudaStream_t st);
// The same step with FP8 pooled keys (tile-major E4M3 cache kq, batch stride
// sq_b bytes; k_pooled unused).
cudaError_t launch_fused_decode_e4m3(const lcsw_decode_args *a, uint8_t *kq, int64_t sq_b,
                                     void *ws, int *status, cudaStream_t st);

// The persistent step's append, scores and selection only, writing the k
// selected groups of each sequence to idx_out [B][k] (shapes whose attention
// the persistent kernel does not cover, e.g. the MLA geometry; the fused
// region of `ws` sized for d_v = 128).
cudaError_t launch_fused_select(const lcsw_decode_args *a, int32_t *idx_out, void *ws,
                                int *status, cudaStream_t st);
// IndexCache reuse on the persistent kernel: attention over idx_in [B][k] and
// the merge of the blocks' partial states (one launch).  Supported for
// 2B <= SMs, k <= 2048, H_q a multiple of 16 up to 64.
bool reuse_decode_supported(int B, int H_q, int d_qk, int d_v, int k);
cudaError_t launch_reuse_decode(const lcsw_decode_args *a, const int32_t *idx_in, void *ws,
                                int *status, cudaStream_t st);

}  // namespace lcsw
