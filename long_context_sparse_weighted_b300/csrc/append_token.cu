// Append of a decode step's new token: each sequence's newest row (position
// seq_len[b] - 1) of the raw indexer-key cache, the K cache and the V cache,
// from one packed staging row per sequence, in one launch (the decode step
// then pools the group that row completes: IndexPool's state follows every
// token, reading notes "GLM-5.3-Flash: Hybrid Attention, IndexPool, and
// Vision-in-the-Loop", section 2, sub-head "IndexPool").
#include "common.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

// One block per sequence; thread e moves 16-byte piece e of the packed row
// [k_idx (d_idx) | K (d_qk) | V (d_v)].
__global__ void __launch_bounds__(128) append_token_kernel(
    const uint16_t *__restrict__ rows, int64_t s_rows, const int32_t *__restrict__ seq_len,
    uint16_t *__restrict__ k_idx, int64_t sk_b, int d_idx, uint16_t *__restrict__ K,
    int64_t sK_b, int d_qk, uint16_t *__restrict__ V, int64_t sV_b, int d_v) {
    const int b = blockIdx.x;
    const int L = __ldg(seq_len + b);
    if (L <= 0) return;
    const int64_t t = L - 1;
    const uint16_t *src = rows + int64_t(b) * s_rows;
    const int n8 = (d_idx + d_qk + d_v) / 8;
    for (int e = threadIdx.x; e < n8; e += blockDim.x) {
        const int c = e * 8;
        uint16_t *dst;
        if (c < d_idx) dst = k_idx + int64_t(b) * sk_b + t * d_idx + c;
        else if (c < d_idx + d_qk) dst = K + int64_t(b) * sK_b + t * d_qk + (c - d_idx);
        else dst = V + int64_t(b) * sV_b + t * d_v + (c - d_idx - d_qk);
        *reinterpret_cast<uint4 *>(dst) = ld_nc16(src + c);
    }
}

}  // namespace

cudaError_t launch_append_token(const uint16_t *rows, int64_t s_rows, const int32_t *seq_len,
                                int B, uint16_t *k_idx, int64_t sk_b, int d_idx, uint16_t *K,
                                int64_t sK_b, int d_qk, uint16_t *V, int64_t sV_b, int d_v,
                                cudaStream_t st) {
    if (B == 0) return cudaSuccess;
    append_token_kernel<<<unsigned(B), 128, 0, st>>>(rows, s_rows, seq_len, k_idx, sk_b, d_idx,
                                                      K, sK_b, d_qk, V, sV_b, d_v);
    return cudaGetLastError();
}

}  // namespace lcsw
