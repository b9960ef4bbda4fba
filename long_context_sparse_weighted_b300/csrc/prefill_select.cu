// Fused top-k selection for chunked prefill: the query rows' top-k groups are
// chosen without materialising the [T][G] score matrix (top-k of the indexer
// score, "G2C Brief -- GLM-5.3-Flash", section "DSA keeps selected global
// access in eleven layers").
//
//   1. A sample pass scores a few group tiles spread over the sequence
//      (index_scores_tc.cu).  Per row, the threshold is the need-th largest
//      sampled key, need = ceil(3 kk s / n) for kk = min(k, n) of n visible
//      groups and s visible sampled groups: about 3 kk groups clear it (the
//      estimate's relative error is about 1/sqrt(need); below kk would take a
//      threefold miss).
//   2. The candidate pass keeps every visible group at or above the threshold
//      (index_scores_tc.cu).
//   3. Per row, if at least kk groups cleared the threshold (and none was
//      dropped), the kk-th largest key K* is at or above it, so every group of
//      the true top kk is a candidate: the exact top kk is selected from the
//      candidates (keys above K*, then the lowest groups equal to K*) and
//      written in ascending group order through a bitmap over the groups.
//      Otherwise the row is flagged, and the caller's fallback (dense scores,
//      then the radix top-k of topk.cu, for flagged rows only) selects it.
#include "common.cuh"
#include "kernels.cuh"
#include "select_core.cuh"

namespace lcsw {
namespace {

constexpr int kSampMax = 2048;  // sampled groups per row (16 tiles of 128)

__global__ void __launch_bounds__(kSelThreads) thresholds_kernel(
    const float *__restrict__ samp, int n_samp, const int32_t *__restrict__ n_valid, int k,
    uint32_t *__restrict__ thr, int force_fallback) {
    __shared__ unsigned keys[kSampMax];
    __shared__ unsigned hist[2048];
    __shared__ int scratch[33], res[2], cnt;
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    if (tid == 0) cnt = 0;
    __syncthreads();
    // a sampled group past the query's visible ones is -inf: key 0, below
    // every visible key, so the selection below (need <= visible count) never
    // reaches it and no compaction is needed
    const float *s = samp + row * n_samp;
    int vis = 0;
    for (int i = tid; i < n_samp; i += kSelThreads) {
        const float v = s[i];
        keys[i] = v > -INFINITY ? score_key(v) : 0u;
        vis += v > -INFINITY;
    }
    vis = __reduce_add_sync(0xffffffffu, vis);
    if ((tid & 31) == 0) atomicAdd(&cnt, vis);
    __syncthreads();
    const int s_vis = cnt, nv = max(0, n_valid[row]), kk = min(k, nv);
    uint32_t key = 0u;  // 0: every visible group is a candidate
    if (force_fallback) {
        key = 0xFFFFFFFFu;  // no candidate: every row with kk > 0 takes the fallback
    } else if (kk < nv && s_vis > 0) {
        const long long need = max(1ll, (3ll * kk * s_vis + nv - 1) / nv);
        if (need <= s_vis) {
            unsigned take;
            key = radix_select_smem(keys, n_samp, unsigned(need), hist, scratch, res, &take);
        }
    }
    if (tid == 0) thr[row] = key;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(
    const unsigned long long *__restrict__ cand, const unsigned *__restrict__ ccount, int cap,
    const int32_t *__restrict__ n_valid, int G_max, int k, int32_t *__restrict__ idx,
    int *__restrict__ fail, int *__restrict__ any_fail) {
    extern __shared__ unsigned dyn[];
    __shared__ unsigned hist[2048];
    __shared__ int scratch[33], res[2];
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    const int W = (G_max + 31) / 32;  // bitmap words
    unsigned *keys = dyn, *sel = dyn + cap, *eq = sel + W;
    int32_t *out = idx + row * k;
    const unsigned n = ccount[row];
    const int nv = min(max(0, n_valid[row]), G_max), kk = min(k, nv);
    if (kk == 0) {
        for (int i = tid; i < k; i += kSelThreads) out[i] = -1;
        return;
    }
    if (n < unsigned(kk) || n > unsigned(cap)) {  // not provably complete: fallback
        if (tid == 0) {
            fail[row] = 1;
            atomicExch(any_fail, 1);
        }
        return;
    }
    const unsigned long long *c = cand + row * cap;
    for (int i = tid; i < int(n); i += kSelThreads) keys[i] = unsigned(c[i]);
    for (int w = tid; w < W; w += kSelThreads) sel[w] = eq[w] = 0u;
    __syncthreads();
    unsigned take_eq;
    const unsigned kth = radix_select_smem(keys, int(n), unsigned(kk), hist, scratch, res, &take_eq);
    for (int i = tid; i < int(n); i += kSelThreads) {
        const unsigned key = keys[i];
        const unsigned g = unsigned(c[i] >> 32);
        if (key > kth) atomicOr(sel + (g >> 5), 1u << (g & 31));
        else if (key == kth) atomicOr(eq + (g >> 5), 1u << (g & 31));
    }
    __syncthreads();
    // the take_eq lowest groups with key K*: a prefix count over the eq bitmap
    const int per = (W + kSelThreads - 1) / kSelThreads;
    const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
    int mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(eq[w]);
    int total;
    int before = block_exclusive_scan(mine, scratch, &total);
    for (int w = w0; w < w1; ++w) {
        unsigned bits = eq[w], keep = 0u;
        while (bits && before < int(take_eq)) {
            const unsigned low = bits & (~bits + 1u);
            keep |= low;
            bits ^= low;
            ++before;
        }
        sel[w] |= keep;
    }
    __syncthreads();
    // emit the selected groups in ascending order
    mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(sel[w]);
    int pos = block_exclusive_scan(mine, scratch, &total);
    for (int w = w0; w < w1; ++w) {
        unsigned bits = sel[w];
        while (bits) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1u;
            if (LCSW_INBOUNDS(pos < k, 401)) out[pos] = w * 32 + b;
            ++pos;
        }
    }
    for (int i = kk + tid; i < k; i += kSelThreads) out[i] = -1;
}

}  // namespace

cudaError_t launch_prefill_thresholds(const float *samp, int n_samp, const int32_t *n_valid,
                                      int64_t rows, int k, uint32_t *thr, bool force_fallback,
                                      cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    if (n_samp > kSampMax || rows > 0x7FFFFFFF) return cudaErrorInvalidValue;
    thresholds_kernel<<<unsigned(rows), kSelThreads, 0, st>>>(samp, n_samp, n_valid, k, thr,
                                                              force_fallback ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_prefill_select(const unsigned long long *cand, const unsigned *ccount, int cap,
                                  const int32_t *n_valid, int64_t rows, int G_max, int k,
                                  int32_t *idx, int *fail, int *any_fail, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const int W = (G_max + 31) / 32;
    const size_t smem = (size_t(cap) + 2 * size_t(W)) * 4;
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    select_kernel<<<unsigned(rows), kSelThreads, smem, st>>>(cand, ccount, cap, n_valid, G_max, k,
                                                             idx, fail, any_fail);
    return cudaGetLastError();
}

}  // namespace lcsw
