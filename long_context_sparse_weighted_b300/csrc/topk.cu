// Top-k groups per query row ("learned sparse selection (top 2048)",
// "G2C Brief -- GLM-5.3-Flash", DSA section; index_topk 2048 = 512 groups of
// 4 tokens).  Exact and deterministic:
//
//   * scores become order-preserving uint32 keys (-0 and +0 equal);
//   * a 3-pass radix select (11 + 11 + 10 bits, shared-memory histograms
//     with warp-aggregated increments) finds the k-th largest key K*;
//   * a final pass in ascending group order keeps every key > K* and the
//     lowest-indexed keys == K* until k are kept, writing them in ascending
//     order (block-wide prefix sums give each kept group its slot).
//
// One thread block per row: rows are independent (chunked prefill has
// thousands), and a row of up to a few hundred thousand scores stays in L2
// across the four passes.
#include "common.cuh"
#include "kernels.cuh"
#include "select_core.cuh"

namespace lcsw {
namespace {

constexpr int kTopkThreads = kSelThreads;
constexpr int kBins = 2048;

__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(
    const float *__restrict__ scores, const int32_t *__restrict__ n_valid,
    const int32_t *__restrict__ seq_len, int P, int T, int G_max, int k,
    int32_t *__restrict__ idx, const int32_t *__restrict__ row_mask) {
    if (row_mask && row_mask[blockIdx.x] == 0) return;  // row already selected elsewhere
    __shared__ unsigned hist[kBins];
    __shared__ int scratch[33];
    __shared__ int res[2];
    __shared__ int running[2];
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    const float *s = scores + row * G_max;
    int32_t *out = idx + row * k;
    int n = n_valid ? n_valid[row] : seq_len[row / T] / P;
    n = n < 0 ? 0 : (n > G_max ? G_max : n);

    if (n <= k) {  // every valid group, ascending, then padding
        for (int j = tid; j < k; j += kTopkThreads) out[j] = j < n ? j : -1;
        return;
    }

    // ---- radix select of the k-th largest key -------------------------------
    unsigned prefix = 0, mask = 0, need = unsigned(k);
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        for (int i = tid; i < kBins; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        const int n_round = (n + 31) & ~31;
        for (int i = tid; i < n_round; i += kTopkThreads) {
            unsigned key = 0;
            bool on = false;
            if (i < n) {
                key = score_key(__ldg(s + i));
                on = (key & mask) == prefix;
            }
            hist_add(hist, (key >> sh) & unsigned(nb - 1), on);
        }
        __syncthreads();
        unsigned above;
        const int d = find_digit(hist, nb, need, &above, scratch, res);
        need -= above;
        prefix |= unsigned(d) << sh;
        mask |= unsigned(nb - 1) << sh;
    }
    const unsigned kth = prefix;  // exact k-th largest key
    const unsigned take_eq = need;  // how many keys == kth to keep (lowest index first)

    // ---- ordered compaction --------------------------------------------------
    if (tid == 0) { running[0] = 0; running[1] = 0; }  // eq seen, written
    __syncthreads();
    constexpr int kItems = 4;
    for (int base = 0; base < n; base += kTopkThreads * kItems) {
        unsigned keys[kItems];
        int n_eq = 0;
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int i = base + tid * kItems + j;
            keys[j] = i < n ? score_key(__ldg(s + i)) : 0u;
            n_eq += (i < n && keys[j] == kth);
        }
        const int eq_seen = running[0], written = running[1];
        int tot_eq;
        int eq_before = eq_seen + block_exclusive_scan(n_eq, scratch, &tot_eq);
        bool sel[kItems];
        int n_sel = 0;
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int i = base + tid * kItems + j;
            bool keep = false;
            if (i < n) {
                if (keys[j] > kth) keep = true;
                else if (keys[j] == kth) keep = unsigned(eq_before++) < take_eq;
            }
            sel[j] = keep;
            n_sel += keep;
        }
        int tot_sel;
        int pos = written + block_exclusive_scan(n_sel, scratch, &tot_sel);
#pragma unroll
        for (int j = 0; j < kItems; ++j)
            if (sel[j]) {
                if (pos < k) out[pos] = base + tid * kItems + j;
                ++pos;
            }
        if (tid == 0) { running[0] = eq_seen + tot_eq; running[1] = written + tot_sel; }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_topk_rows(const float *scores, const int32_t *n_valid,
                             const int32_t *seq_len, int P, int T, int64_t rows, int G_max,
                             int k, int32_t *idx, cudaStream_t st, const int32_t *row_mask) {
    if (rows == 0) return cudaSuccess;
    if (rows > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    topk_rows_kernel<<<unsigned(rows), kTopkThreads, 0, st>>>(scores, n_valid, seq_len, P, T,
                                                              G_max, k, idx, row_mask);
    return cudaGetLastError();
}

}  // namespace lcsw
