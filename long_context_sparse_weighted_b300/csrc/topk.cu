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
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "select_core.cuh"

namespace lcsw {
namespace {

constexpr int kTopkThreads = kSelThreads;
constexpr int kBins = 2048;

// Visible groups of a row: n_valid[row], else seq_len[row / T] / P, clamped.
__device__ __forceinline__ int row_count(const int32_t *n_valid, const int32_t *seq_len, int P,
                                         int T, int G_max, int64_t row) {
    int n = n_valid ? n_valid[row] : seq_len[row / T] / P;
    return n < 0 ? 0 : (n > G_max ? G_max : n);
}

// The whole selection of one row by one block of kTopkThreads threads.
__device__ __noinline__ void topk_row(const float *__restrict__ scores,
                                      const int32_t *__restrict__ n_valid,
                                      const int32_t *__restrict__ seq_len, int P, int T,
                                      int G_max, int k, int32_t *__restrict__ idx, int64_t row) {
    __shared__ unsigned hist[kBins];
    __shared__ int scratch[33];
    __shared__ int res[2];
    __shared__ int running[2];
    const int tid = threadIdx.x;
    const float *s = scores + row * G_max;
    int32_t *out = idx + row * k;
    const int n = row_count(n_valid, seq_len, P, T, G_max, row);

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
                if (LCSW_INBOUNDS(pos < k, 201)) out[pos] = base + tid * kItems + j;
                ++pos;
            }
        if (tid == 0) { running[0] = eq_seen + tot_eq; running[1] = written + tot_sel; }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(
    const float *__restrict__ scores, const int32_t *__restrict__ n_valid,
    const int32_t *__restrict__ seq_len, int P, int T, int G_max, int k,
    int32_t *__restrict__ idx, const int32_t *__restrict__ row_mask) {
    if (row_mask && row_mask[blockIdx.x] == 0) return;  // row already selected elsewhere
    topk_row(scores, n_valid, seq_len, P, T, G_max, k, idx, blockIdx.x);
}

// ---------------------------------------------------------------------------
// Few long rows (a decode step's one row per sequence): one block per row
// would leave all but a few SMs idle and walk the row four times from one SM.
// Instead, three launches spread each row over many blocks:
//   1. every block adds the top-11-bit digits of its slice of the row into
//      the row's histogram (shared-memory counts, then one global atomic per
//      bin);
//   2. every block finds the digit D1 holding the k-th largest key from that
//      histogram, then lists its keys with a higher digit (all selected) and
//      its keys with digit D1 (the candidates, as (key << 32) | group);
//   3. one block per row finds the k-th key K* among the candidates (radix
//      select in shared memory), marks the selected groups in a bitmap of the
//      row -- the listed ones, candidates above K*, and the lowest-indexed
//      candidates equal to K* -- and writes them in ascending order.
// A row whose candidates overflow the list takes the one-block selection in
// step 3.  Workspace per row: the histogram, two counters, the two lists.
constexpr int kWideCap = 8192;            // candidates kept per row
constexpr int kWideMaxG = 524288;         // bitmap of a row in shared memory
constexpr int kWideFilterThreads = kSelThreads;

struct WideWs {
    unsigned *hist;                // [rows][kBins]
    unsigned *cnt;                 // [rows][4]: listed above, candidates
    int32_t *above;                // [rows][k]
    unsigned long long *cand;      // [rows][kWideCap]
};

__device__ __forceinline__ void wide_slice(int n, int &lo, int &hi) {
    const int per = (n + gridDim.x - 1) / gridDim.x;
    lo = min(n, int(blockIdx.x) * per);
    hi = min(n, lo + per);
}

__global__ void __launch_bounds__(256) topk_wide_hist_kernel(
    const float *__restrict__ scores, const int32_t *__restrict__ n_valid,
    const int32_t *__restrict__ seq_len, int P, int T, int G_max, int k, WideWs w) {
    const int64_t row = blockIdx.y;
    const int n = row_count(n_valid, seq_len, P, T, G_max, row);
    if (n <= k) return;
    __shared__ unsigned h[kBins];
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
    __syncthreads();
    int lo, hi;
    wide_slice(n, lo, hi);
    const float *s = scores + row * G_max;
    constexpr int kIt = 8;  // loads in flight per thread
    for (int base = lo; base < hi; base += 256 * kIt) {
        unsigned key[kIt];
#pragma unroll
        for (int j = 0; j < kIt; ++j) {
            const int i = base + j * 256 + threadIdx.x;
            key[j] = i < hi ? score_key(__ldg(s + i)) : 0u;
        }
#pragma unroll
        for (int j = 0; j < kIt; ++j) {
            const int i = base + j * 256 + threadIdx.x;
            hist_add(h, key[j] >> 21, i < hi);
        }
    }
    __syncthreads();
    unsigned *gh = w.hist + row * kBins;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x)
        if (h[i]) atomicAdd(gh + i, h[i]);
}

__global__ void __launch_bounds__(kWideFilterThreads) topk_wide_filter_kernel(
    const float *__restrict__ scores, const int32_t *__restrict__ n_valid,
    const int32_t *__restrict__ seq_len, int P, int T, int G_max, int k, WideWs w) {
    const int64_t row = blockIdx.y;
    const int n = row_count(n_valid, seq_len, P, T, G_max, row);
    if (n <= k) return;
    __shared__ unsigned h[kBins];
    __shared__ int scratch[33];
    __shared__ int res[2];
    const unsigned *gh = w.hist + row * kBins;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = __ldcg(gh + i);
    __syncthreads();
    unsigned above;
    const unsigned d1 = unsigned(find_digit(h, kBins, unsigned(k), &above, scratch, res));
    int lo, hi;
    wide_slice(n, lo, hi);
    const float *s = scores + row * G_max;
    unsigned *cnt = w.cnt + row * 4;
    int32_t *abl = w.above + row * k;
    unsigned long long *cl = w.cand + row * kWideCap;
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    constexpr int kIt = 4;
    for (int base = lo; base < hi; base += kWideFilterThreads * kIt) {
        unsigned key[kIt];
#pragma unroll
        for (int j = 0; j < kIt; ++j) {
            const int i = base + j * kWideFilterThreads + threadIdx.x;
            key[j] = i < hi ? score_key(__ldg(s + i)) : 0u;
        }
#pragma unroll
        for (int j = 0; j < kIt; ++j) {
            const int i = base + j * kWideFilterThreads + threadIdx.x;
            const unsigned dg = key[j] >> 21;
            const bool up = i < hi && dg > d1, eq = i < hi && dg == d1;
            const unsigned mu = __ballot_sync(0xffffffffu, up);
            const unsigned me = __ballot_sync(0xffffffffu, eq);
            unsigned bu = 0, be = 0;
            if (lane == 0) {
                if (mu) bu = atomicAdd(cnt, __popc(mu));
                if (me) be = atomicAdd(cnt + 1, __popc(me));
            }
            bu = __shfl_sync(0xffffffffu, bu, 0);
            be = __shfl_sync(0xffffffffu, be, 0);
            if (up) {
                const unsigned pos = bu + __popc(mu & lt);
                if (LCSW_INBOUNDS(pos < unsigned(k), 202)) abl[pos] = i;
            }
            if (eq) {
                const unsigned pos = be + __popc(me & lt);
                if (pos < unsigned(kWideCap))
                    cl[pos] = (static_cast<unsigned long long>(key[j]) << 32) | unsigned(i);
            }
        }
    }
}

// dynamic shared memory: bitmaps sel and eqm [kWideMaxG / 32] each, then the
// candidate keys [kWideCap]
constexpr int kWideSmem = 2 * (kWideMaxG / 32) * 4 + kWideCap * 4;

__global__ void __launch_bounds__(kTopkThreads) topk_wide_final_kernel(
    const float *__restrict__ scores, const int32_t *__restrict__ n_valid,
    const int32_t *__restrict__ seq_len, int P, int T, int G_max, int k,
    int32_t *__restrict__ idx, WideWs w) {
    extern __shared__ __align__(16) unsigned char dsm[];
    unsigned *sel = reinterpret_cast<unsigned *>(dsm);
    unsigned *eqm = sel + kWideMaxG / 32;
    unsigned *ckey = eqm + kWideMaxG / 32;
    __shared__ unsigned hist[kBins];
    __shared__ int scratch[33];
    __shared__ int res[2];
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    const int n = row_count(n_valid, seq_len, P, T, G_max, row);
    int32_t *out = idx + row * k;
    if (n <= k) {
        for (int j = tid; j < k; j += kTopkThreads) out[j] = j < n ? j : -1;
        return;
    }
    const unsigned *cnt = w.cnt + row * 4;
    const int n_up = int(__ldcg(cnt)), m = int(__ldcg(cnt + 1));
    if (m > kWideCap || n_up >= k) {  // (the second cannot happen: D1 holds the k-th key)
        topk_row(scores, n_valid, seq_len, P, T, G_max, k, idx, row);
        return;
    }
    const int nw = (n + 31) / 32;
    for (int i = tid; i < nw; i += kTopkThreads) sel[i] = eqm[i] = 0u;
    const unsigned long long *cl = w.cand + row * kWideCap;
    for (int i = tid; i < m; i += kTopkThreads) ckey[i] = unsigned(__ldcg(cl + i) >> 32);
    __syncthreads();
    unsigned take_eq;
    const unsigned kth = radix_select_smem(ckey, m, unsigned(k - n_up), hist, scratch, res,
                                           &take_eq);
    const int32_t *abl = w.above + row * k;
    for (int i = tid; i < n_up; i += kTopkThreads) {
        const int g = __ldcg(abl + i);
        if (LCSW_INBOUNDS(g >= 0 && g < n, 204)) atomicOr(sel + (g >> 5), 1u << (g & 31));
    }
    for (int i = tid; i < m; i += kTopkThreads) {
        const unsigned long long e = __ldcg(cl + i);
        const unsigned key = unsigned(e >> 32);
        const int g = int(e & 0xFFFFFFFFu);
        if (!LCSW_INBOUNDS(g >= 0 && g < n, 204)) continue;
        if (key > kth) atomicOr(sel + (g >> 5), 1u << (g & 31));
        else if (key == kth) atomicOr(eqm + (g >> 5), 1u << (g & 31));
    }
    __syncthreads();
    // the take_eq lowest-indexed keys equal to K*, then every selected group
    // in ascending order: thread t owns words [t*wpt, (t+1)*wpt)
    const int wpt = (nw + kTopkThreads - 1) / kTopkThreads;
    const int w0 = min(nw, tid * wpt), w1 = min(nw, w0 + wpt);
    int ce = 0;
    for (int i = w0; i < w1; ++i) ce += __popc(eqm[i]);
    int tot;
    int eq_before = block_exclusive_scan(ce, scratch, &tot);
    for (int i = w0; i < w1; ++i) {
        unsigned e = eqm[i];
        while (e) {
            const int b = __ffs(e) - 1;
            e &= e - 1;
            if (unsigned(eq_before++) < take_eq) sel[i] |= 1u << b;
        }
    }
    int cs = 0;
    for (int i = w0; i < w1; ++i) cs += __popc(sel[i]);
    int pos = block_exclusive_scan(cs, scratch, &tot);
    for (int i = w0; i < w1; ++i) {
        unsigned v = sel[i];
        while (v) {
            const int b = __ffs(v) - 1;
            v &= v - 1;
            if (LCSW_INBOUNDS(pos < k, 203)) out[pos] = i * 32 + b;
            ++pos;
        }
    }
}

}  // namespace

bool topk_wide_supported(int64_t rows, int G_max, int k) {
    return rows >= 1 && rows <= 32 && G_max >= 16384 && G_max <= kWideMaxG && k >= 1 &&
           k <= G_max;
}

size_t topk_wide_ws_bytes(int64_t rows, int G_max, int k) {
    if (!topk_wide_supported(rows, G_max, k)) return 0;
    auto r = [](size_t b) { return (b + 255) & ~size_t(255); };
    return r(size_t(rows) * (kBins + 4) * 4) + r(size_t(rows) * k * 4) +
           r(size_t(rows) * kWideCap * 8);
}

cudaError_t launch_topk_rows_wide(const float *scores, const int32_t *n_valid,
                                  const int32_t *seq_len, int P, int T, int64_t rows, int G_max,
                                  int k, int32_t *idx, void *ws, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    auto r = [](size_t b) { return (b + 255) & ~size_t(255); };
    char *base = static_cast<char *>(ws);
    WideWs w;
    w.hist = reinterpret_cast<unsigned *>(base);
    w.cnt = w.hist + size_t(rows) * kBins;
    w.above = reinterpret_cast<int32_t *>(base + r(size_t(rows) * (kBins + 4) * 4));
    w.cand = reinterpret_cast<unsigned long long *>(base + r(size_t(rows) * (kBins + 4) * 4) +
                                                    r(size_t(rows) * k * 4));
    cudaError_t e = cudaMemsetAsync(w.hist, 0, size_t(rows) * (kBins + 4) * 4, st);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // about two blocks per SM over all rows, at least 1,024 scores a block
    int nb = int(std::max<int64_t>(1, 2 * sms / rows));
    nb = std::min(nb, std::max(1, G_max / 1024));
    topk_wide_hist_kernel<<<dim3(nb, unsigned(rows)), 256, 0, st>>>(scores, n_valid, seq_len, P,
                                                                     T, G_max, k, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_wide_filter_kernel<<<dim3(nb, unsigned(rows)), kWideFilterThreads, 0, st>>>(
        scores, n_valid, seq_len, P, T, G_max, k, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk_wide_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kWideSmem);
    if (e != cudaSuccess) return e;
    topk_wide_final_kernel<<<unsigned(rows), kTopkThreads, kWideSmem, st>>>(
        scores, n_valid, seq_len, P, T, G_max, k, idx, w);
    return cudaGetLastError();
}

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
