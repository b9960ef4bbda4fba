// Block-wide radix-select helpers (blockDim.x == kSelThreads), shared by the
// per-row top-k kernel and the fused decode step.
#pragma once

#include "common.cuh"

namespace lcsw {

constexpr int kSelThreads = 512;

__device__ __forceinline__ void hist_add(unsigned *hist, unsigned bin, bool on) {
    // lanes that hit the same bin add once, by the lowest such lane
    const unsigned act = __ballot_sync(0xffffffffu, on);
    if (!on) return;
    const unsigned peers = __match_any_sync(act, bin);
    const int lane = threadIdx.x & 31;
    if ((__ffs(peers) - 1) == lane) atomicAdd(hist + bin, __popc(peers));
}

// Among the bins, find D such that (count of bins > D) < need <= (count of
// bins >= D).  Returns D; *above = count of bins > D.  512 threads x 4 bins.
__device__ __forceinline__ int find_digit(const unsigned *hist, int nbins, unsigned need, unsigned *above,
                          int *scratch, int *res) {
    const int tid = threadIdx.x;
    const int per = nbins / kSelThreads;  // 4 (11-bit) or 2 (10-bit)
    // thread tid owns bins [tid*per, tid*per+per); suffix sums over threads run
    // from the top, so scan thread (511 - tid)'s sums in increasing order.
    unsigned mine = 0;
    for (int i = 0; i < per; ++i) mine += hist[tid * per + i];
    // exclusive scan in reversed thread order
    const int rt = kSelThreads - 1 - tid;
    // scan by "rt" order: emulate with a scan over values placed at rt
    __shared__ unsigned rev[kSelThreads];
    rev[rt] = mine;
    __syncthreads();
    int tot;
    const unsigned before_rev = unsigned(block_exclusive_scan(int(rev[tid]), scratch, &tot));
    // before_rev at position tid (in reversed order) = sum over reversed
    // positions < tid = sum over threads with larger index than (511 - tid)
    __shared__ unsigned suffix[kSelThreads];
    suffix[kSelThreads - 1 - tid] = before_rev;
    __syncthreads();
    unsigned cum = suffix[tid];  // count in bins owned by threads > tid
    for (int i = per - 1; i >= 0; --i) {
        const unsigned h = hist[tid * per + i];
        if (cum < need && cum + h >= need) {
            res[0] = tid * per + i;
            res[1] = int(cum);
        }
        cum += h;
    }
    __syncthreads();
    *above = unsigned(res[1]);
    const int d = res[0];
    __syncthreads();
    return d;
}

// k-th largest of n keys held in shared memory (k <= n): returns the key K*
// and, in *take_eq, how many keys equal to K* belong to the top k (the rest of
// the top k is every key > K*).  hist: 2048 words of shared scratch.
__device__ __forceinline__ unsigned radix_select_smem(const unsigned *keys, int n, unsigned k,
                                                      unsigned *hist, int *scratch, int *res,
                                                      unsigned *take_eq) {
    const int tid = threadIdx.x;
    unsigned prefix = 0, mask = 0, need = k;
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        for (int i = tid; i < 2048; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        const int n_round = (n + 31) & ~31;
        for (int i = tid; i < n_round; i += kSelThreads) {
            unsigned key = 0;
            bool on = false;
            if (i < n) {
                key = keys[i];
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
    *take_eq = need;
    return prefix;
}

}  // namespace lcsw
