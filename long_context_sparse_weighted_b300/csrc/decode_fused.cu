// Persistent fused decode step: [append] -> indexer scores -> top-k groups ->
// sparse attention -> split-K combine, in one cooperative launch of one
// thread block per SM (the DSA retrieval chain of "G2C Brief --
// GLM-5.3-Flash", section "DSA keeps selected global access in eleven
// layers"; IndexPool from the reading notes, section 2).
//
// Work split.  Every sequence b gets a contiguous set of n_b >= 1 blocks,
// proportional to its number of pooled groups G_b; block j of the set owns a
// contiguous chunk of 16-group tiles.  All cross-block waits are per sequence
// and bounded (clock64 budget; on expiry the block records LCSW_ERR_TIMEOUT in
// the workspace status word, raises an abort flag that every other wait
// honours, and returns).
//
// Phase 1 (HBM stream).  Warps stream their tiles' pooled keys straight into
// mma.sync A fragments (the k-permuted layout of index_scores.cu, one tile of
// prefetch in flight per warp), compute the scores, keep them in shared
// memory, and count them in a 65536-bin histogram of the top 16 bits of the
// order-preserving score key (two 16-bit counters per shared word).  The block
// that owns the group completed by the newest token pools it first (the exact
// arithmetic of the pooling kernel) and scores that fresh key.
//
// Selection.  Each block adds its histogram to the sequence's global one, waits
// until half of the sequence's blocks have done so, and reads a lower bound LB
// on the k-th largest key off whatever the global histogram holds: any subset
// of the scores has a k-th largest no larger than the full set's, so every
// member of the true top k has its 16-bit key prefix >= LB.  The block writes
// its keys with prefix >= LB, in ascending group order, to its segment of the
// candidate list and arrives at barrier A.  After A, if the candidates of the
// sequence fit in shared memory, every block that has attention work loads
// them (in ascending group order), radix-selects the exact k-th key K*, and
// keeps keys > K* plus the lowest-indexed keys == K* -- the exact top k,
// ascending.  Otherwise all blocks of the sequence run the exact multi-pass
// selection over their own scores (full level-1 histogram, a level-2
// histogram of the low 16 bits, per-block counts for the tie rule and the
// output offsets), with three more sequence barriers.
//
// Attention.  The selected groups are split into S_b slices of >= 64 tokens
// (x head groups of 64 heads); slice items go round-robin to the sequence's
// blocks, which gather K/V rows with cp.async into double-buffered shared
// memory and run the mma.sync online-softmax tile of attn_core.cuh.  With
// S_b > 1 the partial (m, l, o) states meet at a sequence barrier and the
// participating blocks each merge a subset of the heads.
#include "attn_core.cuh"
#include "common.cuh"
#include "fused.cuh"
#include "kernels.cuh"
#include "pool_core.cuh"
#include "select_core.cuh"

namespace lcsw {
namespace {

constexpr int kThreads = kSelThreads;  // 512
constexpr int kWarps = kThreads / 32;
constexpr int kFine = 65536, kCoarse = 256, kHistWords = kFine + kCoarse;
constexpr int kChunkCap = 12288;   // scores of a block's chunk kept in shared memory
constexpr int kSelCap = 8192;      // candidates selected in shared memory
constexpr int kMaxK = 2048;        // selected groups per sequence
constexpr int kCtlWords = 32;      // control words per sequence
constexpr int kMaxCtas = 160;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// control words (per sequence): arrival counters of the step's sync points,
// reset to zero by the last block to leave the kernel
constexpr int kFlushed = 0, kCands = 1, kSlowB = 2, kSlowC = 3, kSlowD = 4, kSlowE = 5,
              kAtt = 6, kDepart = 7, kNumCounters = 8;

// shared memory map (bytes)
constexpr int kU = 0;                                 // 128 KB union region
constexpr int kUBytes = kFine * 2;                    // 16-bit counters
constexpr int kSelG = kU;                             // selected groups [kMaxK]
constexpr int kCandKey = kU + kMaxK * 4;              // [kSelCap]
constexpr int kCandG = kCandKey + kSelCap * 4;        // [kSelCap]
constexpr int kRHist = kCandG + kSelCap * 4;          // [2048]
constexpr int kKV = kU + kMaxK * 4;                   // attention K/V buffers
constexpr int kState = kU + kMaxK * 4;                // merge state (after the chunks)
constexpr int kScores = kU + kUBytes;                 // [kChunkCap] floats
constexpr int kQ = kScores + kChunkCap * 4;           // Q tile [64][QP]

struct Params {
    const uint16_t *q_idx;
    const float *w_head;
    uint16_t *k_pooled;
    int64_t sp_b;
    const uint16_t *k_idx;
    int64_t sk_b;
    const float *pool_w;
    int64_t sw_b;
    const uint16_t *q;
    const uint16_t *K;
    int64_t sK_b;
    const uint16_t *V;
    int64_t sV_b;
    const int32_t *seq_len;
    int B, G_max, H_i, P, k, H_q, S_max, force_slow, skip_arrive;
    float scale_log2;
    uint16_t *out;
    float *lse;
    int32_t *idx_out;
    float *scores_out;
    // workspace
    unsigned *ctl;        // [B][kCtlWords]
    unsigned *hist;       // [B][2][kHistWords]: level 1, level 2 (zero between calls)
    unsigned *cand_key;   // [B][G_max]
    int32_t *cand_g;      // [B][G_max]
    float *gscore;        // [B][G_max] spill of scores past kChunkCap
    unsigned *cta_cnt;    // [3][ncta]: candidate count, > K*, == K*
    int32_t *idx_ws;      // [B][k]
    float *part_o;        // [B][S_max][H_q][d_v]
    float2 *part_ml;      // [B][S_max][H_q]
    int *status;          // ws word 0
    int *abort_flag;      // ws word 1
};

// ------------------------------------------------------------ phase timers -
// Built with -DLCSW_PHASE_TIMERS, block 0 thread 0 of every block records the
// first and last %globaltimer reading of each phase mark across blocks.
#ifdef LCSW_PHASE_TIMERS
__device__ unsigned long long g_phase_first[16];
__device__ unsigned long long g_phase_last[16];
__device__ unsigned g_dbg_max[4];
#define DBG_MAX(i, v)                                   \
    do {                                                \
        if (threadIdx.x == 0) atomicMax(&g_dbg_max[i], unsigned(v)); \
    } while (0)
#define PHASE_MARK(i)                                                           \
    do {                                                                        \
        if (threadIdx.x == 0) {                                                 \
            unsigned long long t_;                                              \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));              \
            atomicMin(&g_phase_first[i], t_);                                   \
            atomicMax(&g_phase_last[i], t_);                                    \
        }                                                                       \
    } while (0)
#else
#define PHASE_MARK(i) \
    do {              \
    } while (0)
#define DBG_MAX(i, v) \
    do {              \
    } while (0)
#endif

// ------------------------------------------------------------ coherence ----

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned ld_cg(const unsigned *p) {
    unsigned v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_cg_f(const float *p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_cg4(const void *p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ bool aborted(const int *f) {
    return *reinterpret_cast<const volatile int *>(f) != 0;
}
__device__ void raise_timeout(const Params &p, int where) {
    atomicCAS(p.status, 0, int(LCSW_ERR_TIMEOUT) * 256 + where);
    atomicExch(p.abort_flag, 1);
}

// Sync points are arrival counters: a block makes its global writes visible
// (fence) and adds 1 without waiting for the result; a block that needs the
// others' writes polls until the count reaches its target (bounded wait).
__device__ __forceinline__ void arrive(unsigned *cnt) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(cnt, 1u);  // result unused: a fire-and-forget reduction
}

__device__ bool wait_count(const Params &p, const unsigned *cnt, unsigned target, int where,
                           int *s_ok) {
    if (threadIdx.x == 0) {
        int ok = 1;
        const long long t0 = clock64();
        while (ld_acquire(cnt) < target) {
            if (aborted(p.abort_flag)) { ok = 0; break; }
            if (clock64() - t0 > kSpinBudget) { raise_timeout(p, where); ok = 0; break; }
            __nanosleep(20);
        }
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

// Find, in a 256-bin slice of a global histogram (read at L2), the bin where
// the count from the top reaches `need`.  One warp.  Returns the bin
// (0..255) or -1 if the slice holds fewer than `need`; *above = count of bins
// above it.
__device__ __forceinline__ int warp_find_from_top(const unsigned *bins, unsigned need,
                                                  unsigned *above) {
    const int lane = threadIdx.x & 31;
    const uint4 a = ld_cg4(bins + lane * 8), b = ld_cg4(bins + lane * 8 + 4);
    const unsigned v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    unsigned mine = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mine += v[i];
    unsigned suf = mine;  // inclusive suffix over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += y;
    }
    const unsigned excl = suf - mine;  // lanes above
    const bool here = excl < need && suf >= need;
    const unsigned bal = __ballot_sync(0xffffffffu, here);
    if (bal == 0) return -1;
    const int src = __ffs(bal) - 1;
    int bin = -1;
    unsigned ab = 0;
    if (lane == src) {
        unsigned cum = excl;
        for (int i = 7; i >= 0; --i) {
            if (cum + v[i] >= need) { bin = lane * 8 + i; ab = cum; break; }
            cum += v[i];
        }
    }
    bin = __shfl_sync(0xffffffffu, bin, src);
    *above = __shfl_sync(0xffffffffu, ab, src);
    return bin;
}

// The same search over shared memory: 256 u32 counts, or (pairs) 128 words
// of two 16-bit counts.
__device__ __forceinline__ int smem_find_from_top(const unsigned *bins, unsigned need,
                                                  unsigned *above, bool pairs) {
    const int lane = threadIdx.x & 31;
    unsigned v[8];
    if (pairs) {
        const uint4 a = *reinterpret_cast<const uint4 *>(bins + lane * 4);
        const unsigned w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = w[i] & 0xFFFFu;
            v[2 * i + 1] = w[i] >> 16;
        }
    } else {
        const uint4 a = *reinterpret_cast<const uint4 *>(bins + lane * 8);
        const uint4 b = *reinterpret_cast<const uint4 *>(bins + lane * 8 + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    unsigned mine = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mine += v[i];
    unsigned suf = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += y;
    }
    const unsigned excl = suf - mine;
    const unsigned bal = __ballot_sync(0xffffffffu, excl < need && suf >= need);
    if (bal == 0) return -1;
    const int src = __ffs(bal) - 1;
    int bin = -1;
    unsigned ab = 0;
    if (lane == src) {
        unsigned cum = excl;
        for (int i = 7; i >= 0; --i) {
            if (cum + v[i] >= need) { bin = lane * 8 + i; ab = cum; break; }
            cum += v[i];
        }
    }
    bin = __shfl_sync(0xffffffffu, bin, src);
    *above = __shfl_sync(0xffffffffu, ab, src);
    return bin;
}

// 16-bit key prefix whose bin holds the need-th largest entry of a
// (coarse, fine) global histogram.  Returns -1 if it holds fewer than need;
// with `exact` false an inconsistent snapshot falls back to the coarse bin.
__device__ __forceinline__ int hist_walk(const unsigned *h, unsigned need, bool exact,
                                         unsigned *above) {
    unsigned ab_c = 0, ab_f = 0;
    const int c = warp_find_from_top(h + kFine, need, &ab_c);
    if (c < 0) return -1;
    const int f = warp_find_from_top(h + c * 256, need - ab_c, &ab_f);
    if (f < 0) {
        *above = ab_c;
        return exact ? -1 : c * 256;
    }
    *above = ab_c + ab_f;
    return c * 256 + f;
}

// Add the block's shared 16-bit-pair histogram into a global (fine, coarse)
// histogram.  Warp w, pass i covers fine bins [256*(w + 16 i), +256) = one
// coarse bin.
__device__ __forceinline__ void flush_hist(const unsigned *h16, unsigned *g) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = 0; i < kCoarse / kWarps; ++i) {
        const int cb = warp + kWarps * i;
        const uint4 w = *reinterpret_cast<const uint4 *>(h16 + cb * 128 + lane * 4);
        const unsigned ws[4] = {w.x, w.y, w.z, w.w};
        unsigned sum = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const unsigned lo = ws[e] & 0xFFFFu, hi = ws[e] >> 16;
            const int bin = cb * 256 + (lane * 4 + e) * 2;
            if (lo) atomicAdd(g + bin, lo);
            if (hi) atomicAdd(g + bin + 1, hi);
            sum += lo + hi;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0 && sum) atomicAdd(g + kFine + cb, sum);
    }
}

__device__ __forceinline__ void clear_smem(unsigned char *base, int bytes) {
    for (int i = threadIdx.x * 16; i < bytes; i += kThreads * 16)
        *reinterpret_cast<uint4 *>(base + i) = make_uint4(0, 0, 0, 0);
}

template <int NT, int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1) fused_decode_kernel(const Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned *h16 = reinterpret_cast<unsigned *>(smem + kU);
    float *sscore = reinterpret_cast<float *>(smem + kScores);
    constexpr int QP = DQK + 8, VP = DV + 8;
    uint16_t *sq = reinterpret_cast<uint16_t *>(smem + kQ);
    constexpr int kMisc = kQ + 64 * QP * 2;
    uint16_t *newkey = reinterpret_cast<uint16_t *>(smem + kMisc);   // [64], 16-byte aligned
    unsigned *ccoarse = reinterpret_cast<unsigned *>(smem + kMisc + 128);  // [kCoarse]
    int *cta_begin = reinterpret_cast<int *>(smem + kMisc + 128 + kCoarse * 4);  // [kMaxCtas + 1]
    int *offs = cta_begin + kMaxCtas + 1;                            // [kMaxCtas + 1]
    int *sv = offs + kMaxCtas + 1;                                   // scalars [64]
    int *scratch = sv + 64;                                          // [40]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x, ncta = gridDim.x;
    const int B = p.B, P = p.P;
    PHASE_MARK(0);
    if (aborted(p.abort_flag)) return;

    // ---- roles: blocks per sequence, proportional to its groups ------------
    if (warp == 0) {
        // prefix sums of G_b over b (B <= ncta <= kMaxCtas), 5 per lane
        unsigned run = 0;
        for (int base = 0; base < B; base += 32) {
            const int b = base + lane;
            unsigned g = 0;
            if (b < B) {
                int G = __ldg(p.seq_len + b) / P;
                G = G < 0 ? 0 : (G > p.G_max ? p.G_max : G);
                g = unsigned(G);
            }
            unsigned x = g;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (b < B) offs[b] = int(run + x - g);  // exclusive prefix
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) sv[0] = int(run);
    }
    __syncthreads();
    {
        const long long total = sv[0] > 0 ? sv[0] : 1;
        const long long R = ncta - B;
        for (int b = tid; b <= B; b += kThreads)
            cta_begin[b] = b == B ? ncta : b + int(R * (long long)offs[b] / total);
    }
    __syncthreads();
    int b = 0;
    {
        // largest b with cta_begin[b] <= cta
        for (int i = tid; i < B; i += kThreads)
            if (cta_begin[i] <= cta && cta < cta_begin[i + 1]) sv[1] = i;
        __syncthreads();
        b = sv[1];
    }
    const int cb0 = cta_begin[b];
    const int n_b = cta_begin[b + 1] - cb0;
    const int j = cta - cb0;
    const int L_b = __ldg(p.seq_len + b);
    int G_b = L_b / P;
    G_b = G_b < 0 ? 0 : (G_b > p.G_max ? p.G_max : G_b);
    const int tiles_b = (G_b + 15) / 16;
    auto chunk_lo = [&](int jj) { return 16 * int((long long)tiles_b * jj / n_b); };
    const int g_lo = chunk_lo(j);
    const int g_hi = min(G_b, chunk_lo(j + 1));
    const int nloc = g_hi > g_lo ? g_hi - g_lo : 0;
    const int k_b = min(p.k, G_b);
    unsigned *ctl = p.ctl + size_t(b) * kCtlWords;
    unsigned *hist1 = p.hist + size_t(b) * 2 * kHistWords;
    unsigned *hist2 = hist1 + kHistWords;
    const int64_t seg = int64_t(b) * p.G_max;
    int *s_ok = sv + 2;

    // attention items of this sequence
    const int HGs = (p.H_q + 63) / 64;
    int S_b = (k_b * P + kChunk - 1) / kChunk;
    S_b = max(1, min(S_b, min(n_b, p.S_max)));
    const int items = S_b * HGs;
    const int n_att = min(items, n_b);
    const bool has_items = j < n_att;

    PHASE_MARK(11);
    // ---- append: pool the group the newest token completes ------------------
    int g_new = -1;
    if (p.k_idx && G_b > 0 && L_b % P == 0) g_new = G_b - 1;
    const bool own_new = g_new >= g_lo && g_new < g_hi;
    if (own_new && tid < 8) {
        const uint16_t *src = p.k_idx + int64_t(b) * p.sk_b + int64_t(g_new) * P * 64 + tid * 8;
        const float *wp = p.pool_w + int64_t(b) * p.sw_b + int64_t(g_new) * P;
        uint4 o;
#define LCSW_APPEND(PP)                                                        \
    {                                                                          \
        uint4 rows[PP];                                                        \
        float a[PP];                                                           \
        for (int jj = 0; jj < PP; ++jj) {                                      \
            rows[jj] = ld_nc16(src + jj * 64);                                 \
            a[jj] = __ldg(wp + jj);                                            \
        }                                                                      \
        o = pool_chunk<PP>(a, rows);                                           \
    }
        if (P == 1) LCSW_APPEND(1)
        else if (P == 2) LCSW_APPEND(2)
        else if (P == 4) LCSW_APPEND(4)
        else LCSW_APPEND(8)
#undef LCSW_APPEND
        *reinterpret_cast<uint4 *>(newkey + tid * 8) = o;
        *reinterpret_cast<uint4 *>(p.k_pooled + int64_t(b) * p.sp_b + int64_t(g_new) * 64 +
                                   tid * 8) = o;
    }

    // ---- query fragments of the indexer ------------------------------------
    const int r = lane >> 2, c = lane & 3;
    uint32_t bq[NT][4][2];
    float wv[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int head = nt * 8 + r;
        uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
        if (head < p.H_i) {
            const uint16_t *qp = p.q_idx + (int64_t(b) * p.H_i + head) * 64;
            h0 = ld_nc16(qp + 8 * c);
            h1 = ld_nc16(qp + 32 + 8 * c);
        }
        bq[nt][0][0] = h0.x; bq[nt][0][1] = h0.y;
        bq[nt][1][0] = h0.z; bq[nt][1][1] = h0.w;
        bq[nt][2][0] = h1.x; bq[nt][2][1] = h1.y;
        bq[nt][3][0] = h1.z; bq[nt][3][1] = h1.w;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = nt * 8 + 2 * c + e;
            wv[nt][e] = h < p.H_i ? __ldg(p.w_head + int64_t(b) * p.H_i + h) : 0.f;
        }
    }
    clear_smem(smem + kU, kUBytes);
    __syncthreads();
    PHASE_MARK(12);

    // ---- phase 1: stream pooled keys, score, histogram -----------------------
    const uint16_t *kb = p.k_pooled + int64_t(b) * p.sp_b;
    const int n_tiles = (nloc + 15) / 16;
    auto load_tile = [&](int t, uint4 (&A)[4]) {
        const int ga = g_lo + t * 16 + r, gb = ga + 8;
        const uint4 z = make_uint4(0, 0, 0, 0);
        A[0] = A[1] = A[2] = A[3] = z;
        if (ga < g_hi) {
            if (ga == g_new) {
                A[0] = *reinterpret_cast<const uint4 *>(newkey + 8 * c);
                A[1] = *reinterpret_cast<const uint4 *>(newkey + 32 + 8 * c);
            } else {
                A[0] = ld_stream16(kb + int64_t(ga) * 64 + 8 * c);
                A[1] = ld_stream16(kb + int64_t(ga) * 64 + 32 + 8 * c);
            }
        }
        if (gb < g_hi) {
            if (gb == g_new) {
                A[2] = *reinterpret_cast<const uint4 *>(newkey + 8 * c);
                A[3] = *reinterpret_cast<const uint4 *>(newkey + 32 + 8 * c);
            } else {
                A[2] = ld_stream16(kb + int64_t(gb) * 64 + 8 * c);
                A[3] = ld_stream16(kb + int64_t(gb) * 64 + 32 + 8 * c);
            }
        }
    };
    auto score_tile = [&](int t, const uint4 (&A)[4]) {
        const uint32_t A0[4] = {A[0].x, A[0].z, A[1].x, A[1].z};
        const uint32_t A2[4] = {A[0].y, A[0].w, A[1].y, A[1].w};
        const uint32_t A1[4] = {A[2].x, A[2].z, A[3].x, A[3].z};
        const uint32_t A3[4] = {A[2].y, A[2].w, A[3].y, A[3].w};
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma_bf16_16816(acc[nt], A0[s], A1[s], A2[s], A3[s], bq[nt][s][0], bq[nt][s][1]);
        float pa = 0.f, pb = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            pa = __fadd_rn(pa, __fmul_rn(wv[nt][0], fmaxf(acc[nt][0], 0.f)));
            pa = __fadd_rn(pa, __fmul_rn(wv[nt][1], fmaxf(acc[nt][1], 0.f)));
            pb = __fadd_rn(pb, __fmul_rn(wv[nt][0], fmaxf(acc[nt][2], 0.f)));
            pb = __fadd_rn(pb, __fmul_rn(wv[nt][1], fmaxf(acc[nt][3], 0.f)));
        }
        pa = __fadd_rn(pa, __shfl_xor_sync(0xffffffffu, pa, 1));
        pb = __fadd_rn(pb, __shfl_xor_sync(0xffffffffu, pb, 1));
        pa = __fadd_rn(pa, __shfl_xor_sync(0xffffffffu, pa, 2));
        pb = __fadd_rn(pb, __shfl_xor_sync(0xffffffffu, pb, 2));
        if (c < 2) {
            const int li = t * 16 + r + 8 * c;
            const float sc = __fadd_rn(c == 0 ? pa : pb, 0.0f);
            if (g_lo + li < g_hi) {
                if (li < kChunkCap) sscore[li] = sc;
                else p.gscore[seg + g_lo + li] = sc;
                if (p.scores_out) p.scores_out[seg + g_lo + li] = sc;
                const unsigned bin = score_key(sc) >> 16;
                atomicAdd(h16 + (bin >> 1), (bin & 1u) ? 0x10000u : 1u);
            }
        }
    };
    {
        // warp w scores tiles w, w+16, w+32, ...: two per iteration, with the
        // next two already in flight
        int t = warp;
        uint4 c0[4], c1[4];
        if (t < n_tiles) load_tile(t, c0);
        if (t + kWarps < n_tiles) load_tile(t + kWarps, c1);
        for (; t < n_tiles; t += 2 * kWarps) {
            uint4 n0[4], n1[4];
            const bool m0 = t + 2 * kWarps < n_tiles, m1 = t + 3 * kWarps < n_tiles;
            if (m0) load_tile(t + 2 * kWarps, n0);
            if (m1) load_tile(t + 3 * kWarps, n1);
            score_tile(t, c0);
            if (t + kWarps < n_tiles) score_tile(t + kWarps, c1);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (m0) c0[i] = n0[i];
                if (m1) c1[i] = n1[i];
            }
        }
    }
    if (p.scores_out && j == 0)  // -inf past the last complete group: the full row
        for (int g = G_b + tid; g < p.G_max; g += kThreads) p.scores_out[seg + g] = -INFINITY;
    __syncthreads();
    for (int cbin = warp; cbin < kCoarse; cbin += kWarps) {
        const uint4 w = *reinterpret_cast<const uint4 *>(h16 + cbin * 128 + lane * 4);
        unsigned s = (w.x & 0xFFFFu) + (w.x >> 16) + (w.y & 0xFFFFu) + (w.y >> 16) +
                     (w.z & 0xFFFFu) + (w.z >> 16) + (w.w & 0xFFFFu) + (w.w >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) ccoarse[cbin] = s;
    }
    __syncthreads();
    PHASE_MARK(1);
    auto score_at = [&](int li) -> float {
        return li < kChunkCap ? sscore[li] : ld_cg_f(p.gscore + seg + g_lo + li);
    };

    // ---- flush histogram, lower bound from >= half of the sequence ----------
    // Flush only the block's m largest keys (by 16-bit prefix bin): the union
    // over blocks of local top-m sets is a subset of all keys, so the k-th
    // largest key it gives is still a lower bound, and with m a few times
    // k / n_b it is usually the exact k-th -- at a few atomics per block.
    if (warp == 0 && nloc > 0 && k_b > 0) {
        const int m = min(nloc, 4 * ((k_b + n_b - 1) / n_b) + 8);
        unsigned ab_c = 0, ab_f = 0;
        const int cm = smem_find_from_top(ccoarse, unsigned(m), &ab_c, false);
        const int fm = cm < 0 ? 0 : smem_find_from_top(h16 + cm * 128, unsigned(m) - ab_c, &ab_f, true);
        if (lane == 0) { sv[16] = cm; sv[17] = fm; }
    }
    __syncthreads();
    // mode 0: add the top-m bins; 1: add the other bins; 2: zero the top-m bins
    auto level1_bins = [&](int mode) {
        if (nloc == 0 || k_b == 0) return;
        const int cm = sv[16] < 0 ? 0 : sv[16], fm = sv[16] < 0 ? 0 : sv[17];
        const int c_stop = mode == 1 ? 0 : cm;
        for (int cbin = kCoarse - 1 - warp; cbin >= c_stop; cbin -= kWarps) {
            if (ccoarse[cbin] == 0) continue;
            if (mode == 1 && cbin > cm) continue;
            const uint4 w = *reinterpret_cast<const uint4 *>(h16 + cbin * 128 + lane * 4);
            const unsigned ws[4] = {w.x, w.y, w.z, w.w};
            unsigned sum = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const unsigned cnt = hf ? ws[e] >> 16 : ws[e] & 0xFFFFu;
                    const int fb = (lane * 4 + e) * 2 + hf;
                    const bool top = cbin > cm || (cbin == cm && fb >= fm);
                    if (cnt && top == (mode != 1)) {
                        if (mode == 2) hist1[cbin * 256 + fb] = 0u;
                        else atomicAdd(hist1 + cbin * 256 + fb, cnt);
                        sum += cnt;
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0 && sum) {
                if (mode == 2) hist1[kFine + cbin] = 0u;
                else atomicAdd(hist1 + kFine + cbin, sum);
            }
        }
    };
    level1_bins(0);
    arrive(ctl + kFlushed);
    PHASE_MARK(2);
    if (tid == 0) {
        const unsigned half = unsigned(n_b + 1) / 2;
        const long long t0 = clock64();
        int ok = 1;
        while (ld_acquire(ctl + kFlushed) < half) {
            if (aborted(p.abort_flag)) { ok = 0; break; }
            if (clock64() - t0 > kSpinBudget) { raise_timeout(p, 1); ok = 0; break; }
            __nanosleep(20);
        }
        *s_ok = ok;
    }
    // Q tile of the first attention item (prefetch; waited before attention)
    if (has_items && S_b * HGs > 0) {
        const int hg = (j % items) / S_b;
        const int h0 = hg * 64, HG = min(64, p.H_q - h0);
        const uint16_t *qrow = p.q + (int64_t(b) * p.H_q + h0) * DQK;
        for (int e = tid; e < HG * (DQK / 8); e += kThreads) {
            const int h = e / (DQK / 8), c8 = e % (DQK / 8);
            cp_async16(smem_u32(sq + h * QP + c8 * 8), qrow + int64_t(h) * DQK + c8 * 8, 16);
        }
        cp_async_commit();
    }
    __syncthreads();
    PHASE_MARK(3);
    if (!*s_ok) { cp_async_wait<0>(); return; }
    if (warp == 0) {
        unsigned above = 0;
        int lb = hist_walk(hist1, unsigned(k_b), false, &above);
        if (lane == 0) sv[3] = lb < 0 ? 0 : lb;
    }
    __syncthreads();
    const unsigned lb_bin = unsigned(sv[3]);
    PHASE_MARK(4);

    // ---- candidates: keys with prefix >= lb, ascending, to the segment ------
    {
        const int per = (nloc + kThreads - 1) / kThreads;
        const int i0 = min(nloc, tid * per), i1 = min(nloc, i0 + per);
        int cnt = 0;
        for (int i = i0; i < i1; ++i) cnt += (score_key(score_at(i)) >> 16) >= lb_bin;
        int total;
        int pos = block_exclusive_scan(cnt, scratch, &total);
        unsigned *ck = p.cand_key + seg + g_lo;
        int32_t *cg = p.cand_g + seg + g_lo;
        for (int i = i0; i < i1; ++i) {
            const unsigned key = score_key(score_at(i));
            if ((key >> 16) >= lb_bin) {
                ck[pos] = key;
                cg[pos] = g_lo + i;
                ++pos;
            }
        }
        if (tid == 0) p.cta_cnt[cta] = unsigned(total);
    }
    if (p.skip_arrive && j == n_b - 1 && n_b > 1) {  // failure-detection test only
        cp_async_wait<0>();
        return;
    }
    PHASE_MARK(5);
    arrive(ctl + kCands);
    if (!wait_count(p, ctl + kCands, unsigned(n_b), 2, s_ok)) {
        cp_async_wait<0>();
        return;
    }
    PHASE_MARK(6);

    // ---- exact selection ------------------------------------------------------
    // candidate counts and segment offsets of the sequence's blocks
    if (warp == 0) {
        int run = 0;
        for (int base = 0; base < n_b; base += 32) {
            const int jj = base + lane;
            const int v = jj < n_b ? int(ld_cg(p.cta_cnt + cb0 + jj)) : 0;
            int x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (jj < n_b) offs[jj] = run + x - v;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) { offs[n_b] = run; sv[4] = run; }
    }
    __syncthreads();
    const int n_cand = sv[4];
    DBG_MAX(0, n_cand);
    DBG_MAX(1, sv[3]);
    const bool fast = !p.force_slow && n_cand <= kSelCap;
    int32_t *sel_g = reinterpret_cast<int32_t *>(smem + kSelG);
    int32_t *idx_list = p.idx_out ? p.idx_out : p.idx_ws;

    if (fast) {
        level1_bins(2);  // nobody reads the level-1 histogram after barrier A
        __syncthreads();
        if (has_items) {
            unsigned *ckey = reinterpret_cast<unsigned *>(smem + kCandKey);
            int32_t *cgrp = reinterpret_cast<int32_t *>(smem + kCandG);
            unsigned *rh = reinterpret_cast<unsigned *>(smem + kRHist);
            // all candidate loads of a thread are issued before any is stored, so
            // the copy costs one L2 round trip per 8 entries a thread
            for (int i0 = tid; i0 < n_cand; i0 += kThreads * 8) {
                unsigned kv[8], gv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * kThreads;
                    kv[u] = gv[u] = 0u;
                    if (i < n_cand) {
                        int lo = 0, hi = n_b;  // segment jj with offs[jj] <= i < offs[jj+1]
                        while (hi - lo > 1) {
                            const int mid = (lo + hi) >> 1;
                            if (offs[mid] <= i) lo = mid; else hi = mid;
                        }
                        const int64_t src = seg + chunk_lo(lo) + (i - offs[lo]);
                        kv[u] = ld_cg(p.cand_key + src);
                        gv[u] = ld_cg(reinterpret_cast<const unsigned *>(p.cand_g) + src);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * kThreads;
                    if (i < n_cand) {
                        ckey[i] = kv[u];
                        cgrp[i] = int32_t(gv[u]);
                    }
                }
            }
            __syncthreads();
            PHASE_MARK(13);
            unsigned take_eq = 0;
            const unsigned kth = k_b > 0 ? radix_select_smem(ckey, n_cand, unsigned(k_b), rh,
                                                             scratch, sv + 8, &take_eq)
                                         : 0xFFFFFFFFu;
            PHASE_MARK(14);
            // ordered compaction (candidates are in ascending group order)
            if (tid == 0) { sv[5] = 0; sv[6] = 0; }
            __syncthreads();
            for (int base = 0; base < n_cand; base += kThreads * 4) {
                unsigned kk[4];
                int n_eq = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = base + tid * 4 + e;
                    kk[e] = i < n_cand ? ckey[i] : 0u;
                    n_eq += (i < n_cand && kk[e] == kth);
                }
                const int eq_seen = sv[5], written = sv[6];
                int tot_eq;
                int eq_before = eq_seen + block_exclusive_scan(n_eq, scratch, &tot_eq);
                bool sel[4];
                int n_sel = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = base + tid * 4 + e;
                    bool keep = false;
                    if (i < n_cand) {
                        if (kk[e] > kth) keep = true;
                        else if (kk[e] == kth) keep = unsigned(eq_before++) < take_eq;
                    }
                    sel[e] = keep;
                    n_sel += keep;
                }
                int tot_sel;
                int pos = written + block_exclusive_scan(n_sel, scratch, &tot_sel);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (sel[e]) {
                        if (pos < k_b) sel_g[pos] = cgrp[base + tid * 4 + e];
                        ++pos;
                    }
                if (tid == 0) { sv[5] = eq_seen + tot_eq; sv[6] = written + tot_sel; }
                __syncthreads();
            }
            if (p.idx_out && j == 0)
                for (int i = tid; i < p.k; i += kThreads) p.idx_out[int64_t(b) * p.k + i] = i < k_b ? sel_g[i] : -1;
        }
    } else {
        // -------- exact multi-pass selection over the sequence's blocks --------
        level1_bins(1);  // complete the level-1 histogram
        arrive(ctl + kSlowB);
        if (!wait_count(p, ctl + kSlowB, unsigned(n_b), 3, s_ok)) {
            cp_async_wait<0>();
            return;
        }
        if (warp == 0) {
            unsigned above = 0;
            const int t1 = k_b > 0 ? hist_walk(hist1, unsigned(k_b), true, &above) : -1;
            if (lane == 0) { sv[10] = t1; sv[11] = int(above); }
        }
        __syncthreads();
        const int t1 = sv[10];
        const unsigned need2 = unsigned(k_b) - unsigned(sv[11]);
        clear_smem(smem + kU, kUBytes);
        __syncthreads();
        for (int i = tid; i < nloc; i += kThreads) {
            const unsigned key = score_key(score_at(i));
            if (int(key >> 16) == t1) {
                const unsigned lo = key & 0xFFFFu;
                atomicAdd(h16 + (lo >> 1), (lo & 1u) ? 0x10000u : 1u);
            }
        }
        __syncthreads();
        flush_hist(h16, hist2);
        arrive(ctl + kSlowC);
        if (!wait_count(p, ctl + kSlowC, unsigned(n_b), 4, s_ok)) {
            cp_async_wait<0>();
            return;
        }
        if (warp == 0) {
            unsigned above = 0;
            const int lo = (k_b > 0 && t1 >= 0) ? hist_walk(hist2, need2, true, &above) : -1;
            if (lane == 0) { sv[12] = lo; sv[13] = int(above); }
        }
        __syncthreads();
        const bool none = k_b == 0 || t1 < 0 || sv[12] < 0;
        const unsigned kth = none ? 0xFFFFFFFFu : (unsigned(t1) << 16) | unsigned(sv[12]);
        const unsigned take_eq = none ? 0u : need2 - unsigned(sv[13]);
        // own counts for the tie rule and the output offsets
        {
            int gt = 0, eq = 0;
            for (int i = tid; i < nloc; i += kThreads) {
                const unsigned key = score_key(score_at(i));
                gt += key > kth;
                eq += key == kth;
            }
            int tgt, teq;
            block_exclusive_scan(gt, scratch, &tgt);
            block_exclusive_scan(eq, scratch, &teq);
            if (tid == 0) {
                p.cta_cnt[ncta + cta] = unsigned(tgt);
                p.cta_cnt[2 * ncta + cta] = unsigned(teq);
            }
        }
        arrive(ctl + kSlowD);
        if (!wait_count(p, ctl + kSlowD, unsigned(n_b), 5, s_ok)) {
            cp_async_wait<0>();
            return;
        }
        if (warp == 0) {
            // offsets of the blocks before this one: each takes its keys > K* and
            // the next ties in group order (blocks hold ascending group ranges)
            unsigned out_off = 0, eq_run = 0;
            for (int base = 0; base < j; base += 32) {
                const int jj = base + lane;
                const unsigned gtj = jj < j ? ld_cg(p.cta_cnt + ncta + cb0 + jj) : 0u;
                const unsigned eqj = jj < j ? ld_cg(p.cta_cnt + 2 * ncta + cb0 + jj) : 0u;
                unsigned x = eqj;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                const unsigned eq_before = eq_run + x - eqj;
                const unsigned take = take_eq > eq_before ? min(eqj, take_eq - eq_before) : 0u;
                unsigned add = gtj + take;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) add += __shfl_xor_sync(0xffffffffu, add, o);
                out_off += add;
                eq_run += __shfl_sync(0xffffffffu, x, 31);
            }
            if (lane == 0) {
                sv[14] = int(out_off);
                sv[15] = int(take_eq > eq_run ? take_eq - eq_run : 0u);  // my ties to take
            }
        }
        __syncthreads();
        {
            const int per = (nloc + kThreads - 1) / kThreads;
            const int i0 = min(nloc, tid * per), i1 = min(nloc, i0 + per);
            int n_eq = 0;
            for (int i = i0; i < i1; ++i) n_eq += score_key(score_at(i)) == kth;
            int tot;
            const int eq_start = block_exclusive_scan(n_eq, scratch, &tot);
            int eq_before = eq_start;
            const unsigned my_take = unsigned(sv[15]);
            int n_sel = 0;
            for (int i = i0; i < i1; ++i) {
                const unsigned key = score_key(score_at(i));
                n_sel += key > kth || (key == kth && unsigned(eq_before++) < my_take);
            }
            int pos = sv[14] + block_exclusive_scan(n_sel, scratch, &tot);
            eq_before = eq_start;
            for (int i = i0; i < i1; ++i) {
                const unsigned key = score_key(score_at(i));
                const bool keep = key > kth || (key == kth && unsigned(eq_before++) < my_take);
                if (keep) {
                    if (pos < k_b) idx_list[int64_t(b) * p.k + pos] = g_lo + i;
                    ++pos;
                }
            }
            if (j == 0)
                for (int i = k_b + tid; i < p.k; i += kThreads) idx_list[int64_t(b) * p.k + i] = -1;
        }
        // neither histogram is read by anyone any more: zero this block's slice of
        // the level-1 histogram, and the level-2 fine bins this block counted
        // (still in shared memory) plus a slice of the level-2 coarse bins
        {
            const int w0 = int((long long)kHistWords / 4 * j / n_b) * 4;
            const int w1 = int((long long)kHistWords / 4 * (j + 1) / n_b) * 4;
            for (int w = w0 + tid * 4; w < w1; w += kThreads * 4)
                *reinterpret_cast<uint4 *>(hist1 + w) = make_uint4(0, 0, 0, 0);
        }
        for (int w = tid; w < kFine / 2; w += kThreads) {
            const unsigned v = h16[w];
            if (v & 0xFFFFu) hist2[2 * w] = 0u;
            if (v >> 16) hist2[2 * w + 1] = 0u;
        }
        for (int cbin = int((long long)kCoarse * j / n_b) + tid;
             cbin < int((long long)kCoarse * (j + 1) / n_b); cbin += kThreads)
            hist2[kFine + cbin] = 0u;
        arrive(ctl + kSlowE);
        if (!wait_count(p, ctl + kSlowE, unsigned(n_b), 7, s_ok)) {
            cp_async_wait<0>();
            return;
        }
        if (has_items) {
            for (int i = tid; i < k_b; i += kThreads)
                sel_g[i] = int32_t(ld_cg(reinterpret_cast<const unsigned *>(idx_list) +
                                         int64_t(b) * p.k + i));
        }
        __syncthreads();
    }

    PHASE_MARK(7);
    // ---- attention items -------------------------------------------------------
    if (has_items) {
        const int gps = (k_b + S_b - 1) / S_b;
        const uint16_t *Kb = p.K + int64_t(b) * p.sK_b;
        const uint16_t *Vb = p.V + int64_t(b) * p.sV_b;
        uint16_t *skb = reinterpret_cast<uint16_t *>(smem + kKV);
        uint16_t *svb = skb + 2 * kChunk * QP;
        int *sgrp = reinterpret_cast<int *>(svb + 2 * kChunk * VP);
        float *state = reinterpret_cast<float *>(smem + kState);
        bool first = true;
        for (int it = j; it < items; it += n_b) {
            const int s = it % S_b, hg = it / S_b;
            const int h0 = hg * 64, HG = min(64, p.H_q - h0);
            const int MT = HG / 16, TS = 4;
            const int n_aw = MT * TS;  // attention warps
            if (!first) {
                __syncthreads();
                const uint16_t *qrow = p.q + (int64_t(b) * p.H_q + h0) * DQK;
                for (int e = tid; e < HG * (DQK / 8); e += kThreads) {
                    const int h = e / (DQK / 8), c8 = e % (DQK / 8);
                    cp_async16(smem_u32(sq + h * QP + c8 * 8), qrow + int64_t(h) * DQK + c8 * 8, 16);
                }
                cp_async_commit();
            }
            first = false;
            const int j0 = s * gps, j1 = min(k_b, j0 + gps);
            const int gpc = kChunk / P;
            const int nchunks = j1 > j0 ? (j1 - j0 + gpc - 1) / gpc : 0;
            auto issue = [&](int ci, int buf) {
                const int jb = j0 + ci * gpc;
                gather_chunk<DQK, DV>(skb + buf * kChunk * QP, svb + buf * kChunk * VP,
                                      sgrp + buf * kChunk, sel_g + jb, min(gpc, j1 - jb), P,
                                      G_b, Kb, Vb, QP, VP, tid, kThreads);
            };
            cp_async_wait<0>();
            __syncthreads();
            if (nchunks > 0) issue(0, 0);
            const int mt = warp % MT, ts = warp / MT;
            const int ntok = kChunk / TS, tok0 = ts * ntok;
            uint32_t qa[DQK / 16][4];  // unused: fragments come from shared memory
            AttnWarpState<DV> st;
            st.init();
            for (int ci = 0; ci < nchunks; ++ci) {
                const int buf = ci & 1;
                if (ci + 1 < nchunks) {
                    issue(ci + 1, buf ^ 1);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                __syncthreads();
                if (warp < n_aw)
                    attn_chunk<DQK, DV, 2, true>(st, qa, skb + buf * kChunk * QP,
                                                 svb + buf * kChunk * VP, sgrp + buf * kChunk, QP,
                                                 VP, P, tok0, ntok, p.scale_log2, sq, mt);
                __syncthreads();
            }
            PHASE_MARK(15);
            if (warp < n_aw) store_warp_state<DV>(st, state + warp * 16 * (DV + 2));
            __syncthreads();
            for (int e = tid; e < HG * (DV / 2); e += kThreads) {
                const int hl = e / (DV / 2), d2 = (e % (DV / 2)) * 2;
                float Lsum;
                const float4 rr = merge_states<DV>(state, MT, TS, hl, d2, Lsum);
                const int h = h0 + hl;
                if (S_b == 1) {
                    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
                    *reinterpret_cast<uint32_t *>(p.out + (int64_t(b) * p.H_q + h) * DV + d2) =
                        pack_bf2(rr.z * inv, rr.w * inv);
                    if (p.lse && d2 == 0)
                        p.lse[int64_t(b) * p.H_q + h] =
                            Lsum > 0.f ? (rr.x + log2f(Lsum)) * kLn2 : -INFINITY;
                } else {
                    const int64_t pi = (int64_t(b) * p.S_max + s) * p.H_q + h;
                    *reinterpret_cast<float2 *>(p.part_o + pi * DV + d2) = make_float2(rr.z, rr.w);
                    if (d2 == 0) p.part_ml[pi] = make_float2(rr.x, Lsum);
                }
            }
        }
        cp_async_wait<0>();
    }

    PHASE_MARK(8);
    // ---- combine the partial states ---------------------------------------------
    if (S_b > 1 && has_items) {
        arrive(ctl + kAtt);
        if (!wait_count(p, ctl + kAtt, unsigned(n_att), 6, s_ok)) return;
        PHASE_MARK(9);
        constexpr int PER = DV / 32;
        float *fw = reinterpret_cast<float *>(smem + kState) + warp * kMaxCtas;  // split weights
        for (int h = j + n_att * warp; h < p.H_q; h += n_att * kWarps) {
            const float2 *mlh = p.part_ml + int64_t(b) * p.S_max * p.H_q + h;
            float M = -INFINITY;
            for (int s0 = 0; s0 < S_b; s0 += 32) {
                const int s = s0 + lane;
                float m = -INFINITY;
                if (s < S_b) m = ld_cg_f(reinterpret_cast<const float *>(mlh + int64_t(s) * p.H_q));
                M = fmaxf(M, m);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float ref = M == -INFINITY ? 0.f : M;
            float Lsum = 0.f;
            for (int s0 = 0; s0 < S_b; s0 += 32) {
                const int s = s0 + lane;
                float wgt = 0.f;
                if (s < S_b) {
                    const float *ml = reinterpret_cast<const float *>(mlh + int64_t(s) * p.H_q);
                    wgt = exp2f(ld_cg_f(ml) - ref);
                    Lsum += wgt * ld_cg_f(ml + 1);
                    fw[s] = wgt;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
            __syncwarp();
            float acc[PER];
#pragma unroll
            for (int i = 0; i < PER; ++i) acc[i] = 0.f;
            const float *po = p.part_o + (int64_t(b) * p.S_max * p.H_q + h) * DV + lane * PER;
            const int64_t sstride = int64_t(p.H_q) * DV;
            int s = 0;
            for (; s + 8 <= S_b; s += 8) {
                float v[8][PER];
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int i = 0; i < PER; ++i) v[u][i] = ld_cg_f(po + (s + u) * sstride + i);
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int i = 0; i < PER; ++i) acc[i] += fw[s + u] * v[u][i];
            }
            for (; s < S_b; ++s)
#pragma unroll
                for (int i = 0; i < PER; ++i) acc[i] += fw[s] * ld_cg_f(po + s * sstride + i);
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
            uint16_t *orow = p.out + (int64_t(b) * p.H_q + h) * DV + lane * PER;
#pragma unroll
            for (int i = 0; i < PER; i += 2)
                *reinterpret_cast<uint32_t *>(orow + i) = pack_bf2(acc[i] * inv, acc[i + 1] * inv);
            if (p.lse && lane == 0)
                p.lse[int64_t(b) * p.H_q + h] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
            __syncwarp();
        }
    }
    PHASE_MARK(10);
    __syncthreads();
    if (tid == 0 && atomicAdd(ctl + kDepart, 1u) == unsigned(n_b) - 1u) {
        for (int i = 0; i < kNumCounters; ++i) ctl[i] = 0u;  // every block is done with them
    }
}

int num_sms() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

int s_max_for(int k, int P, int ncta) {
    int s = (k * P + kChunk - 1) / kChunk;
    return max(1, min(s, ncta));
}

template <int DQK>
constexpr int smem_bytes() {
    return kQ + 64 * (DQK + 8) * 2 + 128 + kCoarse * 4 + (2 * (kMaxCtas + 1) + 64 + 40) * 4;
}

struct WsLayout {
    size_t ctl, hist, cand_key, cand_g, gscore, cta_cnt, idx_ws, part_o, part_ml, total;
};

WsLayout ws_layout(int B, int G_max, int H_q, int d_v, int k, int P, int ncta) {
    WsLayout w;
    size_t off = 256;  // status + abort words
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    const int S_max = s_max_for(k, P, ncta);
    w.ctl = take(size_t(B) * kCtlWords * 4);
    w.hist = take(size_t(B) * 2 * kHistWords * 4);
    w.cand_key = take(size_t(B) * G_max * 4);
    w.cand_g = take(size_t(B) * G_max * 4);
    w.gscore = take(size_t(B) * G_max * 4);
    w.cta_cnt = take(size_t(3) * ncta * 4);
    w.idx_ws = take(size_t(B) * k * 4);
    w.part_o = take(size_t(B) * S_max * H_q * d_v * 4);
    w.part_ml = take(size_t(B) * S_max * H_q * 8);
    w.total = off;
    return w;
}

}  // namespace

bool fused_decode_supported(int B, int G_max, int H_i, int H_q, int d_qk, int d_v, int k, int P) {
    const int ncta = num_sms();
    if (ncta > kMaxCtas || B < 1 || 2 * B > ncta) return false;
    if (H_i > 16 || k > kMaxK || k < 1) return false;
    if (!((d_qk == 64 || d_qk == 128 || d_qk == 192) && (d_v == 64 || d_v == 128))) return false;
    if (!(H_q % 16 == 0 && (H_q <= 32 || H_q % 64 == 0))) return false;
    // 16-bit shared counters: a block's chunk must stay below 65536 groups
    const long long bound = (long long)B * G_max / (ncta - B) + 32;
    if (bound >= 65535) return false;
    (void)P;
    return true;
}

size_t fused_decode_ws_bytes(int B, int G_max, int H_q, int d_v, int k, int P) {
    if (!fused_decode_supported(B, G_max, 1, H_q, 128, d_v, k, P)) return 0;
    return ws_layout(B, G_max, H_q, d_v, k, P, num_sms()).total;
}

template <int NT, int DQK, int DV>
static cudaError_t launch_t(const Params &prm, int ncta, cudaStream_t st) {
    auto kern = fused_decode_kernel<NT, DQK, DV>;
    constexpr int smem = smem_bytes<DQK>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncta);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

#ifdef LCSW_PHASE_TIMERS
extern "C" int lcsw_debug_counters(unsigned *out, int reset) {
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(out, g_dbg_max, sizeof(unsigned) * 4);
    if (reset) {
        unsigned z[4] = {0, 0, 0, 0};
        cudaMemcpyToSymbol(g_dbg_max, z, sizeof z);
    }
    return int(cudaGetLastError());
}

extern "C" int lcsw_debug_phase_times(unsigned long long *first, unsigned long long *last,
                                      int reset) {
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(first, g_phase_first, sizeof(unsigned long long) * 16);
    cudaMemcpyFromSymbol(last, g_phase_last, sizeof(unsigned long long) * 16);
    if (reset) {
        unsigned long long hi[16], lo[16];
        for (int i = 0; i < 16; ++i) { hi[i] = ~0ull; lo[i] = 0ull; }
        cudaMemcpyToSymbol(g_phase_first, hi, sizeof hi);
        cudaMemcpyToSymbol(g_phase_last, lo, sizeof lo);
    }
    return int(cudaGetLastError());
}
#endif

cudaError_t launch_fused_decode(const lcsw_decode_args *a, void *ws, int *status,
                                cudaStream_t st) {
    const int ncta = num_sms();
    const WsLayout w = ws_layout(a->B, a->G_max, a->H_q, a->d_v, a->k, a->P, ncta);
    char *base = static_cast<char *>(ws);
    Params prm;
    prm.q_idx = a->q_idx;
    prm.w_head = a->w_head;
    prm.k_pooled = a->k_pooled;
    prm.sp_b = a->sp_b;
    prm.k_idx = a->k_idx;
    prm.sk_b = a->sk_b;
    prm.pool_w = a->pool_w;
    prm.sw_b = a->sw_b;
    prm.q = a->q;
    prm.K = a->K;
    prm.sK_b = a->sK_b;
    prm.V = a->V;
    prm.sV_b = a->sV_b;
    prm.seq_len = a->seq_len;
    prm.B = a->B;
    prm.G_max = a->G_max;
    prm.H_i = a->H_i;
    prm.P = a->P;
    prm.k = a->k;
    prm.H_q = a->H_q;
    prm.S_max = s_max_for(a->k, a->P, ncta);
    prm.force_slow = (a->flags & LCSW_DECODE_FORCE_MULTIPASS_SELECT) ? 1 : 0;
    prm.skip_arrive = (a->flags & LCSW_DECODE_TEST_SKIP_ARRIVE) ? 1 : 0;
    prm.scale_log2 = a->scale * kLog2e;
    prm.out = a->out;
    prm.lse = a->lse;
    prm.idx_out = a->idx_out;
    prm.scores_out = a->scores_out;
    prm.ctl = reinterpret_cast<unsigned *>(base + w.ctl);
    prm.hist = reinterpret_cast<unsigned *>(base + w.hist);
    prm.cand_key = reinterpret_cast<unsigned *>(base + w.cand_key);
    prm.cand_g = reinterpret_cast<int32_t *>(base + w.cand_g);
    prm.gscore = reinterpret_cast<float *>(base + w.gscore);
    prm.cta_cnt = reinterpret_cast<unsigned *>(base + w.cta_cnt);
    prm.idx_ws = reinterpret_cast<int32_t *>(base + w.idx_ws);
    prm.part_o = reinterpret_cast<float *>(base + w.part_o);
    prm.part_ml = reinterpret_cast<float2 *>(base + w.part_ml);
    prm.status = status;
    prm.abort_flag = status + 1;
    const int NT = a->H_i > 8 ? 2 : 1;
#define LCSW_FD(NTT, DQ, DVV)                                                         \
    if (NT == NTT && a->d_qk == DQ && a->d_v == DVV) return launch_t<NTT, DQ, DVV>(prm, ncta, st);
    LCSW_FD(1, 128, 128)
    LCSW_FD(1, 192, 128)
    LCSW_FD(1, 64, 64)
    LCSW_FD(1, 128, 64)
    LCSW_FD(1, 192, 64)
    LCSW_FD(1, 64, 128)
    LCSW_FD(2, 128, 128)
    LCSW_FD(2, 192, 128)
    LCSW_FD(2, 64, 64)
    LCSW_FD(2, 128, 64)
    LCSW_FD(2, 192, 64)
    LCSW_FD(2, 64, 128)
#undef LCSW_FD
    return cudaErrorInvalidValue;
}

}  // namespace lcsw
