// Persistent fused decode step: [append] -> indexer scores -> exact top-k
// groups -> sparse attention -> split-K combine, in one cooperative launch of
// one thread block per SM (the DSA retrieval chain of "G2C Brief --
// GLM-5.3-Flash", section "DSA keeps selected global access in eleven
// layers"; IndexPool from the reading notes, section 2).
//
// Work split.  Every sequence b gets a contiguous set of n_b >= 1 blocks,
// proportional to its bytes (pooled keys plus the K/V rows of its selected
// groups); block j of the set owns a contiguous chunk of 16-group tiles.
// Blocks exchange data (candidate slots, partial attention states) through
// words that are nonzero once written: a reader polls the data itself, with
// no fence or arrival counter.  Candidate words are double-buffered by a
// per-call parity (each block clears its own words of the idle buffer);
// partial states are cleared by the one block that reads them.  Only the
// exact fallback selection syncs through arrival counters.  On a wait that
// runs out the block records LCSW_ERR_TIMEOUT in the workspace status word,
// raises an abort flag every other wait honours, and returns.
//
// Phase 1 (HBM stream).  All 16 warps stream their tiles' pooled keys with
// bulk copies into per-warp rings in shared memory, load them into mma.sync
// A fragments (the k-permuted layout of index_scores.cu) and keep the scores
// in shared memory.  With one sequence the first copies go out before
// seq_len has arrived, on the guess that the cache is full.  The block that
// owns the group completed by the newest token pools it first (the exact
// arithmetic of the pooling kernel) and scores that fresh key.
//
// Local threshold.  Each block takes t_j, the 16-bit key bin where the count
// of its own keys from the top reaches its quota m_j = 2 x (its fair share
// k G_j / G_b) + 8 (all its keys, with t_j = 0, when that is all of them),
// and publishes every key at or above t_j: a fixed slot (overflow to a
// per-sequence segment) headed by (count, t_j).  No exchange precedes this:
// every key at or above T = max_j t_j is then published.  While the slots
// travel, the block prefetches the K/V rows of its first candidates and the
// query heads.
//
// Selection.  Every block loads every header of its sequence, then every
// candidate.  If at least k of them reach T, they hold the exact top k (every
// key >= K*, the k-th largest, is >= T), and each block ranks its own
// candidates among them by the packed value (key << 32) | ~group: rank < k
// means selected.  Past 32 own candidates, or for the optional full index
// output, the block finds K* instead (a histogram relative to T, then a rank
// count inside the bin).  Otherwise (too few, or too many candidates) every
// block of the sequence runs the exact multi-pass selection over its own
// scores -- a full level-1 histogram, a level-2 histogram of the low 16
// bits, per-block counts for the tie rule and the output order.
//
// Attention.  Each block attends over its own selected groups -- from the
// prefetch when they are among its first candidates, else gathered into
// shared memory (cp.async, 64 tokens a chunk, up to four chunks in flight) --
// with S = Q K^T and O = P V on mma.sync: warp (t, q) holds head tile t (16
// heads) and scores token quarter q of the chunk, the four quarters exchange
// row maxima and P through shared memory, and then warp (t, q) accumulates
// value dims quarter q of O for its heads, so no warp states need merging.
// Each block writes its partial (m, l, O) per head, and every block of the
// set merges the partial states of a share of the heads.
#pragma once

#include "attn_core.cuh"
#include "common.cuh"
#include "e4m3_core.cuh"
#include "fused.cuh"
#include "kernels.cuh"
#include "pool_core.cuh"
#include "select_core.cuh"
#include "tc_core.cuh"

namespace lcsw {
namespace {

constexpr int kThreads = kSelThreads;  // 512
constexpr int kWarps = kThreads / 32;
constexpr int kFine = 65536, kCoarse = 256, kHistWords = kFine + kCoarse;
constexpr int kChunkCap = 12288;   // scores of a block's chunk kept in shared memory
constexpr int kSelCap = 4096;      // candidates selected in shared memory (fast path)
constexpr int kSlot = 25;          // candidates published in a block's fixed slot
constexpr int kSlotWords = 1 + kSlot;  // 64-bit words: header, entries
constexpr int kSlotBytes = kSlotWords * 8;
constexpr int kQuotaPad = 8;       // local quota: 2 x fair share + kQuotaPad keys
constexpr int kTieCap = 256;       // threshold-bin candidates resolved by rank counting
constexpr int kMaxK = 2048;        // selected groups per sequence
constexpr int kCtlWords = 32;      // control words per sequence
constexpr int kMaxCtas = 160;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// control words (per sequence), reset to zero by the last block to leave the
// kernel: arrival counters of the fallback's sync points
constexpr int kSlowB = 1, kSlowC = 2, kSlowD = 3, kNumCounters = 4;
constexpr int kStream = kWarps;    // streaming warps
// Phase 1 streams the block's pooled keys through per-warp rings in shared
// memory filled by bulk copies: warp w scores tiles w, w + 16, w + 32, ... of
// the block's chunk (16 groups, 2 KB each) and keeps kRing of them in flight;
// FP8 tiles are 1088 bytes, so their rings hold kRingF8 of them.
constexpr int kRing = 4;
constexpr int kTileBytes = 16 * 128;
constexpr int kRingF8 = 7;
constexpr int kRingMax = kRingF8 > kRing ? kRingF8 : kRing;

// shared memory map (bytes); region U is reused phase by phase:
//   stream      per-warp rings [kWarps][kRing][kTileBytes]
//   threshold   local histogram [2048] u32 (at SelLayout::hist)
//   attention   AttLayout below, over region U and the scores after it once
//               they are dead; its Q rows and chunk buffer 0 receive the
//               block's own first candidates while the slots travel
//   selection   SelLayout below, right after chunk buffer 0 so that the
//               prefetch survives it
//   fallback    the 16-bit-pair histogram of the multi-pass selection
constexpr int kU = 0;
constexpr int kUBytes = kFine * 2;
static_assert(kWarps * kRing * kTileBytes <= kUBytes, "stream rings overflow region U");
static_assert(kWarps * kRingF8 * (16 * 64 + 16 * 4) <= kUBytes, "FP8 rings overflow region U");
constexpr int kScores = kU + kUBytes;                 // [kChunkCap] floats
constexpr int kMisc = kScores + kChunkCap * 4;        // small arrays and scalars
constexpr int kRankDirect = 32;    // own candidates ranked directly (else the K* path)
constexpr int kRankMax = 96;       // capacity of the rank counters (up to three warp rounds)
constexpr int kMiscBytes = 128 + (3 * (kMaxCtas + 1) + 64 + 40 + 64 + kChunk + kRankMax) * 4;
static_assert(kMiscBytes <= 4096, "small arrays overflow their region");
constexpr int kSelList = kMisc + 4096;                // own selected groups [kMaxK]
constexpr int kNewRows = kSelList + kMaxK * 4;        // newest group: [8][64] bf16, [8] f32
constexpr int kNewCode = kNewRows + 8 * 128 + 8 * 4;  // its FP8 row: [64] codes, scale
constexpr int kRingBars = kNewCode + 64 + 16;         // [kWarps][ring depth] mbarriers
constexpr int kQCode = (kRingBars + kWarps * kRingMax * 8 + 15) / 16 * 16;  // FP8 query: [16][64] codes, [16] scales
// the attention chunk buffers' group ids [4][kChunk] (-1 = masked), apart from
// region U and the scores: the prefetch writes buffer 0's row while the
// block's scores are still live
constexpr int kGids = (kQCode + 16 * 64 + 16 * 4 + 15) / 16 * 16;
constexpr int kSmemBytes = kGids + 4 * kChunk * 4;
static_assert(kRingBars % 8 == 0, "mbarrier alignment");

// Attention operands: Q [64 heads][QP], NBUF chunk buffers (each K [64
// tokens][QP] then V [64][VP]), P [64 heads][PP] bf16, per-quarter row maxima
// and sums [4][64] f32 (the chunks' group ids are at kGids).  Row pitches are
// padded by 16 bytes so ldmatrix rows fall on distinct banks.
constexpr int kAttBytes = kMisc - kU;
template <int DQK, int DV>
struct AttLayout {
    static constexpr int QP = DQK + 8, VP = DV + 8, PP = kChunk + 8;
    static constexpr int kv_bytes = kChunk * (QP + VP) * 2;
    static constexpr int fixed = 64 * QP * 2 + 64 * PP * 2 + 2 * 4 * 64 * 4;
    static constexpr int NBUF = (kAttBytes - fixed) / kv_bytes >= 4 ? 4 : (kAttBytes - fixed) / kv_bytes;
    static constexpr int q = 0;
    static constexpr int buf = q + 64 * QP * 2;  // chunk buffer i at buf + i * kv_bytes
    static constexpr int pt = buf + NBUF * kv_bytes;
    static constexpr int rm = pt + 64 * PP * 2;
    static constexpr int rl = rm + 4 * 64 * 4;
    static constexpr int total = rl + 4 * 64 * 4;
};
static_assert(AttLayout<192, 128>::NBUF >= 2, "attention chunk buffers");
static_assert(AttLayout<192, 128>::total <= kAttBytes, "attention operands overflow");

// Selection workspace: the sequence's slot headers, the candidates (keys and
// groups, or packed (key << 32 | ~group) values for ranking), a 2048-bin
// histogram and the threshold-bin ties.
// The candidate capacity is twice kSelCap where region U has room for it
// (d_qk <= 128: smaller Q rows and prefetch buffer).
template <int DQK, int DV>
struct SelLayout {
    static constexpr int hdr = (AttLayout<DQK, DV>::buf + AttLayout<DQK, DV>::kv_bytes + 15) / 16 * 16;
    static constexpr int key = hdr + kMaxCtas * 8;
    static constexpr int cap =
        key + 2 * kSelCap * 8 + 2048 * 4 + kTieCap * 8 <= kUBytes ? 2 * kSelCap : kSelCap;
    static constexpr int grp = key + cap * 4;
    static constexpr int hist = grp + cap * 4;
    static constexpr int tie = hist + 2048 * 4;
    static constexpr int end = tie + kTieCap * 8;
};
static_assert(SelLayout<192, 128>::end <= kUBytes, "selection overflows region U");
static_assert(SelLayout<128, 128>::end <= kUBytes, "selection overflows region U");

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
    uint8_t *kq;          // FP8 pooled keys (tile-major, e4m3_core.cuh) or null
    int64_t sq_b;         // its batch stride in bytes
    int B, G_max, H_i, P, k, H_q, force_slow, skip_arrive;
    int select_only;      // stop after the selection (idx_out required): no attention
    float scale_log2;
    uint16_t *out;
    float *lse;
    int32_t *idx_out;
    float *scores_out;
    const int32_t *idx_in;  // a given selection [B][k] (reuse kernel only)
    // workspace
    unsigned *ctl;        // [B][kCtlWords]
    unsigned *hist;       // [B][2][kHistWords]: level 1, level 2 (zero between calls)
    // Exchange buffers, two of each: a call uses buffer `parity` and clears its
    // own words of the other one, which the next call uses.  Every word is
    // written once per call and is nonzero once written, so a reader polls the
    // data itself (no fence, no arrival counter).
    unsigned long long *slots; // [2][ncta][kSlotWords]: (count+1 | t_j<<32), (key | g<<32)...
    unsigned long long *cand;  // [2][B][G_max]: entries past a slot's capacity, at g_lo + i
    int2 *ovf;                 // [2][ncta]: (first index, count) of a block's entries in cand
    unsigned *parity;          // ws word 2: buffer of this call, flipped by the last block
    unsigned *gdepart;         // ws word 3: blocks done with this call
    float *gscore;        // [B][G_max] spill of scores past kChunkCap
    unsigned *cta_cnt;    // [2][ncta]: keys > K*, keys == K* (exact path)
    int32_t *idx_ws;      // [B][k]
    float *part_o;        // [ncta][H_q][d_v]
    float2 *part_ml;      // [ncta][H_q]
    int *status;          // ws word 0
    int *abort_flag;      // ws word 1
};

// D = A(16x16, row) * B(16x8, col) + D, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// ------------------------------------------------------------ phase timers -
// Built with -DLCSW_PHASE_TIMERS, thread 0 of every block records the
// %globaltimer reading (ns, comparable across SMs) at each phase mark.
#ifdef LCSW_PHASE_TIMERS
__device__ long long g_stamp[160][40];
__device__ unsigned g_dbg_max[4];
#define DBG_MAX(i, v)                                                    \
    do {                                                                 \
        if (threadIdx.x == 0) atomicMax(&g_dbg_max[i], unsigned(v));     \
    } while (0)
#define DBG_ADD(i, v)                                                    \
    do {                                                                 \
        if (threadIdx.x == 0) atomicAdd(&g_dbg_max[i], unsigned(v));     \
    } while (0)
#define PHASE_MARK(i)                                                    \
    do {                                                                 \
        if (threadIdx.x == 0) g_stamp[blockIdx.x][i] = (long long)globaltimer_ns();        \
    } while (0)
#else
#define DBG_ADD(i, v) \
    do {              \
    } while (0)
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
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const uint4 *p) {
    uint4 r;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long r;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(r) : "l"(p));
    return r;
}
// Partial attention states travel as (float bits) ^ kPartTag: a stored 0 is a
// word not yet written (the tag is a signalling-NaN pattern no arithmetic
// produces).
constexpr unsigned kPartTag = 0x7FBFFFFFu;
__device__ __forceinline__ void st_part2(float *p, float a, float b) {
    asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1,%2};" ::"l"(p),
                 "r"(__float_as_uint(a) ^ kPartTag), "r"(__float_as_uint(b) ^ kPartTag)
                 : "memory");
}
__device__ __forceinline__ uint2 ld_relaxed_u32x2(const void *p) {
    uint2 r;
    asm volatile("ld.relaxed.gpu.global.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
__device__ __forceinline__ void st_relaxed_zero2(void *p) {
    asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1,%1};" ::"l"(p), "r"(0u) : "memory");
}
__device__ __forceinline__ void st_relaxed_zero4(void *p) {
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%1,%1,%1};" ::"l"(p), "r"(0u) : "memory");
}
__device__ __forceinline__ float part_dec(unsigned w) { return __uint_as_float(w ^ kPartTag); }
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
        for (int spin = 0; ld_acquire(cnt) < target; ++spin) {
            if ((spin & 63) == 63 && aborted(p.abort_flag)) { ok = 0; break; }
            if (clock64() - t0 > kSpinBudget) { raise_timeout(p, where); ok = 0; break; }
            __nanosleep(64);
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
__device__ __forceinline__ int find_from_top8(const unsigned (&v)[8], unsigned need,
                                              unsigned *above) {
    const int lane = threadIdx.x & 31;
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
__device__ __forceinline__ int warp_find_from_top(const unsigned *bins, unsigned need,
                                                  unsigned *above) {
    const int lane = threadIdx.x & 31;
    const uint4 a = ld_cg4(bins + lane * 8), b = ld_cg4(bins + lane * 8 + 4);
    const unsigned v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    return find_from_top8(v, need, above);
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

// Q rows of every head into the attention operands (one cp.async group).
template <int DQK, int DV>
__device__ __forceinline__ void att_load_q(unsigned char *u, const uint16_t *qrow, int H_q) {
    using AL = AttLayout<DQK, DV>;
    uint16_t *sq = reinterpret_cast<uint16_t *>(u + AL::q);
    for (int e = threadIdx.x; e < H_q * (DQK / 8); e += kThreads) {
        const int h = e / (DQK / 8), c8 = e % (DQK / 8);
        cp_async16(smem_u32(sq + h * AL::QP + c8 * 8), qrow + int64_t(h) * DQK + c8 * 8, 16);
    }
    cp_async_commit();
}

// The K/V rows of groups glist[0..n) (n <= 64/P) into chunk buffer `buf`
// (one cp.async group); their group ids (-1 = masked) into its row of gids.
template <int DQK, int DV>
__device__ __forceinline__ void att_gather(unsigned char *u, int *gids, int buf,
                                           const int32_t *glist, int n, int G, int P,
                                           const uint16_t *kb, const uint16_t *vb) {
    using AL = AttLayout<DQK, DV>;
    static_assert(AL::NBUF <= 4, "group id rows");
    uint16_t *dk = reinterpret_cast<uint16_t *>(u + AL::buf + buf * AL::kv_bytes);
    gather_chunk<DQK, DV>(dk, dk + kChunk * AL::QP, gids + buf * kChunk, glist, n, P, G, kb, vb,
                          AL::QP, AL::VP, threadIdx.x, kThreads);
}

// Attention of every query head over the tokens of groups own[0..n_own) of
// one sequence (complete groups [0, G)), with its partial state (m in log2
// units, l, unnormalised O) written to this block's slot of part_ml / part_o.
// Warp w = t + 4 q: head tile t (heads 16t..16t+15, t < H_q/16), token
// quarter q of each 64-token chunk for the scores, value dims [q DV/4,
// (q+1) DV/4) for the output.  Per chunk: S for the warp's 16 tokens -> row
// maxima of the quarters through shared memory -> P = 2^(s - m) as bf16 into
// shared memory -> every quarter's warp adds P V for its value dims over all
// 64 tokens.  Chunks stream through NBUF buffers.  With `prefetched` the Q
// rows and a first chunk are already in flight in buffer 0 (att_load_q and
// att_gather, with the unselected groups masked in its id row), and
// own[0..n_own) are the selected groups it does not hold, gathered after it.
// Group ids of the chunk buffers: gids [NBUF][kChunk].  Every wait here is on
// the block's own copies.
template <int DQK, int DV>
__device__ __forceinline__ void attend_groups(unsigned char *u, int *gids, const int32_t *own,
                                              int n_own, int G, int P, const uint16_t *kb,
                                              const uint16_t *vb, const uint16_t *qrow, int H_q,
                                              float scale_log2, float *part_o, float2 *part_ml,
                                              bool prefetched) {
    using AL = AttLayout<DQK, DV>;
    static_assert(AL::total <= kAttBytes && AL::NBUF >= 2, "attention operands overflow");
    constexpr int NBUF = AL::NBUF;
    constexpr int QP = AL::QP, VP = AL::VP, PP = AL::PP;
    constexpr int DW = DV / 4;       // value dims per warp
    constexpr int NTV = DW / 8;      // n-tiles of 8 value dims per warp
    uint16_t *sq = reinterpret_cast<uint16_t *>(u + AL::q);
    uint16_t *sp = reinterpret_cast<uint16_t *>(u + AL::pt);
    float *red_m = reinterpret_cast<float *>(u + AL::rm);  // [4][64]
    float *red_l = reinterpret_cast<float *>(u + AL::rl);  // [4][64]
    const int *sg = gids;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = lane & 3, gq = lane >> 2;
    const int mt = warp & 3, qq = warp >> 2;
    const bool wact = mt * 16 < H_q;
    const int lp2 = 31 - __clz(P);  // P is a power of two
    const int gpc = kChunk >> lp2;
    const int pre = prefetched ? 1 : 0;  // chunk 0 already in buffer 0
    const int nchunks = pre + (n_own + gpc - 1) / gpc;
    // chunk cc >= pre takes groups own[(cc - pre) gpc ..]
    auto gather = [&](int cc) {
        const int o0 = (cc - pre) * gpc;
        att_gather<DQK, DV>(u, gids, cc % NBUF, own + o0, min(gpc, n_own - o0), G, P, kb, vb);
    };

    if (!prefetched) {
        cp_async_wait<0>();  // an unused prefetch lands before its buffers are reused
        __syncthreads();
        att_load_q<DQK, DV>(u, qrow, H_q);
    } else if (nchunks > 1) {
        __syncthreads();  // the selection's shared arrays overlap buffers 1..
    }
    for (int c0 = pre; c0 < NBUF - 1 && c0 < nchunks; ++c0) gather(c0);

    float o[NTV][4];
#pragma unroll
    for (int i = 0; i < NTV; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int h0 = mt * 16 + gq, h1 = h0 + 8;
    for (int ci = 0; ci < nchunks; ++ci) {
        const int buf = ci % NBUF;
        __syncthreads();  // every warp is done with chunk ci - 1, whose buffer comes next
        if (ci + NBUF - 1 < nchunks) gather(ci + NBUF - 1);
        // chunk ci has landed once at most the chunks issued after it are pending
        const int after = min(nchunks - 1, ci + NBUF - 1) - ci;
        if (after >= 3) cp_async_wait<3>();
        else if (after == 2) cp_async_wait<2>();
        else if (after == 1) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();
        const uint16_t *ck = reinterpret_cast<const uint16_t *>(u + AL::buf + buf * AL::kv_bytes);
        const uint16_t *cv = ck + kChunk * QP;
        const int *cg = sg + buf * kChunk;
        float s[2][4];
        if (wact) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < DQK / 16; kk += 2) {
                uint32_t a[2][4];
                const int qr = mt * 16 + (lane & 15), qc = (lane >> 4) * 8;
                ldmatrix_x4(smem_u32(sq + qr * QP + kk * 16 + qc), a[0][0], a[0][1], a[0][2],
                            a[0][3]);
                ldmatrix_x4(smem_u32(sq + qr * QP + (kk + 1) * 16 + qc), a[1][0], a[1][1],
                            a[1][2], a[1][3]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int trow = qq * 16 + nt * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(smem_u32(ck + trow * QP + kk * 16 + (lane >> 3) * 8), b0, b1, b2,
                                b3);
                    mma_bf16_16816(s[nt], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
                    mma_bf16_16816(s[nt], a[1][0], a[1][1], a[1][2], a[1][3], b2, b3);
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int n0 = qq * 16 + nt * 8 + 2 * c;
                const bool v0 = cg[n0 >> lp2] >= 0, v1 = cg[(n0 + 1) >> lp2] >= 0;
                s[nt][0] = v0 ? s[nt][0] * scale_log2 : -INFINITY;
                s[nt][1] = v1 ? s[nt][1] * scale_log2 : -INFINITY;
                s[nt][2] = v0 ? s[nt][2] * scale_log2 : -INFINITY;
                s[nt][3] = v1 ? s[nt][3] * scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
                mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            if (c == 0) {
                red_m[qq * 64 + h0] = mx0;
                red_m[qq * 64 + h1] = mx1;
            }
        }
        __syncthreads();
        float al0 = 1.f, al1 = 1.f;
        if (wact) {
            float cm0 = red_m[h0], cm1 = red_m[h1];
#pragma unroll
            for (int q2 = 1; q2 < 4; ++q2) {
                cm0 = fmaxf(cm0, red_m[q2 * 64 + h0]);
                cm1 = fmaxf(cm1, red_m[q2 * 64 + h1]);
            }
            const float mn0 = fmaxf(m0, cm0), mn1 = fmaxf(m1, cm1);
            const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
            const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
            al0 = exp2f(m0 - ref0);
            al1 = exp2f(m1 - ref1);
            m0 = mn0;
            m1 = mn1;
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                s[nt][0] = exp2f(s[nt][0] - ref0);
                s[nt][1] = exp2f(s[nt][1] - ref0);
                s[nt][2] = exp2f(s[nt][2] - ref1);
                s[nt][3] = exp2f(s[nt][3] - ref1);
                ls0 += s[nt][0] + s[nt][1];
                ls1 += s[nt][2] + s[nt][3];
                const int col = qq * 16 + nt * 8 + 2 * c;
                *reinterpret_cast<uint32_t *>(sp + h0 * PP + col) = pack_bf2(s[nt][0], s[nt][1]);
                *reinterpret_cast<uint32_t *>(sp + h1 * PP + col) = pack_bf2(s[nt][2], s[nt][3]);
            }
            ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
            ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
            ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
            ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
            if (c == 0) {
                red_l[qq * 64 + h0] = ls0;
                red_l[qq * 64 + h1] = ls1;
            }
        }
        __syncthreads();
        if (wact) {
            l0 = l0 * al0 + red_l[h0] + red_l[64 + h0] + red_l[128 + h0] + red_l[192 + h0];
            l1 = l1 * al1 + red_l[h1] + red_l[64 + h1] + red_l[128 + h1] + red_l[192 + h1];
#pragma unroll
            for (int i = 0; i < NTV; ++i) {
                o[i][0] *= al0; o[i][1] *= al0;
                o[i][2] *= al1; o[i][3] *= al1;
            }
#pragma unroll
            for (int kt = 0; kt < kChunk / 16; ++kt) {
                uint32_t pa0, pa1, pa2, pa3;
                ldmatrix_x4(smem_u32(sp + (mt * 16 + (lane & 15)) * PP + kt * 16 + (lane >> 4) * 8),
                            pa0, pa1, pa2, pa3);
                const int vrow = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int dt = 0; dt < NTV; dt += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(smem_u32(cv + vrow * VP + qq * DW + (dt + (lane >> 4)) * 8),
                                      b0, b1, b2, b3);
                    mma_bf16_16816(o[dt], pa0, pa1, pa2, pa3, b0, b1);
                    mma_bf16_16816(o[dt + 1], pa0, pa1, pa2, pa3, b2, b3);
                }
            }
        }
    }
    cp_async_wait<0>();  // the Q rows, when there was no chunk
    // the block's partial state: O rows in tagged words, (m, l) by quarter 0
    if (wact) {
#pragma unroll
        for (int i = 0; i < NTV; ++i) {
            const int d = qq * DW + i * 8 + 2 * c;
            st_part2(part_o + int64_t(h0) * DV + d, o[i][0], o[i][1]);
            st_part2(part_o + int64_t(h1) * DV + d, o[i][2], o[i][3]);
        }
        if (qq == 0 && c == 0) {
            st_part2(reinterpret_cast<float *>(part_ml + h0), l0 > 0.f ? m0 : -INFINITY, l0);
            st_part2(reinterpret_cast<float *>(part_ml + h1), l1 > 0.f ? m1 : -INFINITY, l1);
        }
    }
}

// Blocks per sequence for per-sequence costs w[0..B) (shared memory, B <= 96):
// n_b = max(1, ceil(w_b / L)) for the smallest L with sum_b n_b <= ncta, to
// within 1/256 (L0 = ceil(sum_b w_b / (ncta - B)) always fits, since each
// ceiling adds less than one block), the blocks left over go to the sequence
// with the largest cost per block.  This minimises the largest per-block cost
// (proportional shares rounded down can leave a short sequence with almost
// two blocks' work on one).  The search for L splits its interval in 17 per
// round, one trial L a warp (the interval shrinks 289-fold in two rounds; a
// one-warp bisection took several microseconds at B = 64).  Writes
// cta_begin[0..B] (prefix sums, shared); every thread of the block calls it;
// scratch: kWarps words of shared memory.
__device__ __noinline__ void assign_blocks(const int *w, int B, int ncta, int *cta_begin,
                                           int *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned lo, hi, wmin, wmax;
    {
        unsigned wl[3];
        bool on[3];
        unsigned tot = 0;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int bb = 3 * lane + i;
            on[i] = bb < B;
            wl[i] = on[i] ? unsigned(max(0, w[bb])) : 0u;
            tot += wl[i];
        }
        tot = __reduce_add_sync(0xffffffffu, tot);
        wmin = 0xFFFFFFFFu;
        wmax = 0u;
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (on[i]) {
                wmin = min(wmin, wl[i]);
                wmax = max(wmax, wl[i]);
            }
        wmin = __reduce_min_sync(0xffffffffu, wmin);
        wmax = __reduce_max_sync(0xffffffffu, wmax);
        // L >= tot / ncta is necessary, L = ceil(tot / (ncta - B)) sufficient
        lo = max(1u, tot / unsigned(ncta));
        hi = max(1u, (tot + (ncta - B) - 1) / (ncta - B));
        if (wmin == wmax) lo = hi;  // equal costs: no search, the split below is even
        while (hi - lo > max(1u, hi >> 8)) {  // block-uniform
            const unsigned step = (hi - lo + kWarps) / (kWarps + 1);
            const unsigned L = min(hi, lo + step * unsigned(warp + 1));
            int c = 0;
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (on[i]) c += wl[i] > 0 ? int((wl[i] + L - 1) / L) : 1;
            c = __reduce_add_sync(0xffffffffu, c);
            if (lane == 0) scratch[warp] = c <= ncta ? 1 : 0;
            __syncthreads();
            // the first trial that fits is the new hi, the one before it the new lo
            int f = kWarps;
#pragma unroll
            for (int w2 = kWarps - 1; w2 >= 0; --w2)
                if (scratch[w2]) f = w2;
            const unsigned nlo = f > 0 ? min(hi, lo + step * unsigned(f)) : lo;
            if (f < kWarps) hi = min(hi, lo + step * unsigned(f + 1));
            lo = nlo;
            __syncthreads();  // scratch is rewritten next round
        }
    }
    if (threadIdx.x < 32) {
        unsigned wl[3];
        bool on[3];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int bb = 3 * lane + i;
            on[i] = bb < B;
            wl[i] = on[i] ? unsigned(max(0, w[bb])) : 0u;
        }
        int n[3];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int bb = 3 * lane + i;
            if (wmin == wmax)  // floor(ncta / B) each, one more for the first ncta % B
                n[i] = on[i] ? ncta / B + (bb < ncta % B ? 1 : 0) : 0;
            else
                n[i] = on[i] ? (wl[i] > 0 ? int((wl[i] + hi - 1) / hi) : 1) : 0;
        }
        int left = n[0] + n[1] + n[2];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) left += __shfl_xor_sync(0xffffffffu, left, o);
        left = ncta - left;
        if (left > 0) {
            // the sequence with the largest w / n (cross-multiplied; lowest index on ties)
            unsigned bw = 0, bn = 1;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (on[i] && (bi == 0x7fffffff ||
                              (unsigned long long)wl[i] * bn > (unsigned long long)bw * n[i])) {
                    bw = wl[i];
                    bn = unsigned(n[i]);
                    bi = 3 * lane + i;
                }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned ow = __shfl_xor_sync(0xffffffffu, bw, o);
                const unsigned on_ = __shfl_xor_sync(0xffffffffu, bn, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (oi == 0x7fffffff) continue;
                const unsigned long long a = (unsigned long long)ow * bn,
                                         c = (unsigned long long)bw * on_;
                if (bi == 0x7fffffff || a > c || (a == c && oi < bi)) {
                    bw = ow;
                    bn = on_;
                    bi = oi;
                }
            }
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (3 * lane + i == bi) n[i] += left;
        }
        // prefix sums: lane holds sequences 3 lane .. 3 lane + 2
        const int mine = n[0] + n[1] + n[2];
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int at = incl - mine;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int bb = 3 * lane + i;
            if (bb < B) cta_begin[bb] = at;
            at += n[i];
        }
        if (lane == 31) cta_begin[B] = incl;  // = ncta
    }
    __syncthreads();
}

// Merge of the partial states of one sequence's blocks, head by head: block j
// of the n_b blocks cb0.. of sequence b merges heads j, j + n_b, ...: it polls
// the partial words of every block of the sequence until all are written,
// writes the normalised output row, then clears the words it read for the
// next call.  Returns false if a bounded wait ran out (the status word is set).
// Few sources (a sequence with at most kFewSources blocks): a warp merges a
// whole head on its own, lane = a float4 column of the head's DV dims (two
// heads a warp for DV = 64), running over the sources with an online
// rescale, so the block's heads go 16 (or 32) at a time with no block-wide
// barrier.  A sequence of one block still writes and reads its one partial
// state, which keeps the words' protocol the same for every shape.
constexpr int kFewSources = 16;
template <int DV>
__device__ __forceinline__ bool merge_few(const Params &p, int b, int j, int n_b, int cb0) {
    constexpr int D4 = DV / 4;                 // 32 (DV = 128) or 16 lanes a head
    constexpr int HPW = 32 / D4;               // heads a warp merges at once
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int dc = lane % D4, sub = lane / D4;
    const int nh = (p.H_q - j + n_b - 1) / n_b;  // this block's heads: j, j + n_b, ...
    bool ok = true;
    for (int i0 = warp * HPW; i0 < nh && ok; i0 += kWarps * HPW) {  // warp-uniform
        const int hi = i0 + sub;
        const bool act = hi < nh;
        const int h = j + hi * n_b;
        float m_run = -INFINITY, l_run = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const long long t0 = clock64();
        for (int u = 0; u < n_b; ++u) {
            const int64_t pi = int64_t(cb0 + u) * p.H_q + (act ? h : 0);
            uint2 mlw = make_uint2(1u, 1u);
            uint4 ow = make_uint4(1u, 1u, 1u, 1u);
            if (act) {
                mlw = ld_relaxed_u32x2(p.part_ml + pi);
                ow = ld_relaxed_v4(reinterpret_cast<const uint4 *>(p.part_o + pi * DV + dc * 4));
            }
            for (int spin = 0;; ++spin) {
                const bool pend = act && (mlw.x == 0u || mlw.y == 0u || ow.x == 0u || ow.y == 0u ||
                                          ow.z == 0u || ow.w == 0u);
                if (!__any_sync(0xffffffffu, pend)) break;
                const bool give_up = clock64() - t0 > kSpinBudget ||
                                     ((spin & 63) == 63 && aborted(p.abort_flag));
                if (__any_sync(0xffffffffu, give_up)) {  // (warp-uniform)
                    ok = false;
                    break;
                }
                __nanosleep(64);
                if (pend) {
                    mlw = ld_relaxed_u32x2(p.part_ml + pi);
                    ow = ld_relaxed_v4(reinterpret_cast<const uint4 *>(p.part_o + pi * DV + dc * 4));
                }
            }
            if (!ok) break;
            const float ms = part_dec(mlw.x), ls = part_dec(mlw.y);
            if (act && ls > 0.f) {
                const float mn = fmaxf(m_run, ms);
                const float a = m_run == -INFINITY ? 0.f : exp2f(m_run - mn);
                const float w = exp2f(ms - mn);
                acc.x = acc.x * a + w * part_dec(ow.x);
                acc.y = acc.y * a + w * part_dec(ow.y);
                acc.z = acc.z * a + w * part_dec(ow.z);
                acc.w = acc.w * a + w * part_dec(ow.w);
                l_run = l_run * a + w * ls;
                m_run = mn;
            }
        }
        if (!ok) break;
        if (act) {
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            *reinterpret_cast<uint2 *>(p.out + (int64_t(b) * p.H_q + h) * DV + dc * 4) =
                make_uint2(pack_bf2(acc.x * inv, acc.y * inv), pack_bf2(acc.z * inv, acc.w * inv));
            if (p.lse && dc == 0)
                p.lse[int64_t(b) * p.H_q + h] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
        }
        __syncwarp();  // every lane of the head has read the (m, l) words
        // the words read are cleared for the next call
        if (act)
            for (int u = 0; u < n_b; ++u) {
                const int64_t pi = int64_t(cb0 + u) * p.H_q + h;
                st_relaxed_zero4(p.part_o + pi * DV + dc * 4);
                if (dc == 0) st_relaxed_zero2(p.part_ml + pi);
            }
    }
    if (!__syncthreads_and(ok)) {
        if (threadIdx.x == 0) raise_timeout(p, 6);
        return false;
    }
    return true;
}

template <int DV>
__device__ __forceinline__ bool merge_partials(const Params &p, unsigned char *smem, int *sv,
                                               float *sred, int b, int j, int n_b, int cb0) {
    if (n_b <= kFewSources) return merge_few<DV>(p, b, j, n_b, cb0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_src = n_b;
    auto src_cta = [&](int u) { return cb0 + u; };
    float *wsm = reinterpret_cast<float *>(smem + kU);       // [kMaxCtas] weights
    float *lsm = wsm + kMaxCtas;                              // [kWarps] sums of w l
    float *red = lsm + kMaxCtas;                              // [ngrp][DV]
    constexpr int D4 = DV / 4;                                // float4 columns
    const int sg = tid / D4, dc = tid % D4;                   // source group, column
    const int ngrp = kThreads / D4;                           // 16 (DV=128) or 32 (DV=64)
    // (no barrier: wsm, lsm and red overlap only the Q rows, which every warp
    // of the attention finished reading before its last P V)
    for (int h = j; h < p.H_q; h += n_b) {
        constexpr int kU4 = (kMaxCtas + 15) / 16;
        const int nu = (n_src - sg + ngrp - 1) / ngrp;
        float2 *mlp = p.part_ml + int64_t(src_cta(min(tid, n_src - 1))) * p.H_q + h;
        auto op_at = [&](int u) {
            return p.part_o + (int64_t(src_cta(sg + u * ngrp)) * p.H_q + h) * DV + dc * 4;
        };
        // First every source's (m, l) word, one thread per source (a light
        // poll while the sources are still storing; a source writes it right
        // after its O rows); then the O rows are loaded, and any word still
        // unwritten is polled again.
        uint2 mlw = make_uint2(1u, 1u);
        {
            bool ok = true;
            if (tid < n_src) {
                mlw = ld_relaxed_u32x2(mlp);
                const long long t0 = clock64();
                for (int spin = 0; mlw.x == 0u || mlw.y == 0u; ++spin) {
                    if (clock64() - t0 > kSpinBudget ||
                        ((spin & 63) == 63 && aborted(p.abort_flag))) {
                        ok = false;
                        break;
                    }
                    __nanosleep(spin < 4 ? 64 : 256);
                    mlw = ld_relaxed_u32x2(mlp);
                }
            }
            if (__syncthreads_or(!ok)) {
                if (tid == 0) raise_timeout(p, 6);
                return false;
            }
        }
        uint4 ow[kU4];
#pragma unroll
        for (int u = 0; u < kU4; ++u) {
            ow[u] = make_uint4(1u, 1u, 1u, 1u);
            if (u < nu) ow[u] = ld_relaxed_v4(reinterpret_cast<const uint4 *>(op_at(u)));
        }
        {
            const long long t0 = clock64();
            for (int spin = 0;; ++spin) {
                bool bad = false;
                if (mlw.x == 0u || mlw.y == 0u) {
                    bad = true;
                    mlw = ld_relaxed_u32x2(mlp);
                }
#pragma unroll
                for (int u = 0; u < kU4; ++u) {
                    if (ow[u].x == 0u || ow[u].y == 0u || ow[u].z == 0u || ow[u].w == 0u) {
                        bad = true;
                        ow[u] = ld_relaxed_v4(reinterpret_cast<const uint4 *>(op_at(u)));
                    }
                }
                if (!bad) break;
                if (clock64() - t0 > kSpinBudget ||
                    ((spin & 63) == 63 && aborted(p.abort_flag))) {
                    raise_timeout(p, 6);
                    sv[19] = 1;
                    break;
                }
                __nanosleep(128);
            }
        }
        PHASE_MARK(30);
        float2 ml = make_float2(-INFINITY, 0.f);
        if (tid < n_src) ml = make_float2(part_dec(mlw.x), part_dec(mlw.y));
        float4 ov[kU4];
#pragma unroll
        for (int u = 0; u < kU4; ++u) {
            ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (u < nu)
                ov[u] = make_float4(part_dec(ow[u].x), part_dec(ow[u].y), part_dec(ow[u].z),
                                    part_dec(ow[u].w));
        }
        // M = max over sources (warp max, then over the warps' maxima)
        float m = ml.x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) sred[warp] = m;
        __syncthreads();
        if (sv[19]) return false;  // a partial state never arrived
        PHASE_MARK(31);
        float M = lane < kWarps ? sred[lane] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float ref = M == -INFINITY ? 0.f : M;
        // source weights 2^(m_s - M) and L = sum of w_s l_s (warp sums first)
        float wl = 0.f;
        if (tid < n_src) {
            const float wgt = ml.y > 0.f ? exp2f(ml.x - ref) : 0.f;
            wsm[tid] = wgt;
            wl = wgt * ml.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wl += __shfl_xor_sync(0xffffffffu, wl, o);
        if (lane == 0) lsm[warp] = wl;
        __syncthreads();
        PHASE_MARK(32);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kU4; ++u) {
            if (u < nu) {
                const float wgt = wsm[sg + u * ngrp];
                if (wgt != 0.f) {
                    acc.x += wgt * ov[u].x;
                    acc.y += wgt * ov[u].y;
                    acc.z += wgt * ov[u].z;
                    acc.w += wgt * ov[u].w;
                }
            }
        }
        *reinterpret_cast<float4 *>(red + sg * DV + dc * 4) = acc;
        __syncthreads();
        if (tid < DV / 2) {
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) L += lsm[w];
            float a0 = 0.f, a1 = 0.f;
            for (int g2 = 0; g2 < ngrp; ++g2) {
                a0 += red[g2 * DV + 2 * tid];
                a1 += red[g2 * DV + 2 * tid + 1];
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            *reinterpret_cast<uint32_t *>(p.out + (int64_t(b) * p.H_q + h) * DV + 2 * tid) =
                pack_bf2(a0 * inv, a1 * inv);
            if (p.lse && tid == 0)
                p.lse[int64_t(b) * p.H_q + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        // the words read are cleared for the next call (after the output:
        // a barrier right behind global stores waits for them)
        if (tid < n_src) st_relaxed_zero2(mlp);
#pragma unroll
        for (int u = 0; u < kU4; ++u)
            if (u < nu) st_relaxed_zero4(op_at(u));
        if (h + n_b < p.H_q) __syncthreads();
    }
    return true;
}

template <int NT, int DQK, int DV, bool F8>
__global__ void __launch_bounds__(kThreads, 1) fused_decode_kernel(const Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned *h16 = reinterpret_cast<unsigned *>(smem + kU);
    float *sscore = reinterpret_cast<float *>(smem + kScores);
    uint16_t *newkey = reinterpret_cast<uint16_t *>(smem + kMisc);            // [64]
    int *cta_begin = reinterpret_cast<int *>(smem + kMisc + 128);             // [kMaxCtas + 1]
    int *offs = cta_begin + kMaxCtas + 1;                                     // [kMaxCtas + 1]
    int *lens = offs + kMaxCtas + 1;                                          // [kMaxCtas]
    int *sv = lens + kMaxCtas;                                                // scalars [64]
    int *scratch = sv + 64;                                                   // [40]
    float *sred = reinterpret_cast<float *>(scratch + 40);                    // [64]
    int *spec_g = reinterpret_cast<int *>(sred + 64);                         // [kChunk]
    int *rank = spec_g + kChunk;                                              // [kRankMax]
    int32_t *sel = reinterpret_cast<int32_t *>(smem + kSelList);              // [kMaxK]
    int *gids = reinterpret_cast<int *>(smem + kGids);                        // [4][kChunk]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x, ncta = gridDim.x;
    const int B = p.B, P = p.P;
    PHASE_MARK(0);
    // this call's exchange buffers (the previous call's last block flipped it)
    const int par = int(ld_cg(p.parity) & 1u);
    unsigned long long *slots_cur = p.slots + size_t(par) * ncta * kSlotWords;
    unsigned long long *cand_cur = p.cand + size_t(par) * p.B * p.G_max;
    // where this block's overflow entries went in the previous call (cleared at
    // the end of this one)
    const int2 ovf_old = p.ovf[(par ^ 1) * ncta + cta];

    // Each warp streams through its own ring of RING tiles (lane 0 issues the
    // bulk copies; completion on the slot's mbarrier).
    constexpr int RING = F8 ? kRingF8 : kRing;
    constexpr int SLOT = F8 ? kE4m3TileBytes : kTileBytes;
    unsigned char *ring = smem + kU + warp * RING * SLOT;
    uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + kRingBars) + warp * RING;
    int n_issued = 0;  // lane 0: tiles of this warp issued so far
    // lane 0: this warp's tile kk of the chunk [lo, hi) of sequence bb's pooled
    // keys (bf16 rows, or whole FP8 tiles of 16 groups)
    auto issue_tile_of = [&](int bb, int lo, int hi, int kk) {
        const int g0 = lo + (warp + kk * kStream) * 16;
        const void *src;
        uint32_t bytes;
        if constexpr (F8) {
            src = p.kq + int64_t(bb) * p.sq_b + int64_t(g0 / 16) * kE4m3TileBytes;
            bytes = kE4m3TileBytes;
        } else {
            src = p.k_pooled + int64_t(bb) * p.sp_b + int64_t(g0) * 64;
            bytes = uint32_t(min(16, hi - g0)) * 128u;
        }
        mbar_expect_tx(wbar + kk % RING, bytes);
        bulk_load(ring + (kk % RING) * SLOT, src, bytes, wbar + kk % RING);
        ++n_issued;
    };
    auto warp_tiles = [&](int lo, int hi) {
        const int nt = hi > lo ? (hi - lo + 15) / 16 : 0;
        return nt > warp ? (nt - warp + kStream - 1) / kStream : 0;
    };
    if (lane == 0) {
        for (int i = 0; i < RING; ++i) mbar_init(wbar + i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the indexer query of sequence bb as mma.sync B fragments (head nt*8 + r,
    // k-permuted like the keys) and its head weights
    const int r = lane >> 2, c = lane & 3;
    uint32_t bq[NT][4][2];
    float wv[NT][2];
    // The indexer query of sequence bb: raw bf16 loads first (fetch_query),
    // then its fragments (prep_query).  bf16: head nt*8 + r as mma.sync B
    // fragments, k-permuted like the keys.  FP8: warp w quantizes head w
    // once for the block (two dims a lane, the head's amax by shuffles) into
    // shared memory, and every warp then takes as f16 pairs the codes of
    // dims 16c + 4s .. 16c + 4s + 3 for k-step s.
    uint4 qraw[NT][2];
    uint32_t qpair = 0u;  // FP8: dims 2 lane, 2 lane + 1 of head `warp`
    uint8_t *qcode = smem + kQCode;
    float *qscale = reinterpret_cast<float *>(smem + kQCode + 16 * 64);
    auto fetch_query = [&](int bb) {
        if constexpr (F8) {
            if (warp < p.H_i)
                qpair = __ldg(reinterpret_cast<const uint32_t *>(
                    p.q_idx + (int64_t(bb) * p.H_i + warp) * 64 + 2 * lane));
        } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int head = nt * 8 + r;
                qraw[nt][0] = qraw[nt][1] = make_uint4(0, 0, 0, 0);
                if (head < p.H_i) {
                    const uint16_t *qp = p.q_idx + (int64_t(bb) * p.H_i + head) * 64;
                    qraw[nt][0] = ld_nc16(qp + 8 * c);
                    qraw[nt][1] = ld_nc16(qp + 32 + 8 * c);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = nt * 8 + 2 * c + e;
                wv[nt][e] = h < p.H_i ? __ldg(p.w_head + int64_t(bb) * p.H_i + h) : 0.f;
            }
    };
    auto prep_query = [&]() {
        if constexpr (F8) {
            if (warp < NT * 8) {  // warp-uniform
                const float x0 = bf_lo(qpair), x1 = bf_hi(qpair);
                float amax = fmaxf(fabsf(x0), fabsf(x1));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const float sc = e4m3_row_scale(amax);
                uint32_t cw = 0u;
                if (sc != 0.f) {
                    const float inv = __frcp_rn(sc);
                    cw = e4m3_quantize(x0, sc, inv) | (e4m3_quantize(x1, sc, inv) << 8);
                }
                *reinterpret_cast<uint16_t *>(qcode + warp * 64 + 2 * lane) = uint16_t(cw);
                if (lane == 0) qscale[warp] = sc;
            }
            __syncthreads();
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int head = nt * 8 + r;
                const uint4 w4 = *reinterpret_cast<const uint4 *>(qcode + head * 64 + 16 * c);
                const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2) {
                    bq[nt][s2][0] = e4m3x2_f16x2(w[s2]);
                    bq[nt][s2][1] = e4m3x2_f16x2(w[s2] >> 16);
                }
                // the accumulator's heads nt*8 + 2c + e take that head's query scale
#pragma unroll
                for (int e = 0; e < 2; ++e) wv[nt][e] *= qscale[nt * 8 + 2 * c + e];
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint4 h0 = qraw[nt][0], h1 = qraw[nt][1];
                bq[nt][0][0] = h0.x; bq[nt][0][1] = h0.y;
                bq[nt][1][0] = h0.z; bq[nt][1][1] = h0.w;
                bq[nt][2][0] = h1.x; bq[nt][2][1] = h1.y;
                bq[nt][3][0] = h1.z; bq[nt][3][1] = h1.w;
            }
        }
    };
    // One sequence: its length and query go out first (small loads that must
    // not queue behind the burst below), then, since the chunk split depends
    // only on G_b, the warp's first copies on the guess that the cache is full
    // (G_b = G_max); if it is not, they are waited out and reissued below.
    // Several sequences: the copies wait for the split.  Issued before the
    // lengths arrive, on the guess that every cache is full, they delayed the
    // length loads behind them by about 3 us.
    int L_first = 0;
    if (B == 1) {
        L_first = __ldg(p.seq_len);
        fetch_query(0);
    }
    int spec_lo = 0, spec_hi = 0;
    if (B == 1 && lane == 0) {
        const int tiles0 = (p.G_max + 15) / 16;
        spec_lo = 16 * int((long long)tiles0 * cta / ncta);
        spec_hi = min(p.G_max, 16 * int((long long)tiles0 * (cta + 1) / ncta));
        const int n0 = warp_tiles(spec_lo, spec_hi);
        for (int kk = 0; kk < min(RING, n0); ++kk) issue_tile_of(0, spec_lo, spec_hi, kk);
    }
    // even split: ncta / B blocks a sequence, one more for the first ncta % B
    auto even_seq = [&](int cc) {
        const int q = ncta / B, rr = ncta % B;
        return cc < rr * (q + 1) ? cc / (q + 1) : rr + (cc - rr * (q + 1)) / q;
    };
    auto even_begin = [&](int bb) { return bb * (ncta / B) + min(bb, ncta % B); };

    // ---- roles: blocks per sequence, proportional to its cost ------------------
    int b, cb0, n_b, L_b, G_b;
    if (tid == 0) {
        sv[19] = 0; sv[27] = 0; sv[31] = 0; sv[32] = 0; sv[33] = 0; sv[34] = 0;
        sv[36] = 0; sv[37] = 0;
    }
    if (B == 1) {
        L_b = L_first;
        G_b = L_b / P;
        G_b = G_b < 0 ? 0 : (G_b > p.G_max ? p.G_max : G_b);
        b = 0;
        cb0 = 0;
        n_b = ncta;
        __syncthreads();
    } else {
        // cost of a sequence, in 64-byte units: its pooled keys plus the K/V
        // rows of its selected groups
        int wv = 0;
        if (tid < B) {
            const int L = __ldg(p.seq_len + tid);
            lens[tid] = L;
            int G = L / P;
            G = G < 0 ? 0 : (G > p.G_max ? p.G_max : G);
            // (a selected token weighs twice its bytes: a block attends more
            // slowly than it streams keys, about 64 tokens a microsecond)
            wv = 2 * G + min(p.k, G) * P * ((DQK + DV) / 16);
        }
        if (tid < B) offs[tid] = wv;
        __syncthreads();
        if (__syncthreads_and(tid >= B || offs[tid] == offs[0])) {
            // equal costs: the even split, which is what assign_blocks gives them
            b = even_seq(cta);
            cb0 = even_begin(b);
            n_b = even_begin(b + 1) - cb0;
        } else {
            assign_blocks(offs, B, ncta, cta_begin, scratch);
            for (int bb = tid; bb < B; bb += kThreads)
                if (cta_begin[bb] <= cta && cta < cta_begin[bb + 1]) sv[1] = bb;
            __syncthreads();
            b = sv[1];
            cb0 = cta_begin[b];
            n_b = cta_begin[b + 1] - cb0;
        }
        L_b = lens[b];
        G_b = L_b / P;
        G_b = G_b < 0 ? 0 : (G_b > p.G_max ? p.G_max : G_b);
    }
    const int j = cta - cb0;
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
    const uint16_t *Kb = p.K + int64_t(b) * p.sK_b;
    const uint16_t *Vb = p.V + int64_t(b) * p.sV_b;
    int *s_ok = sv + 2;
    PHASE_MARK(1);

    // ---- phase-1 prologue: first tiles in flight, indexer query, append -------
    // The block's chunk of pooled keys is one contiguous range.  Lane 0 of each
    // warp has the warp's first RING tiles in flight (one sequence: issued
    // above when the guessed chunk was right), so the prologue's own loads
    // overlap them, and refills a slot as soon as the warp has read it.
    const int n_mine = warp_tiles(g_lo, g_hi);
    auto issue_tile = [&](int kk) { issue_tile_of(b, g_lo, g_hi, kk); };
    if (lane == 0) {
        if (B == 1 && (spec_lo != g_lo || spec_hi != g_hi)) {
            // the guess was wrong: let its copies land, then start over
            for (int kk = 0; kk < n_issued; ++kk) mbar_wait(wbar + kk, 0u, kWaitNs);
            for (int i = 0; i < RING; ++i) {
                asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(wbar + i))
                             : "memory");
                mbar_init(wbar + i, 1);
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            n_issued = 0;
        }
        for (int kk = n_issued; kk < min(RING, n_mine); ++kk) issue_tile(kk);
    }
    if (B > 1) fetch_query(b);
    prep_query();

    PHASE_MARK(23);
    // append: the group the newest token completes is pooled by the warp
    // whose tile holds it, just before it scores that tile, from rows staged
    // here
    int g_new = -1;
    if (p.k_idx && G_b > 0 && L_b % P == 0) g_new = G_b - 1;
    const int t_new = g_new >= g_lo && g_new < g_hi ? (g_new - g_lo) / 16 : -1;
    uint16_t *krows = reinterpret_cast<uint16_t *>(smem + kNewRows);  // [P][64]
    float *kw = reinterpret_cast<float *>(smem + kNewRows + 8 * 128);  // [P]
    if (t_new >= 0 && warp == t_new % kStream) {
        const uint16_t *src = p.k_idx + int64_t(b) * p.sk_b + int64_t(g_new) * P * 64;
        for (int e = lane; e < P * 8; e += 32) cp_async16(smem_u32(krows + e * 8), src + e * 8, 16);
        if (lane < P) cp_async4(smem_u32(kw + lane), p.pool_w + int64_t(b) * p.sw_b + int64_t(g_new) * P + lane);
        cp_async_commit();
    }
    PHASE_MARK(2);

    // ---- phase 1: stream pooled keys, score ----------------------------------
    unsigned kmax16 = 0;  // largest 16-bit key bin this thread scored
    const uint8_t *newcode = smem + kNewCode;  // the newest group's FP8 row
    const float *newscale = reinterpret_cast<const float *>(smem + kNewCode + 64);
    auto score_tile = [&](int t, const unsigned char *tile) {
        const int ga = g_lo + t * 16 + r, gb = ga + 8;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        float ska = 1.f, skb = 1.f;  // FP8: the two rows' key scales
        if constexpr (F8) {
            // rows r and r + 8: codes [16c, 16c + 16); word s feeds k-step s
            uint4 Ar = *reinterpret_cast<const uint4 *>(tile + r * 64 + 16 * c);
            uint4 Ab = *reinterpret_cast<const uint4 *>(tile + (r + 8) * 64 + 16 * c);
            ska = *reinterpret_cast<const float *>(tile + 1024 + 4 * r);
            skb = *reinterpret_cast<const float *>(tile + 1024 + 4 * (r + 8));
            if (ga == g_new) {  // the freshly pooled and quantized key
                Ar = *reinterpret_cast<const uint4 *>(newcode + 16 * c);
                ska = *newscale;
            }
            if (gb == g_new) {
                Ab = *reinterpret_cast<const uint4 *>(newcode + 16 * c);
                skb = *newscale;
            }
            const uint32_t wr[4] = {Ar.x, Ar.y, Ar.z, Ar.w}, wb[4] = {Ab.x, Ab.y, Ab.z, Ab.w};
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                const uint32_t a0 = e4m3x2_f16x2(wr[s2]), a2 = e4m3x2_f16x2(wr[s2] >> 16);
                const uint32_t a1 = e4m3x2_f16x2(wb[s2]), a3 = e4m3x2_f16x2(wb[s2] >> 16);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_f16_16816(acc[nt], a0, a1, a2, a3, bq[nt][s2][0], bq[nt][s2][1]);
            }
        } else {
            uint4 A[4];
            A[0] = *reinterpret_cast<const uint4 *>(tile + r * 128 + 16 * c);
            A[1] = *reinterpret_cast<const uint4 *>(tile + r * 128 + 64 + 16 * c);
            A[2] = *reinterpret_cast<const uint4 *>(tile + (r + 8) * 128 + 16 * c);
            A[3] = *reinterpret_cast<const uint4 *>(tile + (r + 8) * 128 + 64 + 16 * c);
            if (ga == g_new) {  // the freshly pooled key replaces the stale cache row
                A[0] = *reinterpret_cast<const uint4 *>(newkey + 8 * c);
                A[1] = *reinterpret_cast<const uint4 *>(newkey + 32 + 8 * c);
            }
            if (gb == g_new) {
                A[2] = *reinterpret_cast<const uint4 *>(newkey + 8 * c);
                A[3] = *reinterpret_cast<const uint4 *>(newkey + 32 + 8 * c);
            }
            const uint32_t A0[4] = {A[0].x, A[0].z, A[1].x, A[1].z};
            const uint32_t A2[4] = {A[0].y, A[0].w, A[1].y, A[1].w};
            const uint32_t A1[4] = {A[2].x, A[2].z, A[3].x, A[3].z};
            const uint32_t A3[4] = {A[2].y, A[2].w, A[3].y, A[3].w};
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_bf16_16816(acc[nt], A0[s2], A1[s2], A2[s2], A3[s2], bq[nt][s2][0],
                                   bq[nt][s2][1]);
        }
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
        const int li = t * 16 + r + 8 * c;
        const bool mine = c < 2 && g_lo + li < g_hi;
        // FP8: the row's key scale (>= 0) comes out of the head sum
        const float sc = __fadd_rn(F8 ? (c == 0 ? __fmul_rn(pa, ska) : __fmul_rn(pb, skb))
                                      : (c == 0 ? pa : pb),
                                   0.0f);
        if (mine) {
            if (li < kChunkCap) sscore[li] = sc;
            else p.gscore[seg + g_lo + li] = sc;
            if (p.scores_out) p.scores_out[seg + g_lo + li] = sc;
            kmax16 = max(kmax16, score_key(sc) >> 16);
        }
    };
    // Warp w scores its tiles in order.  A tile that never lands stops the
    // warp's work but not its barriers.
    bool stream_ok = true;
    for (int kk = 0; kk < n_mine; ++kk) {
        const int slot = kk % RING, t = warp + kk * kStream;
        if (stream_ok &&
            !__all_sync(0xffffffffu, mbar_wait(wbar + slot, unsigned(kk / RING) & 1u, kWaitNs))) {
            stream_ok = false;  // warp-uniform: score_tile shuffles across the warp
            raise_timeout(p, 7);
            sv[19] = 1;
        }
        if (t == t_new) {  // this warp pools the newest group before scoring its tile
            cp_async_wait<0>();
            __syncwarp();
            pool_staged(P, krows, kw, lane, newkey,
                        F8 ? nullptr : p.k_pooled + int64_t(b) * p.sp_b + int64_t(g_new) * 64);
            __syncwarp();
            if constexpr (F8) {  // ... and quantizes it into the FP8 cache
                if (lane < 8) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(newkey + 8 * lane);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                    float amax = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        amax = fmaxf(amax, fmaxf(fabsf(bf_lo(ws[i])), fabsf(bf_hi(ws[i]))));
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFu, amax, 1));
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFu, amax, 2));
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFu, amax, 4));
                    const float sc = e4m3_row_scale(amax);
                    uint32_t cw[2] = {0u, 0u};
                    if (sc != 0.f) {
                        const float inv = __frcp_rn(sc);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float x = (i & 1) ? bf_hi(ws[i / 2]) : bf_lo(ws[i / 2]);
                            cw[i / 4] |= e4m3_quantize(x, sc, inv) << (8 * (i % 4));
                        }
                    }
                    uint8_t *trow = p.kq + int64_t(b) * p.sq_b +
                                    int64_t(g_new / 16) * kE4m3TileBytes;
                    *reinterpret_cast<uint2 *>(smem + kNewCode + 8 * lane) = make_uint2(cw[0], cw[1]);
                    *reinterpret_cast<uint2 *>(trow + (g_new % 16) * 64 + 8 * lane) =
                        make_uint2(cw[0], cw[1]);
                    if (lane == 0) {
                        *reinterpret_cast<float *>(smem + kNewCode + 64) = sc;
                        *reinterpret_cast<float *>(trow + 1024 + (g_new % 16) * 4) = sc;
                    }
                }
                __syncwarp();
            }
        }
        if (stream_ok) score_tile(t, ring + slot * SLOT);
        __syncwarp();
        if (lane == 0 && stream_ok && kk + RING < n_mine) {
            fence_async_smem();  // the warp's reads of the slot come before the copy
            issue_tile(kk + RING);
        }
    }
    if (lane == 0) {
        if (stream_ok) {  // every copy landed: retire the barriers
            for (int i = 0; i < RING; ++i)
                asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(wbar + i))
                             : "memory");
        } else {  // the copies in flight land before the block leaves or reuses the ring
            for (int kk = max(0, n_issued - RING); kk < n_issued; ++kk)
                mbar_wait(wbar + kk % RING, unsigned(kk / RING) & 1u, kWaitNs);
        }
    }
    kmax16 = __reduce_max_sync(0xffffffffu, kmax16);
    if (lane == 0) atomicMax(sv + 27, int(kmax16));
    PHASE_MARK(4);
    __syncthreads();  // every warp is done with its ring: region U is free
    if (sv[19]) return;  // a key tile never landed (the status word says so)
    if (p.scores_out && j == 0)  // -inf past the last complete group: the full row
        for (int g = G_b + tid; g < p.G_max; g += kThreads) p.scores_out[seg + g] = -INFINITY;
    auto score_at = [&](int li) -> float {
        return li < kChunkCap ? sscore[li] : ld_cg_f(p.gscore + seg + g_lo + li);
    };

    // ---- local threshold: the bin of this block's quota-th largest key ---------
    // quota = min(nloc, 2 ceil(k_b nloc / G_b) + kQuotaPad).  The 2048 bins
    // below the block's largest 16-bit bin (tracked while streaming) hold the
    // count; a key further down counts in bin 0, and a threshold there
    // publishes every key.  One warp walks the bins from the top.
    {
        const int share = G_b > 0 ? int(((long long)k_b * nloc + G_b - 1) / G_b) : 0;
        const int quota = min(nloc, 2 * share + kQuotaPad);
        unsigned *lh = reinterpret_cast<unsigned *>(smem + SelLayout<DQK, DV>::hist);
        if (quota > 0 && quota < nloc) {  // block-uniform
            const unsigned base = unsigned(max(0, sv[27] - 2047));
            for (int i = tid; i < 2048; i += kThreads) lh[i] = 0u;
            __syncthreads();
            for (int i = tid; i < nloc; i += kThreads) {
                const unsigned bin = max(score_key(score_at(i)) >> 16, base) - base;
                if (LCSW_INBOUNDS(bin < 2048u, 103)) atomicAdd(lh + bin, 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l holds bins [2048 - 64 (l + 1), 2048 - 64 l): lane 0 the top
                const unsigned *hb = lh + 2048 - 64 * (lane + 1);
                unsigned mine = 0;
#pragma unroll
                for (int i = 0; i < 64; i += 4) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(hb + i);
                    mine += v.x + v.y + v.z + v.w;
                }
                unsigned incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const unsigned excl = incl - mine;
                const unsigned bal =
                    __ballot_sync(0xffffffffu, excl < unsigned(quota) && incl >= unsigned(quota));
                const int src = bal ? __ffs(bal) - 1 : 31;
                int tb = 0;
                if (lane == src) {
                    unsigned cum = excl;
                    for (int i = 63; i >= 0; --i) {
                        cum += hb[i];
                        if (cum >= unsigned(quota)) {
                            tb = 2048 - 64 * (lane + 1) + i;
                            break;
                        }
                    }
                }
                tb = __shfl_sync(0xffffffffu, tb, src);
                if (lane == 0) sv[3] = tb == 0 ? 0 : int(base) + tb;
            }
        } else if (tid == 0) {
            // a block whose quota is all of its keys publishes them all with the
            // threshold 0, so it never raises T
            sv[3] = 0;
        }
        __syncthreads();
    }
    PHASE_MARK(3);

    // ---- candidates: this block's keys at or above its threshold -------------
    // The prefetch list (spec_g) takes the keys above the threshold bin first
    // (fewer than the quota, so all of them fit): the block's selected groups
    // are its highest keys.
    const unsigned tj = unsigned(sv[3]);
    int cand_tot;
    {
        const int per = (nloc + kThreads - 1) / kThreads;
        const int i0 = min(nloc, tid * per), i1 = min(nloc, i0 + per);
        int nc = 0, na = 0;
        for (int i = i0; i < i1; ++i) {
            const unsigned k16 = score_key(score_at(i)) >> 16;
            nc += k16 >= tj;
            na += k16 > tj;
        }
        na = __reduce_add_sync(0xffffffffu, na);
        if (lane == 0 && na) atomicAdd(sv + 32, na);
        PHASE_MARK(5);
        int pos = block_exclusive_scan(nc, scratch, &cand_tot);  // (synchronises)
        const int n_above = sv[32];
        unsigned long long *slot = slots_cur + size_t(cta) * kSlotWords;
        // the header (count + 1, nonzero once written, and t_j) goes out first:
        // readers check every entry it announces for themselves
        if (tid == 0 && !(p.skip_arrive && j == n_b - 1 && n_b > 1)) {
            st_relaxed_u64(slot, (unsigned(cand_tot) + 1u) | ((unsigned long long)tj << 32));
            p.ovf[par * ncta + cta] = make_int2(int(seg + g_lo), max(0, cand_tot - kSlot));
        }
        for (int i = i0; i < i1; ++i) {
            const unsigned key = score_key(score_at(i));
            if ((key >> 16) >= tj) {
                const unsigned long long e = key | ((unsigned long long)(g_lo + i) << 32);
                if (pos < kSlot) st_relaxed_u64(slot + 1 + pos, e);
                else if (LCSW_INBOUNDS(pos - kSlot < nloc, 105))
                    st_relaxed_u64(cand_cur + seg + g_lo + pos - kSlot, e);
                const int sp = (key >> 16) > tj ? atomicAdd(sv + 33, 1)
                                                : n_above + atomicAdd(sv + 34, 1);
                if (sp < kChunk / P) spec_g[sp] = g_lo + i;
                ++pos;
            }
        }
    }
    __syncthreads();
    PHASE_MARK(7);
    if (p.skip_arrive && j == n_b - 1 && n_b > 1) {  // failure-detection test only
        return;
    }
    PHASE_MARK(8);

    // ---- prefetch: Q rows and this block's first candidate groups ------------------
    // They travel while the slots do; the attention uses them if the block's
    // selected groups are among them.
    using AL = AttLayout<DQK, DV>;
    using SL = SelLayout<DQK, DV>;
    static_assert(SL::end <= kUBytes, "selection overflows region U");
    const int spec_cap = kChunk / P;
    const int n_spec = min(cand_tot, spec_cap);
    const uint16_t *qrow = p.q + int64_t(b) * p.H_q * DQK;
    if (!p.select_only) {
        att_load_q<DQK, DV>(smem + kU, qrow, p.H_q);
        att_gather<DQK, DV>(smem + kU, gids, 0, spec_g, n_spec, G_b, P, Kb, Vb);
    }
    PHASE_MARK(9);

    // ---- exchange: every slot header of the sequence, then every candidate -------
    unsigned long long *hdrs = reinterpret_cast<unsigned long long *>(smem + SL::hdr);
    unsigned *ckey = reinterpret_cast<unsigned *>(smem + SL::key);
    int32_t *cgrp = reinterpret_cast<int32_t *>(smem + SL::grp);
    // packed (key << 32) | ~group, in the same bytes, when ranking own candidates
    unsigned long long *crank = reinterpret_cast<unsigned long long *>(smem + SL::key);
    {
        bool ok = true;
        if (tid < n_b) {  // one thread per slot polls its header (nonzero once written)
            const unsigned long long *hp = slots_cur + size_t(cb0 + tid) * kSlotWords;
            unsigned long long h = ld_relaxed_u64(hp);
            const long long t0 = clock64();
            for (int spin = 0; h == 0ull; ++spin) {
                if (clock64() - t0 > kSpinBudget ||
                    ((spin & 63) == 63 && aborted(p.abort_flag))) {
                    ok = false;
                    break;
                }
                __nanosleep(spin < 4 ? 64 : 256);
                h = ld_relaxed_u64(hp);
            }
            hdrs[tid] = h;
        }
        if (tid < kRankMax) rank[tid] = 0;
        if (__syncthreads_or(!ok)) {
            if (tid == 0) raise_timeout(p, 2);
            cp_async_wait<0>();
            return;
        }
    }
    PHASE_MARK(10);
    if (warp == 0) {
        // counts -> offsets (each lane owns up to 5 consecutive blocks);
        // T = the largest threshold of a block that published keys
        constexpr int kPer = (kMaxCtas + 31) / 32;
        int v[kPer];
        int s = 0;
        unsigned maxt = 0;
        int over = 0;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int jj = lane * kPer + u;
            v[u] = 0;
            if (jj < n_b) {
                const unsigned long long h = hdrs[jj];
                v[u] = int(unsigned(h)) - 1;
                if (v[u] > 0) maxt = max(maxt, unsigned(h >> 32));
                over |= v[u] > kSlot;
            }
            s += v[u];
        }
        int x = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        int run = x - s;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int jj = lane * kPer + u;
            if (jj < n_b) offs[jj] = run;
            run += v[u];
        }
        maxt = __reduce_max_sync(0xffffffffu, maxt);
        over = __reduce_or_sync(0xffffffffu, over);
        const int total = __shfl_sync(0xffffffffu, x, 31);
        if (lane == 0) {
            offs[n_b] = total;
            sv[6] = total;
            sv[7] = int(maxt);
            sv[9] = over;
        }
    }
    __syncthreads();
    const int n_cand = sv[6];
    const unsigned T = unsigned(sv[7]);
    bool fast = !p.force_slow && n_cand <= SelLayout<DQK, DV>::cap && n_cand >= k_b;
    // With at least k candidates at or above T, the candidates hold the true
    // top k; a block then only needs the rank of each of its own candidates
    // (keys descending, groups ascending), i.e. the order of the packed
    // value (key << 32) | ~group.  The k-th key K* is computed only for the
    // optional full index output or past 32 own candidates.
    const int own0 = offs[j], m_own = offs[j + 1] - offs[j];
    // (past 32 own candidates the K* path is cheaper: decode_b8, about 66 own
    // candidates a block, ran 8.6 us slower when ranking them all)
    const bool rank_fmt = fast && k_b > 0 && m_own <= kRankDirect && !(p.idx_out && j == 0);
    auto put_cand = [&](int o, unsigned key, unsigned g) {
        if (!LCSW_INBOUNDS((o >= 0 && o < SelLayout<DQK, DV>::cap), 101)) return;
        if (rank_fmt) {
            crank[o] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - g);
        } else {
            ckey[o] = key;
            cgrp[o] = int32_t(g);
        }
    };
    if (fast) {
        // every candidate, in slot order (= ascending group).  A thread loads all
        // of its entry words at once, then polls again only those not yet written.
        constexpr int kE = (kMaxCtas * kSlot + kThreads - 1) / kThreads;
        const long long t0 = clock64();
        bool ok = true;
        {
            unsigned long long w[kE];
            int dst[kE];
#pragma unroll
            for (int u = 0; u < kE; ++u) {
                const int q = tid + u * kThreads;
                dst[u] = -1;
                w[u] = 1ull;
                if (q < n_b * kSlot) {
                    const int jj = q / kSlot, e = q - jj * kSlot;
                    if (e < int(unsigned(hdrs[jj])) - 1) {
                        dst[u] = offs[jj] + e;
                        w[u] = ld_relaxed_u64(slots_cur + size_t(cb0 + jj) * kSlotWords + 1 + e);
                    }
                }
            }
            for (int spin = 0;; ++spin) {
                bool pend = false;
#pragma unroll
                for (int u = 0; u < kE; ++u) {
                    if (dst[u] < 0 || unsigned(w[u]) != 0u) continue;
                    pend = true;
                    const int q = tid + u * kThreads, jj = q / kSlot, e = q - jj * kSlot;
                    w[u] = ld_relaxed_u64(slots_cur + size_t(cb0 + jj) * kSlotWords + 1 + e);
                }
                if (!pend) break;
                if (clock64() - t0 > kSpinBudget ||
                    ((spin & 63) == 63 && aborted(p.abort_flag))) {
                    ok = false;
                    break;
                }
                __nanosleep(64);
            }
#pragma unroll
            for (int u = 0; u < kE; ++u)
                if (dst[u] >= 0) put_cand(dst[u], unsigned(w[u]), unsigned(w[u] >> 32));
        }
        if (sv[9]) {  // candidates past a slot's capacity come from the block's segment
            for (int jj = warp; jj < n_b; jj += kWarps) {
                const int cnt = int(unsigned(hdrs[jj])) - 1, o0 = offs[jj];
                const unsigned long long *s0 = cand_cur + seg + chunk_lo(jj) - kSlot;
                for (int e0 = kSlot; e0 < cnt; e0 += 4 * 32) {  // four words per lane at a time
                    unsigned long long w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e = e0 + lane + 32 * u;
                        w[u] = e < cnt ? ld_relaxed_u64(s0 + e) : 1ull;
                    }
                    for (int spin = 0; ok; ++spin) {
                        bool pend = false;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int e = e0 + lane + 32 * u;
                            if (e < cnt && unsigned(w[u]) == 0u) {
                                pend = true;
                                w[u] = ld_relaxed_u64(s0 + e);
                            }
                        }
                        if (!pend) break;
                        if (clock64() - t0 > kSpinBudget ||
                            ((spin & 63) == 63 && aborted(p.abort_flag))) ok = false;
                        __nanosleep(64);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e = e0 + lane + 32 * u;
                        if (e < cnt) put_cand(o0 + e, unsigned(w[u]), unsigned(w[u] >> 32));
                    }
                }
            }
        }
        if (!ok) {
            raise_timeout(p, 2);
            sv[19] = 1;
        }
    }
    __syncthreads();  // every candidate is in shared memory
    if (sv[19]) {  // a candidate never arrived
        cp_async_wait<0>();
        return;
    }
    // survivors (candidates at or above T) and, when ranking, the rank of each
    // own candidate: every thread takes candidates tid, tid + 512, ... and
    // counts, for each own candidate, how many of them rank above it
    if (fast) {
        constexpr int kEC = kSelCap / kThreads;  // candidates a thread holds per pass
        int ns = 0;
        if (rank_fmt) {
            for (int base = 0; base < n_cand; base += kSelCap) {  // one pass per kSelCap
                unsigned long long mine[kEC];
#pragma unroll
                for (int u = 0; u < kEC; ++u) {
                    const int i = base + tid + u * kThreads;
                    mine[u] = i < n_cand ? crank[i] : 0ull;
                    ns += i < n_cand && unsigned(mine[u] >> 48) >= T;
                }
                for (int o = 0; o < m_own; ++o) {
                    const unsigned long long rl = crank[own0 + o];
                    // below T a candidate is not selected (when the survivors
                    // are at least k) and outranks no survivor: skip it
                    if (unsigned(rl >> 48) < T) continue;  // warp-uniform
                    int cnt = 0;
#pragma unroll
                    for (int u = 0; u < kEC; ++u) cnt += mine[u] > rl;
                    cnt = __reduce_add_sync(0xffffffffu, cnt);
                    if (lane == 0 && cnt) atomicAdd(rank + o, cnt);
                }
            }
        } else {
            for (int i = tid; i < n_cand; i += kThreads) ns += (ckey[i] >> 16) >= T;
        }
        ns = __reduce_add_sync(0xffffffffu, ns);
        if (lane == 0 && ns) atomicAdd(sv + 31, ns);
        __syncthreads();
        fast = sv[31] >= k_b;
    }
    PHASE_MARK(11);
    const bool by_rank = rank_fmt && fast;
    int32_t *own = sel;
    int n_own = 0;
    bool use_spec = false;
    if (by_rank) {
        if (warp == 0) {
            // own candidates in rounds of 32, in slot (= ascending group) order
            int np = 0;
            for (int r0 = 0; r0 < m_own; r0 += 32) {
                const int o = r0 + lane;
                const unsigned long long rl = o < m_own ? crank[own0 + o] : ~0ull;
                const bool pick = o < m_own && unsigned(rl >> 48) >= T && rank[o] < k_b;
                const unsigned bsel = __ballot_sync(0xffffffffu, pick);
                const int grp = int(0xFFFFFFFFu - unsigned(rl));
                if (pick && LCSW_INBOUNDS(np + __popc(bsel) <= kRankMax, 102))
                    own[np + __popc(bsel & ((1u << lane) - 1u))] = grp;
                np += __popc(bsel);
            }
            if (lane == 0) sv[16] = np;
        }
        __syncthreads();
        n_own = sv[16];
    } else if (fast) {
        unsigned kth = 0xFFFFFFFFu, take_eq = 0;
        if (k_b > 0) {
            // K*, the k-th largest key: a histogram of the survivors' 16-bit
            // bins relative to T, then a rank count inside the bin (or a radix
            // select over the candidates when the bin is crowded)
            unsigned *sh = reinterpret_cast<unsigned *>(smem + SL::hist);
            for (int i = tid; i < 2048; i += kThreads) sh[i] = 0u;
            if (tid == 0) sv[10] = 0;
            __syncthreads();
            for (int i = tid; i < n_cand; i += kThreads) {
                const unsigned k16 = ckey[i] >> 16;
                if (k16 >= T) atomicAdd(sh + min(2047u, k16 - T), 1u);
            }
            __syncthreads();
            unsigned above;
            const int Tb = find_digit(sh, 2048, unsigned(k_b), &above, scratch, sv + 12);
            const unsigned need_t = unsigned(k_b) - above;
            const int m_t = int(sh[Tb]);
            if (Tb < 2047 && m_t <= kTieCap) {
                unsigned *tie = reinterpret_cast<unsigned *>(smem + SL::tie);
                for (int i = tid; i < n_cand; i += kThreads) {
                    const unsigned k16 = ckey[i] >> 16;
                    if (k16 >= T && k16 - T == unsigned(Tb)) {
                        const int s2 = atomicAdd(sv + 10, 1);
                        tie[2 * s2] = ckey[i];
                        tie[2 * s2 + 1] = unsigned(i);
                    }
                }
                __syncthreads();
                unsigned rk = 0, ke = 0;
                if (tid < m_t) {
                    ke = tie[2 * tid];
                    const unsigned ie = tie[2 * tid + 1];
                    for (int f = 0; f < m_t; ++f) {
                        const unsigned kf = tie[2 * f], jf = tie[2 * f + 1];
                        rk += kf > ke || (kf == ke && jf < ie);
                    }
                    if (rk == need_t - 1) sv[14] = int(ke);  // the k-th largest key
                }
                if (tid == 0) sv[15] = 0;
                __syncthreads();
                kth = unsigned(sv[14]);
                if (tid < m_t && ke == kth && rk < need_t) atomicAdd(sv + 15, 1);
                __syncthreads();
                take_eq = unsigned(sv[15]);
            } else {
                kth = radix_select_smem(ckey, n_cand, unsigned(k_b), sh, scratch, sv + 12,
                                        &take_eq);
            }
        }
        PHASE_MARK(12);
        // this block's selected groups, ascending: its candidates are the range
        // [offs[j], offs[j+1]); ties at K* go to the lowest candidate index
        const int o0 = offs[j], o1 = offs[j + 1];
        int eqb = 0;
        for (int i = tid; i < o0; i += kThreads) eqb += ckey[i] == kth;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) eqb += __shfl_xor_sync(0xffffffffu, eqb, o);
        if (lane == 0) scratch[warp] = eqb;
        __syncthreads();
        if (warp == 0) {
            int eqr = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) eqr += __shfl_xor_sync(0xffffffffu, eqr, o);
            int np = 0;
            for (int base = o0; base < o1; base += 32) {
                const int i = base + lane;
                const unsigned kk = i < o1 ? ckey[i] : 0u;
                const bool gt = i < o1 && kk > kth, eq = i < o1 && kk == kth;
                const unsigned beq = __ballot_sync(0xffffffffu, eq);
                const int eq_rank = eqr + __popc(beq & ((1u << lane) - 1u));
                const bool pick = gt || (eq && unsigned(eq_rank) < take_eq);
                const unsigned bsel = __ballot_sync(0xffffffffu, pick);
                if (pick && LCSW_INBOUNDS(np + __popc(bsel & ((1u << lane) - 1u)) < kMaxK, 102))
                    own[np + __popc(bsel & ((1u << lane) - 1u))] = cgrp[i];
                np += __popc(bsel);
                eqr += __popc(beq);
            }
            if (lane == 0) sv[16] = min(np, kMaxK);
        }
        __syncthreads();
        n_own = sv[16];
        PHASE_MARK(13);
        // the full ascending selection, for the optional index output
        if (p.idx_out && j == 0) {
            if (tid == 0) { sv[16] = 0; sv[17] = 0; }
            __syncthreads();
            for (int base = 0; base < n_cand; base += kThreads * 4) {
                unsigned kk[4];
                int ne = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = base + tid * 4 + e;
                    kk[e] = i < n_cand ? ckey[i] : 0u;
                    ne += (i < n_cand && kk[e] == kth);
                }
                const int eq_seen = sv[16], written = sv[17];
                int te;
                int eb = eq_seen + block_exclusive_scan(ne, scratch, &te);
                bool pick[4];
                int ns = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = base + tid * 4 + e;
                    bool keep = false;
                    if (i < n_cand) {
                        if (kk[e] > kth) keep = true;
                        else if (kk[e] == kth) keep = unsigned(eb++) < take_eq;
                    }
                    pick[e] = keep;
                    ns += keep;
                }
                int ts;
                int ps = written + block_exclusive_scan(ns, scratch, &ts);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (pick[e]) {
                        if (ps < k_b) p.idx_out[int64_t(b) * p.k + ps] = cgrp[base + tid * 4 + e];
                        ++ps;
                    }
                if (tid == 0) { sv[16] = eq_seen + te; sv[17] = written + ts; }
                __syncthreads();
            }
            for (int i = k_b + tid; i < p.k; i += kThreads) p.idx_out[int64_t(b) * p.k + i] = -1;
        }
        __syncthreads();
    }
    // The selected groups the prefetch holds stay in chunk buffer 0 as the
    // attention's first chunk; its other slots (prefetched groups not
    // selected, or never filled) take the first of the selected groups it
    // does not hold, and the rest follow in further chunks.  So the chunks
    // are as few as without the prefetch, and only the groups it missed are
    // gathered.
    if (fast && !p.select_only && n_spec > 0) {
        // (1) own[] keeps, in order, the selected groups the prefetch misses;
        // sv[36..37]: bits of the prefetch entries selected
        if (n_own <= 32) {
            if (warp == 0) {
                const int g = lane < n_own ? own[lane] : -1;
                int hit = -1;
                if (lane < n_own)
                    for (int s2 = 0; s2 < n_spec; ++s2) hit = spec_g[s2] == g ? s2 : hit;
                const unsigned keep = __ballot_sync(0xffffffffu, lane < n_own && hit < 0);
                const unsigned h_lo = __reduce_or_sync(0xffffffffu, hit >= 0 && hit < 32 ? 1u << hit : 0u);
                const unsigned h_hi = __reduce_or_sync(0xffffffffu, hit >= 32 ? 1u << (hit - 32) : 0u);
                if ((keep >> lane) & 1u) own[__popc(keep & ((1u << lane) - 1u))] = g;
                if (lane == 0) {
                    sv[36] = int(h_lo);
                    sv[37] = int(h_hi);
                    sv[16] = __popc(keep);
                }
            }
        } else {
            constexpr int kPer = kMaxK / kThreads;
            int gk[kPer];
            int n_keep = 0;
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int i = tid * kPer + e;
                gk[e] = -1;
                if (i < n_own) {
                    const int g = own[i];
                    int hit = -1;
                    for (int s2 = 0; s2 < n_spec; ++s2) hit = spec_g[s2] == g ? s2 : hit;
                    if (hit >= 0)
                        atomicOr(reinterpret_cast<unsigned *>(sv + 36 + (hit >> 5)), 1u << (hit & 31));
                    else gk[e] = g;
                    n_keep += hit < 0;
                }
            }
            int n_rest;
            int at = block_exclusive_scan(n_keep, scratch, &n_rest);  // (every own[] read is done)
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                if (gk[e] >= 0) own[at++] = gk[e];
            if (tid == 0) sv[16] = n_rest;
        }
        __syncthreads();
        const int n_rest = sv[16];
        use_spec = n_rest < n_own;
        if (use_spec) {
            // (2) buffer 0's free slots, in order, take own[0 .. n_fill)
            const unsigned long long taken =
                unsigned(sv[36]) | ((unsigned long long)unsigned(sv[37]) << 32);
            const unsigned long long slots = spec_cap == 64 ? ~0ull : (1ull << spec_cap) - 1ull;
            const unsigned long long freem = slots & ~taken;
            const int n_fill = min(n_rest, __popcll(freem));
            int *fslot = rank;  // free slot of own[q] (the rank counters are dead)
            if (tid < spec_cap && !((taken >> tid) & 1ull)) {
                const int q = __popcll(freem & ((1ull << tid) - 1ull));  // tid is free slot q
                const int g = q < n_fill ? own[q] : -1;
                gids[tid] = (g >= 0 && g < G_b) ? g : -1;  // else: masked
                if (q < n_fill) fslot[q] = tid;
            }
            if (n_fill > 0) {
                // the prefetch has landed before its slots are written again
                cp_async_wait<0>();
                __syncthreads();
                using AL = AttLayout<DQK, DV>;
                uint16_t *dk = reinterpret_cast<uint16_t *>(smem + kU + AL::buf);
                uint16_t *dv = dk + kChunk * AL::QP;
                constexpr int CK = DQK / 8, CV = DV / 8;
                const int lp2 = 31 - __clz(P);  // P is a power of two
                // token row r of the fill (group own[r / P]) goes to row
                // fslot[r / P] P + r % P of buffer 0; a warp a row
                for (int r = warp; r < n_fill * P; r += kWarps) {
                    const int q = r >> lp2, t = r & (P - 1);
                    const int g = own[q];
                    const bool ok = g >= 0 && g < G_b;
                    const int row = fslot[q] * P + t;
                    for (int c8 = lane; c8 < CK + CV; c8 += 32) {
                        if (c8 < CK)
                            cp_async16(smem_u32(dk + row * AL::QP + c8 * 8),
                                       ok ? Kb + (int64_t(g) * P + t) * DQK + c8 * 8 : Kb,
                                       ok ? 16 : 0);
                        else
                            cp_async16(smem_u32(dv + row * AL::VP + (c8 - CK) * 8),
                                       ok ? Vb + (int64_t(g) * P + t) * DV + (c8 - CK) * 8 : Vb,
                                       ok ? 16 : 0);
                    }
                }
                cp_async_commit();
            }
            own += n_fill;
            n_own = n_rest - n_fill;
        }
    }
    PHASE_MARK(14);
    DBG_ADD(0, fast && !by_rank);
    DBG_ADD(1, fast && !use_spec && n_own > 0);
    DBG_MAX(2, m_own);
    DBG_ADD(3, !fast);
    if (!fast) {
        cp_async_wait<0>();  // the prefetch lands before region U is reused
        __syncthreads();
        // ---------- exact multi-pass selection over the sequence's blocks ----------
        // level 1: the full 16-bit-bin histogram of every block's scores
        clear_smem(smem + kU, kUBytes);
        __syncthreads();
        for (int i = tid; i < nloc; i += kThreads) {
            const unsigned bin = score_key(score_at(i)) >> 16;
            atomicAdd(h16 + (bin >> 1), (bin & 1u) ? 0x10000u : 1u);
        }
        __syncthreads();
        flush_hist(h16, hist1);
        arrive(ctl + kSlowB);
        if (!wait_count(p, ctl + kSlowB, unsigned(n_b), 3, s_ok)) return;
        if (warp == 0) {
            unsigned above = 0;
            const int t1 = k_b > 0 ? hist_walk(hist1, unsigned(k_b), true, &above) : -1;
            if (lane == 0) { sv[20] = t1; sv[21] = int(above); }
        }
        __syncthreads();
        const int t1 = sv[20];
        const unsigned need2 = unsigned(k_b) - unsigned(sv[21]);
        // level 2: low 16 bits of the keys in the threshold bin
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
        if (!wait_count(p, ctl + kSlowC, unsigned(n_b), 4, s_ok)) return;
        if (warp == 0) {
            unsigned above = 0;
            const int lo = (k_b > 0 && t1 >= 0) ? hist_walk(hist2, need2, true, &above) : -1;
            if (lane == 0) { sv[22] = lo; sv[23] = int(above); }
        }
        __syncthreads();
        const bool none = k_b == 0 || t1 < 0 || sv[22] < 0;
        const unsigned kth = none ? 0xFFFFFFFFu : (unsigned(t1) << 16) | unsigned(sv[22]);
        const unsigned take_eq = none ? 0u : need2 - unsigned(sv[23]);
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
                p.cta_cnt[cta] = unsigned(tgt);
                p.cta_cnt[ncta + cta] = unsigned(teq);
            }
        }
        arrive(ctl + kSlowD);
        if (!wait_count(p, ctl + kSlowD, unsigned(n_b), 5, s_ok)) return;
        if (warp == 0) {
            // offsets of the blocks before this one: each takes its keys > K* and
            // the next ties in group order (blocks hold ascending group ranges)
            unsigned out_off = 0, eq_run = 0;
            for (int base = 0; base < j; base += 32) {
                const int jj = base + lane;
                const unsigned gtj = jj < j ? ld_cg(p.cta_cnt + cb0 + jj) : 0u;
                const unsigned eqj = jj < j ? ld_cg(p.cta_cnt + ncta + cb0 + jj) : 0u;
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
                sv[24] = int(out_off);
                sv[25] = int(take_eq > eq_run ? take_eq - eq_run : 0u);  // my ties to take
            }
        }
        __syncthreads();
        {
            int32_t *idx_list = p.idx_out ? p.idx_out : p.idx_ws;
            const int per = (nloc + kThreads - 1) / kThreads;
            const int i0 = min(nloc, tid * per), i1 = min(nloc, i0 + per);
            int n_eq = 0;
            for (int i = i0; i < i1; ++i) n_eq += score_key(score_at(i)) == kth;
            int tot;
            const int eq_start = block_exclusive_scan(n_eq, scratch, &tot);
            const unsigned my_take = unsigned(sv[25]);
            int eqr = eq_start, n_sel = 0;
            for (int i = i0; i < i1; ++i) {
                const unsigned key = score_key(score_at(i));
                n_sel += key > kth || (key == kth && unsigned(eqr++) < my_take);
            }
            int tsel;
            int lpos = block_exclusive_scan(n_sel, scratch, &tsel);
            int gpos = sv[24] + lpos;
            eqr = eq_start;
            for (int i = i0; i < i1; ++i) {
                const unsigned key = score_key(score_at(i));
                if (key > kth || (key == kth && unsigned(eqr++) < my_take)) {
                    if (lpos < kMaxK) sel[lpos] = g_lo + i;
                    if (gpos < k_b) idx_list[int64_t(b) * p.k + gpos] = g_lo + i;
                    ++lpos;
                    ++gpos;
                }
            }
            own = sel;
            n_own = min(tsel, kMaxK);
            if (j == 0)
                for (int i = k_b + tid; i < p.k; i += kThreads) idx_list[int64_t(b) * p.k + i] = -1;
        }
        // neither histogram is read by anyone any more: zero this block's slice of
        // the level-1 histogram, the level-2 fine bins it counted (still in shared
        // memory) and a slice of the level-2 coarse bins
        {
            const int w0 = int((long long)kHistWords / 4 * j / n_b) * 4;
            const int w1 = int((long long)kHistWords / 4 * (j + 1) / n_b) * 4;
            for (int w = w0 + tid * 4; w < w1; w += kThreads * 4)
                *reinterpret_cast<uint4 *>(hist1 + w) = make_uint4(0, 0, 0, 0);
            for (int w = tid; w < kFine / 2; w += kThreads) {
                const unsigned v = h16[w];
                if (v & 0xFFFFu) hist2[2 * w] = 0u;
                if (v >> 16) hist2[2 * w + 1] = 0u;
            }
            for (int cbin = int((long long)kCoarse * j / n_b) + tid;
                 cbin < int((long long)kCoarse * (j + 1) / n_b); cbin += kThreads)
                hist2[kFine + cbin] = 0u;
        }
        __syncthreads();
    }
    PHASE_MARK(15);

    if (!p.select_only) {
        // ---- attention over this block's selected groups ---------------------------
        attend_groups<DQK, DV>(smem + kU, gids, own, n_own, G_b, P, Kb, Vb, qrow, p.H_q, p.scale_log2,
                               p.part_o + int64_t(cta) * p.H_q * DV,
                               p.part_ml + int64_t(cta) * p.H_q, use_spec);
        PHASE_MARK(17);

        // ---- merge the partial states, head by head --------------------------------
        if (!merge_partials<DV>(p, smem, sv, sred, b, j, n_b, cb0)) return;
    }
    PHASE_MARK(19);
    __syncthreads();
    // this block's words of the other buffers were read during the previous
    // call: clear them for the next one
    {
        const int op = par ^ 1;
        if (tid < kSlotWords)
            st_relaxed_u64(p.slots + (size_t(op) * ncta + cta) * kSlotWords + tid, 0ull);
        unsigned long long *cold = p.cand + size_t(op) * p.B * p.G_max + ovf_old.x;
        for (int i = tid; i < ovf_old.y; i += kThreads) st_relaxed_u64(cold + i, 0ull);
    }
    // the last block of the grid to finish resets the counters and flips the
    // exchange buffers for the next call
    if (tid == 0 && atomicAdd(p.gdepart, 1u) == unsigned(ncta) - 1u) {
        for (int bb = 0; bb < B; ++bb)
            for (int i = 0; i < kNumCounters; ++i) p.ctl[size_t(bb) * kCtlWords + i] = 0u;
        *p.parity = unsigned(par ^ 1);
        *p.gdepart = 0u;
    }
}

// IndexCache reuse: the attention and merge phases of the fused step, over a
// selection an earlier layer made (p.idx_in [B][k]) instead of one of its own.
// Blocks go to sequences in proportion to their selected groups (one at
// least); block j of a sequence attends over entries [k j / n_b, k (j+1) / n_b)
// of its row (entries outside [0, G_b) are masked) and the blocks merge their
// partial states head by head as in the fused step.
template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1) reuse_decode_kernel(const Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    int *cta_begin = reinterpret_cast<int *>(smem + kMisc + 128);             // [kMaxCtas + 1]
    int *offs = cta_begin + kMaxCtas + 1;                                     // [kMaxCtas + 1]
    int *lens = offs + kMaxCtas + 1;                                          // [kMaxCtas]
    int *sv = lens + kMaxCtas;                                                // scalars [64]
    int *scratch = sv + 64;                                                   // [40]
    float *sred = reinterpret_cast<float *>(scratch + 40);                    // [64]
    int32_t *own = reinterpret_cast<int32_t *>(smem + kSelList);              // [kMaxK]
    const int tid = threadIdx.x;
    const int cta = blockIdx.x, ncta = gridDim.x;
    const int B = p.B, P = p.P;
    if (tid == 0) sv[19] = 0;
    int b, cb0, n_b, G_b;
    if (B == 1) {
        b = 0;
        cb0 = 0;
        n_b = ncta;
        G_b = __ldg(p.seq_len) / P;
    } else {
        if (tid < B) {
            const int L = __ldg(p.seq_len + tid);
            lens[tid] = L;
            offs[tid] = min(p.k, max(0, L / P)) + 1;
        }
        __syncthreads();
        assign_blocks(offs, B, ncta, cta_begin, scratch);
        for (int bb = tid; bb < B; bb += kThreads)
            if (cta_begin[bb] <= cta && cta < cta_begin[bb + 1]) sv[1] = bb;
        __syncthreads();
        b = sv[1];
        cb0 = cta_begin[b];
        n_b = cta_begin[b + 1] - cb0;
        G_b = lens[b] / P;
    }
    G_b = max(0, G_b);
    const int j = cta - cb0;
    const int lo = int((long long)p.k * j / n_b), hi = int((long long)p.k * (j + 1) / n_b);
    const int n_own = hi - lo;
    for (int i = tid; i < n_own; i += kThreads)
        if (LCSW_INBOUNDS(i < kMaxK, 106)) own[i] = __ldg(p.idx_in + int64_t(b) * p.k + lo + i);
    __syncthreads();
    attend_groups<DQK, DV>(smem + kU, reinterpret_cast<int *>(smem + kGids), own, n_own, G_b, P,
                           p.K + int64_t(b) * p.sK_b,
                           p.V + int64_t(b) * p.sV_b, p.q + int64_t(b) * p.H_q * DQK, p.H_q,
                           p.scale_log2, p.part_o + int64_t(cta) * p.H_q * DV,
                           p.part_ml + int64_t(cta) * p.H_q, false);
    merge_partials<DV>(p, smem, sv, sred, b, j, n_b, cb0);
}

int num_sms() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}


struct WsLayout {
    size_t ctl, hist, slots, cand, ovf, gscore, cta_cnt, idx_ws, part_o, part_ml, total;
};

// The partial-state regions come first and are sized for the largest shape
// (64 heads of 128 value dims), so every call on a workspace -- a decode step
// or a reuse step, whatever its G_max, H_q or d_v -- finds them at the same
// place; they hold only zeros between calls.
WsLayout ws_layout(int B, int G_max, int H_q, int d_v, int k, int ncta) {
    (void)H_q;
    (void)d_v;
    WsLayout w;
    size_t off = 256;  // status + abort words
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    w.part_ml = take(size_t(ncta) * 64 * 8);
    w.part_o = take(size_t(ncta) * 64 * 128 * 4);
    w.ctl = take(size_t(B) * kCtlWords * 4);
    w.hist = take(size_t(B) * 2 * kHistWords * 4);
    w.slots = take(size_t(2) * ncta * kSlotBytes);
    w.cand = take(size_t(2) * B * G_max * 8);
    w.ovf = take(size_t(2) * ncta * 8);
    w.gscore = take(size_t(B) * G_max * 4);
    w.cta_cnt = take(size_t(2) * ncta * 4);
    w.idx_ws = take(size_t(B) * k * 4);
    w.total = off;
    return w;
}

template <int NT, int DQK, int DV, bool F8>
cudaError_t launch_t(const Params &prm, int ncta, cudaStream_t st) {
    auto kern = fused_decode_kernel<NT, DQK, DV, F8>;
    constexpr int smem = kSmemBytes;
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

template <int DQK, int DV>
cudaError_t launch_reuse_t(const Params &prm, int ncta, cudaStream_t st) {
    auto kern = reuse_decode_kernel<DQK, DV>;
    constexpr int smem = kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
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

// Kernel parameters of one call (workspace regions carved by ws_layout).
Params make_params(const lcsw_decode_args *a, void *ws, int *status) {
    const int ncta = num_sms();
    const WsLayout w = ws_layout(a->B, a->G_max, a->H_q, a->d_v, a->k, ncta);
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
    prm.force_slow = (a->flags & LCSW_DECODE_FORCE_MULTIPASS_SELECT) ? 1 : 0;
    prm.skip_arrive = (a->flags & LCSW_DECODE_TEST_SKIP_ARRIVE) ? 1 : 0;
    prm.scale_log2 = a->scale * kLog2e;
    prm.out = a->out;
    prm.lse = a->lse;
    prm.idx_out = a->idx_out;
    prm.scores_out = a->scores_out;
    prm.ctl = reinterpret_cast<unsigned *>(base + w.ctl);
    prm.hist = reinterpret_cast<unsigned *>(base + w.hist);
    prm.slots = reinterpret_cast<unsigned long long *>(base + w.slots);
    prm.cand = reinterpret_cast<unsigned long long *>(base + w.cand);
    prm.ovf = reinterpret_cast<int2 *>(base + w.ovf);
    prm.gscore = reinterpret_cast<float *>(base + w.gscore);
    prm.cta_cnt = reinterpret_cast<unsigned *>(base + w.cta_cnt);
    prm.idx_ws = reinterpret_cast<int32_t *>(base + w.idx_ws);
    prm.part_o = reinterpret_cast<float *>(base + w.part_o);
    prm.part_ml = reinterpret_cast<float2 *>(base + w.part_ml);
    prm.status = status;
    prm.abort_flag = status + 1;
    prm.parity = reinterpret_cast<unsigned *>(status + 2);
    prm.gdepart = reinterpret_cast<unsigned *>(status + 3);
    prm.kq = nullptr;
    prm.sq_b = 0;
    prm.idx_in = nullptr;
    prm.select_only = 0;
    return prm;
}

// The kernel instantiation for the call's shape (NT head tiles of the indexer,
// d_qk, d_v); cudaErrorInvalidValue outside them.
template <bool F8>
cudaError_t launch_shape(const Params &prm, const lcsw_decode_args *a, cudaStream_t st) {
    const int ncta = num_sms();
    const int NT = a->H_i > 8 ? 2 : 1;
#define LCSW_FD(NTT, DQ, DVV)                                                         \
    if (NT == NTT && a->d_qk == DQ && a->d_v == DVV) return launch_t<NTT, DQ, DVV, F8>(prm, ncta, st);
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

cudaError_t launch_reuse_shape(const Params &prm, const lcsw_decode_args *a, cudaStream_t st) {
    const int ncta = num_sms();
#define LCSW_RD(DQ, DVV) \
    if (a->d_qk == DQ && a->d_v == DVV) return launch_reuse_t<DQ, DVV>(prm, ncta, st);
    LCSW_RD(128, 128)
    LCSW_RD(192, 128)
    LCSW_RD(64, 64)
    LCSW_RD(128, 64)
    LCSW_RD(192, 64)
    LCSW_RD(64, 128)
#undef LCSW_RD
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace lcsw
