// Persistent fused decode step: [append] -> indexer scores -> exact top-k
// groups -> sparse attention -> split-K combine, in one cooperative launch of
// one thread block per SM (the DSA retrieval chain of "G2C Brief --
// GLM-5.3-Flash", section "DSA keeps selected global access in eleven
// layers"; IndexPool from the reading notes, section 2).
//
// Work split.  Every sequence b gets a contiguous set of n_b >= 1 blocks,
// proportional to its number of pooled groups G_b; block j of the set owns a
// contiguous chunk of 16-group tiles.  Blocks exchange data (sample words,
// candidate slots, partial attention states) through words that are nonzero
// once written: a reader polls the data itself, with no fence or arrival
// counter.  Sample and candidate words are double-buffered by a per-call parity
// (each block clears its own words of the idle buffer); partial states are
// cleared by the one block that reads them.  Only the exact fallback selection
// syncs through arrival counters.  On a wait that runs out the block records
// LCSW_ERR_TIMEOUT in the workspace status word, raises an abort flag every
// other wait honours, and returns.
//
// Phase 1 (HBM stream).  All 16 warps stream their tiles' pooled keys
// straight into mma.sync A fragments (the k-permuted layout of
// index_scores.cu, two tile pairs in flight per warp) and keep the scores in
// shared memory.  The block that owns the group completed by the newest token
// pools it first (the exact arithmetic of the pooling kernel) and scores that
// fresh key.
//
// Threshold guess.  After its first tile pair every warp publishes, as one
// 64-bit word, the 16-bit bins of the four largest keys it has seen.  The words
// validate themselves (0 = not yet written), so no fence or counter is needed.
// Once done streaming, each block reads every sample word of its sequence and
// takes the bin where the count from the top reaches need ~ 1.5 k x (sample
// size)/G_b.  All blocks of a sequence compute the same guess.
//
// Selection.  Each block publishes its keys at or above the guess (a fixed
// slot, overflow to a per-sequence segment) and starts gathering its own
// candidates' K/V rows into shared memory.  After one sync point every block
// loads the candidates and selects the exact k-th key K* (a histogram relative
// to the guess, then a rank count inside the threshold bin).  If at least k
// keys cleared the guess and K* lies at or above it, the candidates hold the
// true top k and the selection is exact; every block then knows which of its
// own groups are selected.  Otherwise (a guess too high, or too many
// candidates) all blocks of the sequence run the exact multi-pass selection
// over their own scores: full level-1 histogram, level-2 histogram of the low
// 16 bits, per-block counts for the tie rule and the output order.
//
// Attention.  Each block attends over its own selected groups -- already in
// shared memory when they were among its prefetched candidates -- with the
// mma.sync online-softmax tile of attn_core.cuh, writes its partial (m, l, o)
// per head, and after a second sync point the blocks merge the partial states
// head by head.
#include "attn_core.cuh"
#include "common.cuh"
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
constexpr int kSpecTok = 64;       // tokens of own candidates prefetched into shared memory
constexpr int kTieCap = 256;       // threshold-bin candidates resolved by rank counting
constexpr int kMaxK = 2048;        // selected groups per sequence
constexpr int kCtlWords = 32;      // control words per sequence
constexpr int kMaxCtas = 160;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// control words (per sequence): arrival counters of the step's sync points,
// reset to zero by the last block to leave the kernel
constexpr int kSlowB = 1, kSlowC = 2, kSlowD = 3, kNumCounters = 4;
constexpr int kStream = kWarps;    // streaming warps
constexpr int kSampW = 4;          // sample bins each warp publishes (one 64-bit word)
constexpr int kSampleN = 2 * kStream * 16;  // sample: the first groups of each block's chunk
// Phase 1 streams the block's pooled keys through per-warp rings in shared
// memory filled by bulk copies: warp w scores tiles w, w + 16, w + 32, ... of
// the block's chunk (16 groups, 2 KB each) and keeps kRing of them in flight.
constexpr int kRing = 4;
constexpr int kTileBytes = 16 * 128;

// shared memory map (bytes); region U is reused phase by phase
constexpr int kU = 0;
constexpr int kUBytes = kFine * 2;                    // phase 1: 16-bit-pair histogram
constexpr int kSpec = kU;                             // prefetched own K/V [64 tok]
constexpr int kSpecBytes = kSpecTok * (192 + 8 + 128 + 8) * 2;
constexpr int kStage = kSpec + kSpecBytes;            // published slots [n_b][kSlotBytes]
constexpr int kCKey = kStage + kMaxCtas * kSlotBytes; // candidate keys [kSelCap]
constexpr int kCG = kCKey + kSelCap * 4;              // candidate groups [kSelCap]
constexpr int kSelHist = kCG + kSelCap * 4;           // [2048]
constexpr int kTie = kSelHist + 2048 * 4;             // [kTieCap] (key, index)
constexpr int kGather = kU;                           // gathered chunks (no prefetch hit)
constexpr int kSelG = kU + kUBytes - kMaxK * 4;       // own selected groups [kMaxK]
constexpr int kScores = kU + kUBytes;                 // [kChunkCap] floats
constexpr int kMisc = kScores + kChunkCap * 4;        // small arrays and scalars (< 8 KB)
constexpr int kQT = kMisc + 8192;                     // Q tile, tensor-core layout
// Attention operand tiles (128-byte-swizzled, see tc_core.cuh).  Q: K-major,
// DQK/64 atom columns of 64 head rows (8 KB each); the MMA reads 128 rows, so
// rows 64..127 of the last column fall on the 8 KB after the tile (values
// unused).  P: K-major, 128 head rows x 64 tokens (16 KB), on the scores,
// which are dead by then.  K: K-major, DQK/64 atom columns of 64 token rows.
// V: MN-major, DV/64 atoms of 8 token groups x 1024 B (LBO 8192 between atoms,
// SBO 1024 between token groups).
constexpr int kMiscBytes = 128 + kCoarse * 4 +
                           (2 * (kMaxCtas + 1) + kMaxCtas + 2 * kSpecTok + 64 + 40 + 64 +
                            2 * kChunk + 4 * 128) * 4 + 2 * 8 + 4;
static_assert(kMiscBytes <= 8192, "small arrays overflow their region");
template <int DQK> constexpr int q_tile_bytes() { return (DQK / 64) * 8192; }
template <int DQK, int DV> constexpr int kv_tile_bytes() { return (DQK / 64 + DV / 64) * 8192; }
constexpr int kPT = kScores;
static_assert(kTie + kTieCap * 8 <= kSelG, "shared-memory map overlap");
constexpr int kRingBase = kU;  // free while the keys stream
static_assert(kRingBase + kWarps * kRing * kTileBytes <= kU + kUBytes, "stream ring overlap");
// While the keys stream, the Q tile's region holds the newest group's staged
// rows ([8][64] bf16 + [8] weights), the guess histogram [2048] and the
// rings' mbarriers [kWarps][kRing] (invalidated before the Q tile lands).
constexpr int kNewRows = kQT;
constexpr int kGuessHist = kQT + 2048;
constexpr int kRingBars = kGuessHist + 2048 * 4;
static_assert(8 * 128 + 8 * 4 <= kGuessHist - kNewRows, "staged rows overlap");
static_assert(kRingBars + kWarps * kRing * 8 <= kQT + q_tile_bytes<64>() + 8192,
              "stream barriers overlap");
static_assert((192 / 64 + 128 / 64) * 8192 <= kSpecBytes, "prefetch tile overlap");
static_assert(kGather + 2 * (192 / 64 + 128 / 64) * 8192 <= kSelG, "gather overlap");

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
    int B, G_max, H_i, P, k, H_q, force_slow, skip_arrive;
    float scale_log2;
    uint16_t *out;
    float *lse;
    int32_t *idx_out;
    float *scores_out;
    // workspace
    unsigned *ctl;        // [B][kCtlWords]
    unsigned *hist;       // [B][2][kHistWords]: level 1, level 2 (zero between calls)
    // Exchange buffers, two of each: a call uses buffer `parity` and clears its
    // own words of the other one, which the next call uses.  Every word is
    // written once per call and is nonzero once written, so a reader polls the
    // data itself (no fence, no arrival counter).
    unsigned long long *samp;  // [2][ncta][kWarps]: each warp's sample bins
    unsigned long long *slots; // [2][ncta][kSlotWords]: (count+1 | guess<<32), (key | g<<32)...
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
#define PHASE_MARK(i)                                                    \
    do {                                                                 \
        if (threadIdx.x == 0) g_stamp[blockIdx.x][i] = (long long)globaltimer_ns();        \
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
__device__ __forceinline__ ulonglong2 ld_relaxed_u64x2(const unsigned long long *p) {
    ulonglong2 r;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(r.x), "=l"(r.y) : "l"(p));
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
__device__ __forceinline__ void st_part4(float *p, float4 v) {
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p),
                 "r"(__float_as_uint(v.x) ^ kPartTag), "r"(__float_as_uint(v.y) ^ kPartTag),
                 "r"(__float_as_uint(v.z) ^ kPartTag), "r"(__float_as_uint(v.w) ^ kPartTag)
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
__device__ __forceinline__ bool all_u16_nonzero(uint4 v) {
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) ok = ok && (w[i] & 0xFFFFu) != 0u && (w[i] >> 16) != 0u;
    return ok;
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

// Gather the K and V rows of one 64-token chunk -- the tokens of groups
// glist[0..n) (n <= 64/P) of a sequence whose complete groups are [0, G) --
// into the attention operand tiles (layouts above kv_tile_bytes).  Invalid
// or missing groups are zero-filled and marked -1 in sg.
template <int DQK, int DV>
__device__ __forceinline__ void gather_tc(unsigned char *tk, int *sg, const int32_t *glist, int n,
                                          int P, int G, const uint16_t *kb, const uint16_t *vb) {
    const int tid = threadIdx.x, lp2 = 31 - __clz(P), gpc = kChunk >> lp2;
    unsigned char *tv = tk + (DQK / 64) * 8192;
    if (tid < gpc) {
        const int g = tid < n ? glist[tid] : -1;
        sg[tid] = (g >= 0 && g < G) ? g : -1;
    }
    for (int e = tid; e < kChunk * (DQK / 8); e += kThreads) {
        const int t = e / (DQK / 8), c8 = e % (DQK / 8);
        const int q = t >> lp2;
        const int g = q < n ? glist[q] : -1;
        const bool ok = g >= 0 && g < G;
        const uint16_t *src = ok ? kb + (int64_t(g) * P + (t & (P - 1))) * DQK + c8 * 8 : kb;
        cp_async16(smem_u32(tk + (c8 / 8) * 8192 + sw128_offset(t, (c8 % 8) * 8, 1024)), src,
                   ok ? 16 : 0);
    }
    for (int e = tid; e < kChunk * (DV / 8); e += kThreads) {
        const int t = e / (DV / 8), c8 = e % (DV / 8);
        const int q = t >> lp2;
        const int g = q < n ? glist[q] : -1;
        const bool ok = g >= 0 && g < G;
        const uint16_t *src = ok ? vb + (int64_t(g) * P + (t & (P - 1))) * DV + c8 * 8 : vb;
        // MN-major: token t is row t%8 of token group t/8, dv chunk c8%8 of atom c8/8
        cp_async16(smem_u32(tv + (c8 / 8) * 8192 + sw128_offset(t, (c8 % 8) * 8, 1024)), src,
                   ok ? 16 : 0);
    }
    cp_async_commit();
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
    unsigned char *qt = smem + kQT;           // Q operand tile
    unsigned char *pt = smem + kPT;           // P operand tile (on the dead scores)
    uint16_t *newkey = reinterpret_cast<uint16_t *>(smem + kMisc);            // [64]
    unsigned *ccoarse = reinterpret_cast<unsigned *>(smem + kMisc + 128);     // [kCoarse]
    int *cta_begin = reinterpret_cast<int *>(ccoarse + kCoarse);              // [kMaxCtas + 1]
    int *offs = cta_begin + kMaxCtas + 1;                                     // [kMaxCtas + 1]
    int *lens = offs + kMaxCtas + 1;                                          // [kMaxCtas]
    int *spec_g = lens + kMaxCtas;                                            // [kSpecTok]
    int *spec_sg = spec_g + kSpecTok;                                         // [kSpecTok]
    int *sv = spec_sg + kSpecTok;                                             // scalars [64]
    int *scratch = sv + 64;                                                   // [40]
    float *sred = reinterpret_cast<float *>(scratch + 40);                    // [64]
    int *gsg = reinterpret_cast<int *>(sred + 64);                            // [2][kChunk]
    float *lpart = reinterpret_cast<float *>(gsg + 2 * kChunk);               // [4][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(lpart + 4 * 128);           // [2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 2);                 // TMEM base

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x, ncta = gridDim.x;
    const int B = p.B, P = p.P;
    PHASE_MARK(0);
    // the operand tiles' swizzle assumes 1024-byte-aligned shared memory
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, int(LCSW_ERR_UNSUPPORTED) * 256);
        return;
    }
    // this call's exchange buffers (the previous call's last block flipped it)
    const int par = int(ld_cg(p.parity) & 1u);
    unsigned long long *samp_cur = p.samp + size_t(par) * ncta * kWarps;
    unsigned long long *slots_cur = p.slots + size_t(par) * ncta * kSlotWords;
    unsigned long long *cand_cur = p.cand + size_t(par) * p.B * p.G_max;
    // where this block's overflow entries went in the previous call (cleared at
    // the end of this one)
    const int2 ovf_old = p.ovf[(par ^ 1) * ncta + cta];

    // ---- roles: blocks per sequence, proportional to its groups --------------
    int b, cb0, n_b, L_b, G_b;
    if (B == 1) {
        L_b = __ldg(p.seq_len);
        G_b = L_b / P;
        G_b = G_b < 0 ? 0 : (G_b > p.G_max ? p.G_max : G_b);
        b = 0;
        cb0 = 0;
        n_b = ncta;
        if (tid == 0) { sv[19] = 0; sv[26] = 0; sv[27] = 0; }
        __syncthreads();
    } else {
        int gv = 0;
        if (tid < B) {
            const int L = __ldg(p.seq_len + tid);
            lens[tid] = L;
            int G = L / P;
            gv = G < 0 ? 0 : (G > p.G_max ? p.G_max : G);
        }
        if (tid == 0) { sv[19] = 0; sv[26] = 0; sv[27] = 0; }
        int total;
        const int pre = block_exclusive_scan(gv, scratch, &total);
        if (tid < B) offs[tid] = pre;
        if (tid == 0) offs[B] = total;
        __syncthreads();
        const double tot = total > 0 ? double(total) : 1.0;
        for (int bb = tid; bb <= B; bb += kThreads)
            cta_begin[bb] = bb == B ? ncta : bb + int(double(ncta - B) * double(offs[bb]) / tot);
        __syncthreads();
        for (int bb = tid; bb < B; bb += kThreads)
            if (cta_begin[bb] <= cta && cta < cta_begin[bb + 1]) sv[1] = bb;
        __syncthreads();
        b = sv[1];
        cb0 = cta_begin[b];
        n_b = cta_begin[b + 1] - cb0;
        L_b = lens[b];
        G_b = offs[b + 1] - offs[b];
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
    // warp issues the warp's first kRing tiles now, so the prologue's own loads
    // overlap them, and refills a slot as soon as the warp has read it.
    const int r = lane >> 2, c = lane & 3;
    const uint16_t *kb = p.k_pooled + int64_t(b) * p.sp_b;
    const int n_tiles = (nloc + 15) / 16;
    const int n_mine = n_tiles > warp ? (n_tiles - warp + kStream - 1) / kStream : 0;
    unsigned char *ring = smem + kRingBase + warp * kRing * kTileBytes;
    uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + kRingBars) + warp * kRing;
    int n_issued = 0;  // lane 0: tiles of this warp issued so far
    auto issue_tile = [&](int kk) {  // lane 0: this warp's tile kk into slot kk % kRing
        const int g0 = g_lo + (warp + kk * kStream) * 16;
        const uint32_t bytes = uint32_t(min(16, g_hi - g0)) * 128u;
        mbar_expect_tx(wbar + kk % kRing, bytes);
        bulk_load(ring + (kk % kRing) * kTileBytes, kb + int64_t(g0) * 64, bytes, wbar + kk % kRing);
        ++n_issued;
    };
    if (lane == 0) {
        for (int i = 0; i < kRing; ++i) mbar_init(wbar + i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int kk = 0; kk < min(kRing, n_mine); ++kk) issue_tile(kk);
    }

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

    PHASE_MARK(23);
    // append: the group the newest token completes is pooled by the warp
    // whose tile holds it, just before it scores that tile, from rows staged
    // here (the Q tile's region is free until the candidates are known)
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
    PHASE_MARK(24);
    // total sample size of the sequence (the chunk split is known to every
    // block; tiles_b * n_b < 2^32 within the supported sizes)
    if (tid < n_b) {
        const int lo = 16 * int(unsigned(tiles_b) * unsigned(tid) / unsigned(n_b));
        const int hi = min(G_b, 16 * int(unsigned(tiles_b) * unsigned(tid + 1) / unsigned(n_b)));
        atomicAdd(sv + 26, min(max(hi - lo, 0), kSampleN));
    }
    __syncthreads();
    PHASE_MARK(2);

    // ---- phase 1: stream pooled keys, score, histogram -------------------------
    auto score_tile = [&](int t, uint4 (&A)[4]) -> unsigned {
        const int ga = g_lo + t * 16 + r, gb = ga + 8;
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
        const int li = t * 16 + r + 8 * c;
        const bool mine = c < 2 && g_lo + li < g_hi;
        const float sc = __fadd_rn(c == 0 ? pa : pb, 0.0f);
        if (mine) {
            if (li < kChunkCap) sscore[li] = sc;
            else p.gscore[seg + g_lo + li] = sc;
            if (p.scores_out) p.scores_out[seg + g_lo + li] = sc;
        }
        return mine ? score_key(sc) >> 16 : 0u;
    };
    // Sample: every warp publishes the bins of the kSampW largest keys of its
    // first two tiles as one 64-bit word of 16-bit entries (a finite score's
    // bin is at least 0x007F; 1 = no key; 0 = not yet written).  The words are
    // self-validating, so readers need no fence or arrival counter.
    auto publish_sample = [&](unsigned ka, unsigned kc) {
        unsigned long long word = 0;
#pragma unroll
        for (int e = 0; e < kSampW; ++e) {
            const unsigned wm = __reduce_max_sync(0xffffffffu, max(ka, kc));
            const unsigned hit = __ballot_sync(0xffffffffu, ka == wm || kc == wm);
            if (lane == __ffs(hit) - 1) {
                if (ka == wm) ka = 0u;
                else kc = 0u;
            }
            word |= (unsigned long long)max(wm, 1u) << (16 * e);
        }
        if (lane == 0) st_relaxed_u64(samp_cur + size_t(cta) * kWarps + warp, word);
    };
    // The guess: the need-th largest published bin of the sequence, need ~
    // 1.5 k x (sample size)/G.  It is only a guess: the selection checks that
    // at least k keys cleared it.  Each thread loads its share of the
    // sequence's sample words (polling until every entry is written), then the
    // block counts the entries in 2048 bins below the largest one and picks
    // the bin where the count from the top reaches need.  It runs
    // once the block is done streaming.  Returns false (block-uniform) if a
    // stage or the sample never completed.
    auto make_guess = [&]() -> bool {
        constexpr int kQ16 = (kMaxCtas * kWarps / 2 + kThreads - 1) / kThreads;
        const int n_q = n_b * kWarps / 2;  // 16-byte chunks of entries
        uint4 v[kQ16];
        unsigned emax = 1;
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(samp_cur + size_t(cb0) * kWarps);
#pragma unroll
            for (int u = 0; u < kQ16; ++u)
                if (tid + u * kThreads < n_q) v[u] = ld_relaxed_v4(src + tid + u * kThreads);
            const long long t0 = clock64();
            bool ok = true;
#pragma unroll
            for (int u = 0; u < kQ16; ++u) {
                const int q = tid + u * kThreads;
                if (q >= n_q) break;
                for (int spin = 0; ok && !all_u16_nonzero(v[u]); ++spin) {
                    if (clock64() - t0 > kSpinBudget ||
                        ((spin & 63) == 63 && aborted(p.abort_flag))) {
                        ok = false;
                        break;
                    }
                    __nanosleep(64);
                    v[u] = ld_relaxed_v4(src + q);
                }
                const unsigned w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) emax = max(emax, max(w[e] & 0xFFFFu, w[e] >> 16));
            }
            if (!ok) {
                raise_timeout(p, 1);
                sv[19] = 1;
            }
            emax = __reduce_max_sync(0xffffffffu, emax);
            if (lane == 0) atomicMax(sv + 27, int(emax));
        }
        // warps zero it while others may still read the ring: it lies outside
        // the ring, in the Q tile's region (free until the candidates are known)
        unsigned *sh = reinterpret_cast<unsigned *>(smem + kGuessHist);
        for (int i = tid; i < 2048; i += kThreads) sh[i] = 0u;
        __syncthreads();
        PHASE_MARK(20);
        if (sv[19]) return false;
        int sguess = 0;
        const unsigned need = unsigned(
            max(1ull, (3ull * unsigned(k_b) * unsigned(sv[26]) + 2ull * G_b - 1) / (2ull * G_b)));
        if (k_b > 0 && n_b > 1 && need <= unsigned(n_q * 8)) {
            const unsigned base = unsigned(max(0, sv[27] - 2047));
#pragma unroll
            for (int u = 0; u < kQ16; ++u) {
                if (tid + u * kThreads >= n_q) break;
                const unsigned w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    atomicAdd(sh + (max(w[e] & 0xFFFFu, base) - base), 1u);
                    atomicAdd(sh + (max(w[e] >> 16, base) - base), 1u);
                }
            }
            __syncthreads();
            PHASE_MARK(21);
            unsigned above = 0;
            sguess = int(base) + find_digit(sh, 2048, need, &above, scratch, sv + 12);
            PHASE_MARK(22);
        }
        if (tid == 0) sv[3] = sguess;
        return true;
    };
    // Warp w scores its tiles in order; its sample is its first two tiles.  A
    // tile that never lands stops the warp's work but not its barriers.
    unsigned key0 = 0u;
    bool stream_ok = true;
    for (int kk = 0; kk < n_mine; ++kk) {
        const int slot = kk % kRing, t = warp + kk * kStream;
        if (stream_ok &&
            !__all_sync(0xffffffffu, mbar_wait(wbar + slot, unsigned(kk / kRing) & 1u, kWaitNs))) {
            stream_ok = false;  // warp-uniform: score_tile shuffles across the warp
            raise_timeout(p, 7);
            sv[19] = 1;
        }
        if (t == t_new) {  // this warp pools the newest group before scoring its tile
            cp_async_wait<0>();
            __syncwarp();
            pool_staged(P, krows, kw, lane, newkey, p.k_pooled + int64_t(b) * p.sp_b + int64_t(g_new) * 64);
            __syncwarp();
        }
        unsigned key = 0u;
        if (stream_ok) {
            const unsigned char *tile = ring + slot * kTileBytes;
            uint4 A[4];
            A[0] = *reinterpret_cast<const uint4 *>(tile + r * 128 + 16 * c);
            A[1] = *reinterpret_cast<const uint4 *>(tile + r * 128 + 64 + 16 * c);
            A[2] = *reinterpret_cast<const uint4 *>(tile + (r + 8) * 128 + 16 * c);
            A[3] = *reinterpret_cast<const uint4 *>(tile + (r + 8) * 128 + 64 + 16 * c);
            key = score_tile(t, A);
        }
        __syncwarp();
        if (lane == 0 && stream_ok && kk + kRing < n_mine) {
            fence_async_smem();  // the warp's reads of the slot come before the copy
            issue_tile(kk + kRing);
        }
        if (kk == 0) key0 = key;
        if (kk == 1) publish_sample(key0, key);
    }
    if (n_mine < 2) publish_sample(key0, 0u);
    if (lane == 0) {
        if (stream_ok) {  // every copy landed: retire the barriers (the Q tile goes there)
            for (int i = 0; i < kRing; ++i)
                asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(wbar + i))
                             : "memory");
        } else {  // the copies in flight land before the block leaves or reuses the ring
            for (int kk = max(0, n_issued - kRing); kk < n_issued; ++kk)
                mbar_wait(wbar + kk % kRing, unsigned(kk / kRing) & 1u, kWaitNs);
        }
    }
    PHASE_MARK(4);
    if (!make_guess()) return;
    if (p.scores_out && j == 0)  // -inf past the last complete group: the full row
        for (int g = G_b + tid; g < p.G_max; g += kThreads) p.scores_out[seg + g] = -INFINITY;
    __syncthreads();
    PHASE_MARK(3);
    auto score_at = [&](int li) -> float {
        return li < kChunkCap ? sscore[li] : ld_cg_f(p.gscore + seg + g_lo + li);
    };

    // ---- candidates: this block's keys at or above the guess --------------------
    const int spec_cap = kSpecTok / P;
    const unsigned guess = unsigned(sv[3]);
    {
        const int per = (nloc + kThreads - 1) / kThreads;
        const int i0 = min(nloc, tid * per), i1 = min(nloc, i0 + per);
        int nc = 0;
        for (int i = i0; i < i1; ++i) nc += (score_key(score_at(i)) >> 16) >= guess;
        PHASE_MARK(5);
        int tot;
        int pos = block_exclusive_scan(nc, scratch, &tot);
        PHASE_MARK(6);
        unsigned long long *slot = slots_cur + size_t(cta) * kSlotWords;
        for (int i = i0; i < i1; ++i) {
            const unsigned key = score_key(score_at(i));
            if ((key >> 16) >= guess) {
                const unsigned long long e = key | ((unsigned long long)(g_lo + i) << 32);
                if (pos < kSlot) st_relaxed_u64(slot + 1 + pos, e);
                else st_relaxed_u64(cand_cur + seg + g_lo + pos - kSlot, e);
                if (pos < spec_cap) spec_g[pos] = g_lo + i;
                ++pos;
            }
        }
        PHASE_MARK(7);
        if (tid == 0) {
            sv[5] = min(tot, spec_cap);  // prefetched groups (the first ones)
            sv[28] = tot;
        }
    }
    __syncthreads();
    PHASE_MARK(8);
    const int n_spec = sv[5];
    if (p.skip_arrive && j == n_b - 1 && n_b > 1) {  // failure-detection test only
        return;
    }
    if (tid == 0) {  // the header: count + 1 (nonzero once written) and the guess
        st_relaxed_u64(slots_cur + size_t(cta) * kSlotWords,
                       (unsigned(sv[28]) + 1u) | ((unsigned long long)guess << 32));
        p.ovf[par * ncta + cta] = make_int2(int(seg + g_lo), max(0, sv[28] - kSlot));
    }
    // prefetch this block's candidates' K/V and the heads' Q into operand tiles
    auto load_q_tile = [&]() {
        const uint16_t *qrow = p.q + int64_t(b) * p.H_q * DQK;
        for (int e = tid; e < p.H_q * (DQK / 8); e += kThreads) {
            const int h = e / (DQK / 8), c8 = e % (DQK / 8);
            cp_async16(smem_u32(qt + (c8 / 8) * 8192 + sw128_offset(h, (c8 % 8) * 8, 1024)),
                       qrow + int64_t(h) * DQK + c8 * 8, 16);
        }
        cp_async_commit();
    };
    gather_tc<DQK, DV>(smem + kSpec, spec_sg, spec_g, n_spec, P, G_b, Kb, Vb);
    load_q_tile();
    PHASE_MARK(9);

    // ---- selection: exact top k from the published candidates -----------------
    // Load every slot of the sequence into shared memory, polling until the
    // header and the entries it announces are written.
    unsigned char *stage = smem + kStage;
    {
        constexpr int kC = kSlotBytes / 16;  // 16-byte chunks per slot
        constexpr int kQ = (kMaxCtas * kC + kThreads - 1) / kThreads;
        const int n16 = n_b * kC;
        const unsigned long long *src = slots_cur + size_t(cb0) * kSlotWords;
        unsigned pend = 0;  // chunks still to load, bit u <-> chunk tid + u*kThreads
#pragma unroll
        for (int u = 0; u < kQ; ++u)
            if (tid + u * kThreads < n16) pend |= 1u << u;
        const long long t0 = clock64();
        for (int spin = 0;; ++spin) {
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                if (!(pend >> u & 1u)) continue;
                const int q = tid + u * kThreads;
                reinterpret_cast<ulonglong2 *>(stage)[q] = ld_relaxed_u64x2(src + 2 * q);
            }
            __syncthreads();
            // a chunk is complete once its slot's header is written and so is
            // every entry the header announces
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                if (!(pend >> u & 1u)) continue;
                const int q = tid + u * kThreads;
                const int jj = q / kC, w0 = 2 * (q % kC);
                const unsigned long long *sl =
                    reinterpret_cast<const unsigned long long *>(stage) + jj * kSlotWords;
                const unsigned h = unsigned(sl[0]);
                bool ok = h != 0u;
                if (ok) {
                    const int nw = 1 + min(int(h) - 1, kSlot);
#pragma unroll
                    for (int w = 0; w < 2; ++w)
                        if (w0 + w < nw && unsigned(sl[w0 + w]) == 0u) ok = false;
                }
                if (ok) pend &= ~(1u << u);
            }
            if (!__syncthreads_or(pend != 0u)) break;
            // thread 0 decides for the block whether to give up
            const bool give_up = tid == 0 && (clock64() - t0 > kSpinBudget ||
                                              ((spin & 63) == 63 && aborted(p.abort_flag)));
            if (__syncthreads_or(give_up)) {
                if (tid == 0) raise_timeout(p, 2);
                cp_async_wait<0>();
                return;
            }
            __nanosleep(64);
        }
    }
    PHASE_MARK(10);
    // Speculative S = Q K^T over this block's prefetched candidates, issued by
    // the last warp while the block ranks its candidates (the softmax masks the
    // ones not selected).  TMEM is held from here to the end of the attention;
    // every exit on the way frees it.
    cp_async_wait<0>();
    fence_async_smem();
    if (tid == 0) {
        mbar_init(bars, 1);      // S ready
        mbar_init(bars + 1, 1);  // O_c ready
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;  // S: columns 0..63, O_c: 64..64+DV
    auto release_tmem = [&]() {  // uniform: every thread of the block
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_free(tb, 256);
    };
    constexpr int kMmaWarp = kWarps - 1;  // issues the tensor-core work
    auto issue_s = [&](const unsigned char *tk) {
        if (warp == kMmaWarp) {
            const uint32_t id = idesc_bf16_f32(128, 64, false, false);
            const uint32_t qa = smem_u32(qt), ka = smem_u32(tk);
            if (elect_one()) {
#pragma unroll
                for (int ks = 0; ks < DQK / 16; ++ks) {
                    const uint32_t ko = (ks / 4) * 8192 + (ks % 4) * 32;
                    tc_mma_bf16(tb, smem_desc(qa + ko, 16, 1024), smem_desc(ka + ko, 16, 1024), id,
                                ks > 0);
                }
                tc_commit(bars);
            }
            __syncwarp();
        }
    };
    int n_s = 0;  // S products committed so far (phases of bars[0])
    if (n_spec > 0) {
        issue_s(smem + kSpec);
        n_s = 1;
    }
    // slot jj as 32-bit words: [0] count + 1, [1] guess, [2 + 2e] key, [3 + 2e] group
    auto hdr = [&](int jj) { return reinterpret_cast<const unsigned *>(stage + jj * kSlotBytes); };
    if (warp == 0) {
        // counts -> offsets (each lane owns up to 5 consecutive blocks)
        constexpr int kPer = (kMaxCtas + 31) / 32;
        int v[kPer];
        int s = 0;
        unsigned minp = kFine, maxp = 0;
        int over = 0;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int jj = lane * kPer + u;
            v[u] = 0;
            if (jj < n_b) {
                const unsigned *h = hdr(jj);
                v[u] = int(h[0]) - 1;
                minp = min(minp, h[1]);
                maxp = max(maxp, h[1]);
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
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            minp = min(minp, __shfl_xor_sync(0xffffffffu, minp, o));
            maxp = max(maxp, __shfl_xor_sync(0xffffffffu, maxp, o));
            over |= __shfl_xor_sync(0xffffffffu, over, o);
        }
        const int total = __shfl_sync(0xffffffffu, x, 31);
        if (lane == 0) {
            offs[n_b] = total;
            sv[6] = total;
            sv[7] = int(maxp);
            sv[8] = int(minp);
            sv[9] = over;
        }
    }
    __syncthreads();
    const int n_cand = sv[6];
    const unsigned maxguess = unsigned(sv[7]);
    bool fast = !p.force_slow && n_cand <= kSelCap && n_cand >= k_b;
    unsigned kth = 0xFFFFFFFFu, take_eq = 0;
    unsigned *ckey = reinterpret_cast<unsigned *>(smem + kCKey);
    int32_t *cgrp = reinterpret_cast<int32_t *>(smem + kCG);
    DBG_MAX(0, n_cand);
    // With one common guess and at least k candidates, the candidates hold the
    // true top k; a block then only needs the rank of each of its own
    // candidates (keys descending, groups ascending), here the order of the
    // packed value (key << 32) | ~group.  The k-th key K* is computed only for
    // the optional full index output or past 32 own candidates.
    const int own0 = offs[j], m_own = offs[j + 1] - offs[j];
    const bool by_rank = fast && k_b > 0 && m_own <= 32 && sv[8] == sv[7] && !(p.idx_out && j == 0);
    // packed candidates on the scores, which the rank path no longer needs
    unsigned long long *crank = reinterpret_cast<unsigned long long *>(smem + kScores);
    int *rank = reinterpret_cast<int *>(lpart);  // [32] ranks of the own candidates
    auto put_cand = [&](int o, unsigned key, unsigned g) {
        if (by_rank) {
            crank[o] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - g);
        } else {
            ckey[o] = key;
            cgrp[o] = int32_t(g);
        }
    };
    if (fast) {
        if (tid < 32) rank[tid] = 0;
        // all candidates, in slot order (= ascending group): one thread per slot entry
        for (int q = tid; q < n_b * kSlot; q += kThreads) {
            const int jj = q / kSlot, e = q - jj * kSlot;
            const unsigned *h = hdr(jj);
            if (e < int(h[0]) - 1) put_cand(offs[jj] + e, h[2 + 2 * e], h[3 + 2 * e]);
        }
        if (sv[9]) {  // candidates past a slot's capacity come from the block's segment
            const long long t0 = clock64();
            bool ok = true;
            for (int jj = warp; jj < n_b; jj += kWarps) {
                const int cnt = int(hdr(jj)[0]) - 1, o0 = offs[jj];
                const unsigned long long *s0 = cand_cur + seg + chunk_lo(jj) - kSlot;
                for (int e = kSlot + lane; e < cnt; e += 32) {
                    unsigned long long w = ld_relaxed_u64(s0 + e);
                    for (int spin = 0; unsigned(w) == 0u && ok; ++spin) {
                        if (clock64() - t0 > kSpinBudget ||
                            ((spin & 63) == 63 && aborted(p.abort_flag))) ok = false;
                        __nanosleep(64);
                        w = ld_relaxed_u64(s0 + e);
                    }
                    put_cand(o0 + e, unsigned(w), unsigned(w >> 32));
                }
            }
            if (!ok) {
                raise_timeout(p, 2);
                sv[19] = 1;
            }
        }
        __syncthreads();
        PHASE_MARK(11);
        if (sv[19]) {  // an overflow entry never arrived
            release_tmem();
            return;
        }
    }
    if (fast && !by_rank) {
        if (k_b > 0) {
            // histogram of the 16-bit bin relative to the smallest guess
            unsigned *sh = reinterpret_cast<unsigned *>(smem + kSelHist);
            const unsigned minp = unsigned(sv[8]);
            for (int i = tid; i < 2048; i += kThreads) sh[i] = 0u;
            if (tid == 0) sv[10] = 0;
            __syncthreads();
            for (int i = tid; i < n_cand; i += kThreads)
                atomicAdd(sh + min(2047u, (ckey[i] >> 16) - minp), 1u);
            __syncthreads();
            unsigned above;
            PHASE_MARK(28);
            const int T = find_digit(sh, 2048, unsigned(k_b), &above, scratch, sv + 12);
            PHASE_MARK(29);
            const unsigned need_t = unsigned(k_b) - above;
            const int m_t = int(sh[T]);
            if (T < 2047 && m_t <= kTieCap) {
                unsigned *tie = reinterpret_cast<unsigned *>(smem + kTie);
                for (int i = tid; i < n_cand; i += kThreads) {
                    if (min(2047u, (ckey[i] >> 16) - minp) == unsigned(T)) {
                        const int s = atomicAdd(sv + 10, 1);
                        tie[2 * s] = ckey[i];
                        tie[2 * s + 1] = unsigned(i);
                    }
                }
                __syncthreads();
                unsigned rank = 0, ke = 0;
                if (tid < m_t) {
                    ke = tie[2 * tid];
                    const unsigned ie = tie[2 * tid + 1];
                    for (int f = 0; f < m_t; ++f) {
                        const unsigned kf = tie[2 * f], jf = tie[2 * f + 1];
                        rank += kf > ke || (kf == ke && jf < ie);
                    }
                    if (rank == need_t - 1) sv[14] = int(ke);  // the k-th largest key
                }
                if (tid == 0) sv[15] = 0;
                __syncthreads();
                kth = unsigned(sv[14]);
                if (tid < m_t && ke == kth && rank < need_t) atomicAdd(sv + 15, 1);
                __syncthreads();
                take_eq = unsigned(sv[15]);
            } else {
                kth = radix_select_smem(ckey, n_cand, unsigned(k_b), sh, scratch, sv + 12,
                                        &take_eq);
            }
            // exact iff every block's guess was at or below K*: then every key a
            // block left out is below K* and cannot be in the top k
            fast = (kth >> 16) >= maxguess;
        }
    }
    PHASE_MARK(12);
    int32_t *own = reinterpret_cast<int32_t *>(smem + kSelG);
    int n_own = 0;
    bool use_spec = false;
    if (by_rank) {
        // rank of each own candidate: lane l of every warp holds own candidate l;
        // warp w counts the candidates of its slice that rank above it
        const unsigned long long rl = lane < m_own ? crank[own0 + lane] : ~0ull;
        const int per = (n_cand + kWarps - 1) / kWarps;
        const int e0 = warp * per, e1 = min(n_cand, e0 + per);
        unsigned cnt = 0;
#pragma unroll 8
        for (int e = e0; e < e1; ++e) cnt += crank[e] > rl ? 1u : 0u;
        if (lane < m_own && cnt) atomicAdd(rank + lane, int(cnt));
        __syncthreads();
        if (warp == 0) {
            const bool sel = lane < m_own && rank[lane] < k_b;
            const unsigned bsel = __ballot_sync(0xffffffffu, sel);
            if (sel) own[__popc(bsel & ((1u << lane) - 1u))] = int(0xFFFFFFFFu - unsigned(rl));
            // the prefetch holds this block's first n_spec candidates
            const bool cover = n_spec >= 32 || (bsel >> n_spec) == 0u;
            if (lane == 0) {
                sv[16] = __popc(bsel);
                sv[18] = cover ? 1 : 0;
            }
        }
        __syncthreads();
        n_own = sv[16];
        use_spec = sv[18] != 0;
        if (use_spec && tid < spec_cap && !(tid < m_own && rank[tid] < k_b))
            spec_sg[tid] = -1;  // prefetched but not selected: masked
    } else if (fast) {
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
                const bool sel = gt || (eq && unsigned(eq_rank) < take_eq);
                const unsigned bsel = __ballot_sync(0xffffffffu, sel);
                if (sel) own[np + __popc(bsel & ((1u << lane) - 1u))] = cgrp[i];
                np += __popc(bsel);
                eqr += __popc(beq);
            }
            // the prefetched groups serve as the attention chunk if they cover ours
            __syncwarp();
            bool ok_l = true;
            for (int i = lane; i < np; i += 32) {
                bool found = false;
                for (int s2 = 0; s2 < n_spec; ++s2) found |= spec_g[s2] == own[i];
                ok_l = ok_l && found;
            }
            const bool cover = np <= n_spec && __all_sync(0xffffffffu, ok_l);
            if (lane == 0) { sv[16] = np; sv[18] = cover ? 1 : 0; }
        }
        __syncthreads();
        n_own = sv[16];
        use_spec = sv[18] != 0 && n_own <= spec_cap;
        if (use_spec && tid < spec_cap) {
            bool keep = false;
            if (tid < n_spec)
                for (int i = 0; i < n_own; ++i) keep |= own[i] == spec_g[tid];
            if (!keep) spec_sg[tid] = -1;  // prefetched but not selected: masked
        }
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
                bool sel[4];
                int ns = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = base + tid * 4 + e;
                    bool keep = false;
                    if (i < n_cand) {
                        if (kk[e] > kth) keep = true;
                        else if (kk[e] == kth) keep = unsigned(eb++) < take_eq;
                    }
                    sel[e] = keep;
                    ns += keep;
                }
                int ts;
                int ps = written + block_exclusive_scan(ns, scratch, &ts);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (sel[e]) {
                        if (ps < k_b) p.idx_out[int64_t(b) * p.k + ps] = cgrp[base + tid * 4 + e];
                        ++ps;
                    }
                if (tid == 0) { sv[16] = eq_seen + te; sv[17] = written + ts; }
                __syncthreads();
            }
            for (int i = k_b + tid; i < p.k; i += kThreads) p.idx_out[int64_t(b) * p.k + i] = -1;
        }
        __syncthreads();
    } else {
        // ---------- exact multi-pass selection over the sequence's blocks ----------
        // level 1: the full 16-bit-bin histogram of every block's scores.  The
        // speculative S product reads shared memory about to be reused: wait
        // for it first.
        const bool s_done = n_s == 0 || mbar_wait(bars, 0, kWaitNs);
        if (!__syncthreads_and(s_done)) {
            raise_timeout(p, 3);
            release_tmem();
            return;
        }
        clear_smem(smem + kU, kUBytes);
        __syncthreads();
        for (int i = tid; i < nloc; i += kThreads) {
            const unsigned bin = score_key(score_at(i)) >> 16;
            atomicAdd(h16 + (bin >> 1), (bin & 1u) ? 0x10000u : 1u);
        }
        __syncthreads();
        flush_hist(h16, hist1);
        arrive(ctl + kSlowB);
        if (!wait_count(p, ctl + kSlowB, unsigned(n_b), 3, s_ok)) {
            release_tmem();
            return;
        }
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
        if (!wait_count(p, ctl + kSlowC, unsigned(n_b), 4, s_ok)) {
            release_tmem();
            return;
        }
        if (warp == 0) {
            unsigned above = 0;
            const int lo = (k_b > 0 && t1 >= 0) ? hist_walk(hist2, need2, true, &above) : -1;
            if (lane == 0) { sv[22] = lo; sv[23] = int(above); }
        }
        __syncthreads();
        const bool none = k_b == 0 || t1 < 0 || sv[22] < 0;
        kth = none ? 0xFFFFFFFFu : (unsigned(t1) << 16) | unsigned(sv[22]);
        take_eq = none ? 0u : need2 - unsigned(sv[23]);
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
        if (!wait_count(p, ctl + kSlowD, unsigned(n_b), 5, s_ok)) {
            release_tmem();
            return;
        }
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
                    if (lpos < kMaxK) own[lpos] = g_lo + i;
                    if (gpos < k_b) idx_list[int64_t(b) * p.k + gpos] = g_lo + i;
                    ++lpos;
                    ++gpos;
                }
            }
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
        load_q_tile();  // the prefetch was drained above
    }
    PHASE_MARK(14);

    // ---- attention over this block's selected groups (tensor cores) ------------
    // Per 64-token chunk: S = Q K^T (M = 128 head rows, N = 64 tokens) into TMEM;
    // each warpgroup reads its head rows' scores, takes the row maximum over
    // the chunk, exponentiates its own 16 token columns into the P tile; then
    // O_c = P V (N = DV) into TMEM, folded into the running output in
    // registers (warpgroup g keeps columns [g DV/4, (g+1) DV/4) of its row).
    {
        constexpr int kTK = (DQK / 64) * 8192;
        constexpr int OC = DV / 4;
        const int gpc = kChunk / P;
        const int nchunks = use_spec ? (n_own > 0 ? 1 : 0) : (n_own + gpc - 1) / gpc;
        unsigned char *gbuf = smem + kGather;  // two chunk buffers (when not prefetched)
        auto issue = [&](int ci, int buf) {
            const int jb = ci * gpc;
            gather_tc<DQK, DV>(gbuf + buf * kv_tile_bytes<DQK, DV>(), gsg + buf * kChunk, own + jb,
                               min(gpc, n_own - jb), P, G_b, Kb, Vb);
        };
        cp_async_wait<0>();  // Q (reloaded on the exact fallback path)
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        PHASE_MARK(15);
        const int wg = warp >> 2, row = (warp & 3) * 32 + lane;
        const int lp2 = 31 - __clz(P);  // P is a power of two
        const uint32_t lane_addr = tb + (uint32_t((warp & 3) * 32) << 16);
        if (!use_spec && nchunks > 0) issue(0, 0);
        float o[OC];
#pragma unroll
        for (int c2 = 0; c2 < OC; ++c2) o[c2] = 0.f;
        float m = -INFINITY, lp = 0.f;  // running max; sum of this warpgroup's columns
        // a parity wait only tells the last two phases apart: let the unused
        // speculative product complete before new ones are issued
        bool ok = use_spec || n_s == 0 || __all_sync(0xffffffffu, mbar_wait(bars, 0, kWaitNs));
        for (int ci = 0; ci < nchunks; ++ci) {
            const int buf = ci & 1;
            unsigned char *tk = use_spec ? smem + kSpec : gbuf + buf * kv_tile_bytes<DQK, DV>();
            const int *cg = use_spec ? spec_sg : gsg + buf * kChunk;
            if (!use_spec) {
                if (ci + 1 < nchunks) {
                    issue(ci + 1, buf ^ 1);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                fence_async_smem();
                tc_fence_before();
                __syncthreads();
                tc_fence_after();
            }
            if (!use_spec) {  // the prefetched chunk's S was issued speculatively
                issue_s(tk);
                ++n_s;
            }
            // validity of the chunk's 64 tokens (the same for every row)
            const unsigned long long vmask =
                (unsigned long long)__ballot_sync(0xffffffffu, cg[lane >> lp2] >= 0) |
                ((unsigned long long)__ballot_sync(0xffffffffu, cg[(lane + 32) >> lp2] >= 0) << 32);
            ok = __all_sync(0xffffffffu, ok && mbar_wait(bars, (n_s - 1) & 1, kWaitNs));
            tc_fence_after();
            PHASE_MARK(25);
            float al = 0.f;
            if (ok) {
                float mx = -INFINITY;
                uint32_t r[16];
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    tc_ld16(lane_addr + c0, r);
                    tc_wait_ld();
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if (vmask >> (c0 + t) & 1ull)
                            mx = fmaxf(mx, __uint_as_float(r[t]) * p.scale_log2);
                }
                const float mn = fmaxf(m, mx);
                const float ref = mn == -INFINITY ? 0.f : mn;
                al = exp2f(m - ref);
                m = mn;
                tc_ld16(lane_addr + 16 * wg, r);  // this warpgroup's 16 token columns
                tc_wait_ld();
                float pv[16];
                float ls = 0.f;
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    pv[t] = (vmask >> (16 * wg + t) & 1ull)
                                ? exp2f(__uint_as_float(r[t]) * p.scale_log2 - ref)
                                : 0.f;
                    ls += pv[t];
                }
                lp = lp * al + ls;
                uint4 w0, w1;
                w0.x = pack_bf2(pv[0], pv[1]);   w0.y = pack_bf2(pv[2], pv[3]);
                w0.z = pack_bf2(pv[4], pv[5]);   w0.w = pack_bf2(pv[6], pv[7]);
                w1.x = pack_bf2(pv[8], pv[9]);   w1.y = pack_bf2(pv[10], pv[11]);
                w1.z = pack_bf2(pv[12], pv[13]); w1.w = pack_bf2(pv[14], pv[15]);
                *reinterpret_cast<uint4 *>(pt + sw128_offset(row, 16 * wg, 1024)) = w0;
                *reinterpret_cast<uint4 *>(pt + sw128_offset(row, 16 * wg + 8, 1024)) = w1;
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            PHASE_MARK(26);
            if (warp == 0) {  // O_c = P V
                const uint32_t id = idesc_bf16_f32(128, DV, false, true);
                const uint32_t pa = smem_u32(pt), va = smem_u32(tk + kTK);
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < kChunk / 16; ++ks)
                        tc_mma_bf16(tb + 64, smem_desc(pa + ks * 32, 16, 1024),
                                    smem_desc(va + ks * 2048, 8192, 1024), id, ks > 0);
                    tc_commit(bars + 1);
                }
                __syncwarp();
            }
            ok = __all_sync(0xffffffffu, ok && mbar_wait(bars + 1, ci & 1, kWaitNs));
            tc_fence_after();
            PHASE_MARK(27);
            if (ok) {
                uint32_t r[16];
#pragma unroll
                for (int c0 = 0; c0 < OC; c0 += 16) {
                    tc_ld16(lane_addr + 64 + wg * OC + c0, r);
                    tc_wait_ld();
#pragma unroll
                    for (int t = 0; t < 16; ++t) o[c0 + t] = o[c0 + t] * al + __uint_as_float(r[t]);
                }
            }
            tc_fence_before();
        }
        PHASE_MARK(16);
        if (!ok) {
            raise_timeout(p, 5);
            sv[19] = 1;
        }
        // stage the O rows in shared memory (the chunk buffers are done) so the
        // partial state goes out in contiguous rows
        constexpr int kOP = DV + 4;  // staged row pitch (floats)
        float *ostage = reinterpret_cast<float *>(smem + kGather);
        lpart[wg * 128 + row] = lp;
        if (row < p.H_q) {
#pragma unroll
            for (int c2 = 0; c2 < OC; c2 += 4)
                *reinterpret_cast<float4 *>(ostage + row * kOP + wg * OC + c2) =
                    make_float4(o[c2], o[c2 + 1], o[c2 + 2], o[c2 + 3]);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_free(tb, 256);
        if (sv[19]) return;  // a tensor-core step never completed
        // the block's partial state of each head: (m, l) and the unnormalised O row
        const int64_t pbase = int64_t(cta) * p.H_q;
        for (int e = tid; e < p.H_q * (DV / 4); e += kThreads) {
            const int h = e / (DV / 4), c4 = e % (DV / 4);
            const float l = lpart[h] + lpart[128 + h] + lpart[256 + h] + lpart[384 + h];
            const float4 v = l > 0.f ? *reinterpret_cast<const float4 *>(ostage + h * kOP + c4 * 4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            st_part4(p.part_o + (pbase + h) * DV + c4 * 4, v);
        }
        if (wg == 0 && row < p.H_q) {
            const float l = lpart[row] + lpart[128 + row] + lpart[256 + row] + lpart[384 + row];
            st_part2(reinterpret_cast<float *>(p.part_ml + pbase + row), l > 0.f ? m : -INFINITY, l);
        }
    }
    PHASE_MARK(17);

    // ---- merge the blocks' partial states, head by head ---------------------------
    // The head's combining block polls the partial words of every block of the
    // sequence until all are written, then clears them for the next call.
    PHASE_MARK(18);
    {
        float *wsm = reinterpret_cast<float *>(smem + kU);       // [kMaxCtas] weights
        float *lsm = wsm + kMaxCtas;                              // [kWarps] sums of w l
        float *red = lsm + kMaxCtas;                              // [ngrp][DV]
        constexpr int D4 = DV / 4;                                // float4 columns
        const int sg = tid / D4, dc = tid % D4;                   // split group, column
        const int ngrp = kThreads / D4;                           // 16 (DV=128) or 32 (DV=64)
        for (int h = j; h < p.H_q; h += n_b) {
            constexpr int kU4 = (kMaxCtas + 15) / 16;
            const int nu = (n_b - sg + ngrp - 1) / ngrp;
            float2 *mlp = p.part_ml + int64_t(cb0 + tid) * p.H_q + h;
            auto op_at = [&](int u) {
                return p.part_o + (int64_t(cb0 + sg + u * ngrp) * p.H_q + h) * DV + dc * 4;
            };
            uint2 mlw = make_uint2(1u, 1u);
            if (tid < n_b) mlw = ld_relaxed_u32x2(mlp);
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
                    __nanosleep(32);
                }
            }
            PHASE_MARK(30);
            float2 ml = make_float2(-INFINITY, 0.f);
            if (tid < n_b) {
                ml = make_float2(part_dec(mlw.x), part_dec(mlw.y));
                st_relaxed_zero2(mlp);
            }
            float4 ov[kU4];
#pragma unroll
            for (int u = 0; u < kU4; ++u) {
                ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (u < nu) {
                    ov[u] = make_float4(part_dec(ow[u].x), part_dec(ow[u].y), part_dec(ow[u].z),
                                        part_dec(ow[u].w));
                    st_relaxed_zero4(op_at(u));
                }
            }
            // M = max over blocks (warp max, then over the warps' maxima)
            float m = ml.x;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) sred[warp] = m;
            __syncthreads();
            if (sv[19]) return;  // a partial state never arrived
            PHASE_MARK(31);
            float M = lane < kWarps ? sred[lane] : -INFINITY;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float ref = M == -INFINITY ? 0.f : M;
            // block weights 2^(m_s - M) and L = sum of w_s l_s (warp sums first)
            float wl = 0.f;
            if (tid < n_b) {
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
            for (int u = 0; u < (kMaxCtas + 15) / 16; ++u) {
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
            __syncthreads();
        }
    }
    PHASE_MARK(19);
    __syncthreads();
    // this block's words of the other buffers were read during the previous
    // call: clear them for the next one
    {
        const int op = par ^ 1;
        if (tid < kSlotWords)
            st_relaxed_u64(p.slots + (size_t(op) * ncta + cta) * kSlotWords + tid, 0ull);
        else if (tid >= 32 && tid < 32 + kWarps)
            st_relaxed_u64(p.samp + (size_t(op) * ncta + cta) * kWarps + (tid - 32), 0ull);
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

int num_sms() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

template <int DQK>
constexpr int smem_bytes() {
    return kQT + q_tile_bytes<DQK>() + 8192;
}

struct WsLayout {
    size_t ctl, hist, samp, slots, cand, ovf, gscore, cta_cnt, idx_ws, part_o, part_ml, total;
};

WsLayout ws_layout(int B, int G_max, int H_q, int d_v, int k, int ncta) {
    WsLayout w;
    size_t off = 256;  // status + abort words
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    w.ctl = take(size_t(B) * kCtlWords * 4);
    w.hist = take(size_t(B) * 2 * kHistWords * 4);
    w.samp = take(size_t(2) * ncta * kWarps * 8);
    w.slots = take(size_t(2) * ncta * kSlotBytes);
    w.cand = take(size_t(2) * B * G_max * 8);
    w.ovf = take(size_t(2) * ncta * 8);
    w.gscore = take(size_t(B) * G_max * 4);
    w.cta_cnt = take(size_t(2) * ncta * 4);
    w.idx_ws = take(size_t(B) * k * 4);
    w.part_o = take(size_t(ncta) * H_q * d_v * 4);
    w.part_ml = take(size_t(ncta) * H_q * 8);
    w.total = off;
    return w;
}

}  // namespace

bool fused_decode_supported(int B, int G_max, int H_i, int H_q, int d_qk, int d_v, int k, int P) {
    const int ncta = num_sms();
    if (ncta > kMaxCtas || B < 1 || 2 * B > ncta) return false;
    if (H_i > 16 || k > kMaxK || k < 1) return false;
    if (!((d_qk == 64 || d_qk == 128 || d_qk == 192) && (d_v == 64 || d_v == 128))) return false;
    if (!(H_q % 16 == 0 && H_q <= 64)) return false;  // one M = 128 tensor-core tile of heads
    // 16-bit shared counters: a block's chunk must stay below 65536 groups
    const long long bound = (long long)B * G_max / (ncta - B) + 32;
    if (bound >= 65535) return false;
    (void)P;
    return true;
}

size_t fused_decode_ws_bytes(int B, int G_max, int H_q, int d_v, int k, int P) {
    if (!fused_decode_supported(B, G_max, 1, H_q, 128, d_v, k, P)) return 0;
    return ws_layout(B, G_max, H_q, d_v, k, num_sms()).total;
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

extern "C" int lcsw_debug_stamps(long long *out) {
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(out, g_stamp, sizeof(long long) * 160 * 40);
    long long z[160 * 40] = {0};
    cudaMemcpyToSymbol(g_stamp, z, sizeof z);
    return int(cudaGetLastError());
}
#endif

cudaError_t launch_fused_decode(const lcsw_decode_args *a, void *ws, int *status,
                                cudaStream_t st) {
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
    prm.samp = reinterpret_cast<unsigned long long *>(base + w.samp);
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
