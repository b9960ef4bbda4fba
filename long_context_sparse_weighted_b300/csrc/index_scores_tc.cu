// Indexer scores for a chunk of prefill queries as a tcgen05 GEMM fed by TMA
// (the indexer score of "G2C Brief -- GLM-5.3-Flash", section "DSA keeps
// selected global access in eleven layers", over pooled keys as in the reading
// notes, section 2):
//
//   scores[b][t][g] = sum_h w[b][t][h] * max(0, q[b][t][h] . k_pooled[b][g])
//
// for the groups visible to query t (g < seq_len[b]/P and, with q_pos,
// P*g + P - 1 <= q_pos[b][t]), -inf for the others.
//
// One CTA per tile of 128 queries x 128 groups, 256 threads, two CTAs per SM.
// TMA brings the group tile once and, per indexer head, the 128 x 64 query
// tile of that head (both 128-byte swizzled, two query buffers).  Head h's
// product D_h = Q_h K^T (M = 128 queries, N = 128 groups, K = 64: four MMAs)
// lands in one of two TMEM buffers, so the MMA of head h + 1 runs while the
// warps fold head h into their running sums: warp w reads TMEM lanes
// 32 (w % 4) .. +31 (its query rows) and columns 64 (w / 4) .. +63, and adds
// w_h * max(0, x) in registers.  Tiles where no group is visible to any of
// the 128 queries are written as -inf without touching the tensor cores.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/lcsw.h"
#include "common.cuh"
#include "kernels.cuh"
#include "tc_core.cuh"
#include "tma_host.h"

namespace lcsw {
namespace {

constexpr int kTM = 128;        // queries per tile
constexpr int kTN = 128;        // groups per tile
constexpr int kThr = 256;       // threads per CTA
constexpr int kTile = 16384;    // one 128-row x 128-byte operand tile
constexpr int kSmem = 3 * kTile + 1024;  // group tile, two query tiles, barriers
constexpr unsigned kIdesc = idesc_bf16_f32(kTM, kTN, false, false);

__global__ void __launch_bounds__(kThr, 2)
    scores_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const float *__restrict__ w_head, const int32_t *__restrict__ seq_len,
                     const int32_t *__restrict__ q_pos, int T, int H_i, int P, int G_max,
                     float *__restrict__ scores, int *status) {
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *sk = sm, *sq = sm + kTile;  // group tile; query tiles [2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + 3 * kTile);  // k, q[2], d[2]
    uint32_t *slot = reinterpret_cast<uint32_t *>(bars + 5);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g0 = blockIdx.x * kTN, t0 = blockIdx.y * kTM, b = blockIdx.z;
    const int row = (warp & 3) * 32 + lane, t = t0 + row, c0 = (warp >> 2) * 64;

    // groups visible to this thread's query
    int nvis = 0;
    if (t < T) {
        nvis = min(max(__ldg(seq_len + b) / P, 0), G_max);
        if (q_pos) nvis = min(nvis, max(0, (__ldg(q_pos + int64_t(b) * T + t) + 1) / P));
    }
    float *orow = scores + (int64_t(b) * T + t) * G_max;
    auto store = [&](const float (&acc)[64]) {
        if (t >= T) return;
        const bool vec = (G_max & 3) == 0;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
            const int g = g0 + c0 + j;
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = g + e < nvis ? acc[j + e] + 0.0f : -INFINITY;
            if (vec && g + 3 < G_max) {
                __stcs(reinterpret_cast<float4 *>(orow + g), make_float4(v[0], v[1], v[2], v[3]));
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (g + e < G_max) __stcs(orow + g + e, v[e]);
            }
        }
    };
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
    if (!__syncthreads_or(g0 < nvis)) {  // nothing visible in this tile
        store(acc);
        return;
    }
    if ((smem_u32(sm) & 1023u) != 0u) {  // the swizzled tiles need 1024-byte alignment
        if (tid == 0 && status) atomicCAS(status, 0, int(LCSW_ERR_UNSUPPORTED) * 256);
        return;
    }
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(bars + i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(bars, kTile);
        tma_load_3d(sk, &tk, bars, 0, g0, b);
        for (int h = 0; h < min(2, H_i); ++h) {
            mbar_expect_tx(bars + 1 + h, kTile);
            tma_load_3d(sq + h * kTile, &tq, bars + 1 + h, 0, h, b * T + t0);
        }
    }
    if (warp == 0) tmem_alloc(slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;  // D buffers: columns 0..127 and 128..255
    const float *wrow = w_head + (int64_t(b) * T + min(t, T - 1)) * H_i;

    bool ok = true;
    // head h's product, issued by one lane of warp 1 once its tiles have landed
    auto issue = [&](int h) {
        if (warp != 1) return;
        bool good = true;
        if (elect_one()) {
            good = (h > 0 || mbar_wait(bars, 0, kWaitNs)) &&
                   mbar_wait(bars + 1 + (h & 1), (h >> 1) & 1, kWaitNs);
            if (good) {
                tc_fence_after();
                const uint32_t qa = smem_u32(sq + (h & 1) * kTile), ka = smem_u32(sk);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc_mma_bf16(tb + (h & 1) * kTN, smem_desc(qa + ks * 32, 16, 1024),
                                smem_desc(ka + ks * 32, 16, 1024), kIdesc, ks > 0);
                tc_commit(bars + 3 + (h & 1));
            }
        }
        ok = __all_sync(0xffffffffu, good) && ok;
    };
    issue(0);
    const uint32_t lane_addr = tb + (uint32_t((warp & 3) * 32) << 16) + c0;
    for (int h = 0; h < H_i; ++h) {
        if (h + 1 < H_i) issue(h + 1);
        const float wh = __ldg(wrow + h);
        ok = __all_sync(0xffffffffu, ok && mbar_wait(bars + 3 + (h & 1), (h >> 1) & 1, kWaitNs));
        tc_fence_after();
        if (ok) {
            uint32_t r[16];
#pragma unroll
            for (int cc = 0; cc < 64; cc += 16) {
                tc_ld16(lane_addr + (h & 1) * kTN + cc, r);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    acc[cc + e] = __fadd_rn(acc[cc + e],
                                            __fmul_rn(wh, fmaxf(__uint_as_float(r[e]), 0.f)));
            }
        }
        tc_fence_before();
        __syncthreads();  // head h's buffers are free again
        if (tid == 0 && h + 2 < H_i && ok) {
            mbar_expect_tx(bars + 1 + (h & 1), kTile);
            tma_load_3d(sq + (h & 1) * kTile, &tq, bars + 1 + (h & 1), 0, h + 2, b * T + t0);
        }
    }
    tc_fence_after();
    if (!__syncthreads_and(ok)) {
        if (tid == 0 && status) atomicCAS(status, 0, int(LCSW_ERR_TIMEOUT) * 256 + 9);
    } else {
        store(acc);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, 256);
}

// Persistent form for H_i <= 8: every query block's H_i query tiles stay in
// shared memory while the CTA walks its range of group tiles, so the loop
// never waits on a query load.  Warp roles: warps 0-15 fold products into
// sums and store (warp w: TMEM lane quarter w % 4, 32 columns from
// 32 (w / 4)), warp 16 is the TMA producer (query tiles per block, group
// tiles through a 2-slot ring), warp 17 issues the MMAs (one product per head
// into four rotating TMEM buffers).  Hand-offs are mbarriers: slot full / empty, buffer full / empty,
// query block loaded / released.  Group tiles past a sequence's length are
// written as -inf without a load or an MMA.
constexpr int kPThr = 576;                    // 16 folding warps + producer + MMA warp
constexpr int kSampleTiles = 16;              // group tiles of the prefill threshold sample
constexpr int kPFold = 16;
constexpr int kPSlots = 2;                    // group-tile ring
constexpr int kPBufs = 4;                     // TMEM product buffers (4 x 128 columns)
constexpr int kPQ = 8 * kTile;                // query tiles of one block
constexpr int kPStage = kPFold * 32 * 128;    // per folding warp: 32 rows x 32 floats
constexpr int kPSmem = kPQ + kPSlots * kTile + kPStage + 1024;

}  // namespace

// One pass of the persistent kernel over (batch, query block, pass tile) units;
// pass tile j is group tile j * gt_stride.  Dense mode writes the scores of
// pass tile j to columns [128 j, 128 j + 128) of out rows of pitch ldo (-inf
// where not visible, columns >= ldo dropped).  Candidate mode keeps, per query
// row, the visible groups whose score key is at or above thr[row], appending
// (key | group << 32) to the row's list of cap entries (count in ccount[row],
// which may exceed cap: the caller treats that row as overflowed).
struct ScorePass {
    int gt_count, gt_stride;
    float *out;
    int64_t ldo;
    const uint32_t *thr;
    unsigned *ccount;
    unsigned long long *cand;
    int cap;
    const int *run_if;  // non-null: the pass runs only when *run_if != 0
};

namespace {

struct PBars {  // mbarrier indices
    static constexpr int qfull = 0, qfree = 1, kfull = 2, kfree = kfull + kPSlots,
                         dfull = kfree + kPSlots, dfree = dfull + kPBufs, n = dfree + kPBufs;
};

template <bool kCands>
__global__ void __launch_bounds__(kPThr, 1)
    scores_tc_persist_kernel(const __grid_constant__ CUtensorMap tq,
                             const __grid_constant__ CUtensorMap tk,
                             const float *__restrict__ w_head, const int32_t *__restrict__ seq_len,
                             const int32_t *__restrict__ q_pos, int B, int T, int H_i, int P,
                             int G_max, const ScorePass ps, int *status) {
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *sq = sm, *sk = sm + kPQ;
    float *stage_all = reinterpret_cast<float *>(sm + kPQ + kPSlots * kTile);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kPQ + kPSlots * kTile + kPStage);
    uint32_t *slot = reinterpret_cast<uint32_t *>(bars + PBars::n);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (ps.run_if && *reinterpret_cast<const volatile int *>(ps.run_if) == 0) return;
    const int nqb = (T + kTM - 1) / kTM, ngt = ps.gt_count;
    const long long n_units = (long long)B * nqb * ngt;
    const long long u0 = n_units * blockIdx.x / gridDim.x;
    const long long u1 = n_units * (blockIdx.x + 1) / gridDim.x;
    if (u0 >= u1) return;
    if ((smem_u32(sm) & 1023u) != 0u) {
        if (tid == 0 && status) atomicCAS(status, 0, int(LCSW_ERR_UNSUPPORTED) * 256);
        return;
    }
    if (tid == 0) {
        for (int i = 0; i < PBars::n; ++i)
            mbar_init(bars + i, (i >= PBars::dfree && i < PBars::dfree + kPBufs) ? kPFold : 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;
    // units are walked in order (batch, query block, group tile): one decode,
    // then increments; Gb = the batch's complete groups (P is a power of two)
    const int lp2 = 31 - __clz(P);
    struct Walk {
        int b, qb, gt, Gb;
    };
    auto start = [&]() {
        Walk w;
        w.gt = int(u0 % ngt);
        w.qb = int((u0 / ngt) % nqb);
        w.b = int(u0 / ((long long)ngt * nqb));
        w.Gb = min(max(__ldg(seq_len + w.b) >> lp2, 0), G_max);
        return w;
    };
    auto next = [&](Walk &w) {
        if (++w.gt == ngt) {
            w.gt = 0;
            if (++w.qb == nqb) {
                w.qb = 0;
                ++w.b;
                if (w.b < B) w.Gb = min(max(__ldg(seq_len + w.b) >> lp2, 0), G_max);
            }
        }
    };
    auto wait = [&](int bar, unsigned parity) {
        if (*abort_flag) return false;
        if (mbar_wait(bars + bar, parity, kWaitNs)) return true;
        *abort_flag = 1;
        return false;
    };

    if (warp == kPFold) {  // ---------------- TMA producer
        if (elect_one()) {
            int kq = 0, nq = 0, prev = -1;
            Walk w = start();
            for (long long u = u0; u < u1 && !*abort_flag; ++u, next(w)) {
                const int b = w.b, qb = w.qb, gt = w.gt;
                if (b * nqb + qb != prev) {  // a new query block: reload its query tiles
                    if (nq > 0 && !wait(PBars::qfree, (nq - 1) & 1)) break;
                    mbar_expect_tx(bars + PBars::qfull, H_i * kTile);
                    for (int h = 0; h < H_i; ++h)
                        tma_load_3d(sq + h * kTile, &tq, bars + PBars::qfull, 0, h, b * T + qb * kTM);
                    prev = b * nqb + qb;
                    ++nq;
                }
                const int gr = gt * ps.gt_stride;  // the group tile itself
                if (gr * kTN >= w.Gb) continue;
                const int s = kq % kPSlots;
                if (kq >= kPSlots && !wait(PBars::kfree + s, ((kq / kPSlots) - 1) & 1)) break;
                mbar_expect_tx(bars + PBars::kfull + s, kTile);
                tma_load_3d(sk + s * kTile, &tk, bars + PBars::kfull + s, 0, gr * kTN, b);
                ++kq;
            }
        }
        __syncwarp();
    } else if (warp == kPFold + 1) {  // ---------------- MMA issuer
        if (elect_one()) {
            int kq = 0, nq = 0, nd = 0, prev = -1;
            Walk w = start();
            for (long long u = u0; u < u1 && !*abort_flag; ++u, next(w)) {
                const int b = w.b, qb = w.qb, gt = w.gt;
                if (b * nqb + qb != prev) {
                    if (nq > 0) tc_commit(bars + PBars::qfree);  // old query tiles released
                    if (!wait(PBars::qfull, nq & 1)) break;
                    prev = b * nqb + qb;
                    ++nq;
                }
                if (gt * ps.gt_stride * kTN >= w.Gb) continue;
                const int s = kq % kPSlots;
                if (!wait(PBars::kfull + s, (kq / kPSlots) & 1)) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(sk + s * kTile);
                bool good = true;
                for (int h = 0; h < H_i && good; ++h, ++nd) {
                    const int d = nd % kPBufs;
                    if (nd >= kPBufs && !wait(PBars::dfree + d, ((nd / kPBufs) - 1) & 1)) {
                        good = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qa = smem_u32(sq + h * kTile);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc_mma_bf16(tb + d * kTN, smem_desc(qa + ks * 32, 16, 1024),
                                    smem_desc(ka + ks * 32, 16, 1024), kIdesc, ks > 0);
                    tc_commit(bars + PBars::dfull + d);
                }
                if (!good) break;
                tc_commit(bars + PBars::kfree + s);  // the slot frees when these MMAs finish
                ++kq;
            }
        }
        __syncwarp();
    } else {  // ---------------- warps 0-15: fold and store
        const int row = (warp & 3) * 32 + lane, c0 = (warp >> 2) * 32;
        const uint32_t lane_addr = tb + (uint32_t((warp & 3) * 32) << 16) + c0;
        int nd = 0, prev = -1, nvis = 0, t = 0;
        float thr = __int_as_float(0x7FFFFFFF);  // threshold as a score (NaN: keep nothing)
        float wv[8];
        Walk w = start();
        for (long long u = u0; u < u1 && !*abort_flag; ++u, next(w)) {
            const int b = w.b, qb = w.qb, gt = w.gt, Gb = w.Gb;
            if (b * nqb + qb != prev) {
                prev = b * nqb + qb;
                t = qb * kTM + row;
                nvis = 0;
                if (t < T) {
                    nvis = Gb;
                    if (q_pos) nvis = min(nvis, max(0, (__ldg(q_pos + int64_t(b) * T + t) + 1) >> lp2));
                }
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    wv[h] = (h < H_i && t < T) ? __ldg(w_head + (int64_t(b) * T + t) * H_i + h) : 0.f;
                if (kCands) {
                    // key >= thr key  <=>  score >= the score of that key (finite scores)
                    const uint32_t tk = t < T ? __ldg(ps.thr + int64_t(b) * T + t) : 0xFFFFFFFFu;
                    thr = tk == 0u ? -INFINITY
                                   : __uint_as_float((tk & 0x80000000u) ? (tk & 0x7FFFFFFFu) : ~tk);
                }
            }
            const int gr = gt * ps.gt_stride;
            const int g0 = gr * kTN + c0;  // first group of this thread's 32 columns
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.f;
            if (gr * kTN < Gb) {
                bool good = true;
#pragma unroll 1
                for (int h = 0; h < H_i; ++h, ++nd) {
                    const int d = nd % kPBufs;
                    good = __all_sync(0xffffffffu, good && wait(PBars::dfull + d, (nd / kPBufs) & 1));
                    tc_fence_after();
                    uint32_t r[32];
                    if (good) {
                        tc_ld32(lane_addr + d * kTN, r);
                        tc_wait_ld();
                    }
                    // buffer d is in registers: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                                                    smem_u32(bars + PBars::dfree + d))
                                                : "memory");
                    if (good) {
                        float wh = wv[0];
#pragma unroll
                        for (int hh = 1; hh < 8; ++hh) wh = h == hh ? wv[hh] : wh;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            acc[e] = fmaf(wh, fmaxf(__uint_as_float(r[e]), 0.f), acc[e]);
                    }
                }
                if (!good) break;
            }
            if (kCands) {
                // visible groups at or above the row's threshold join its list
                if (t < T && gr * kTN < Gb) {
                    unsigned keep = 0u;
#pragma unroll
                    for (int e = 0; e < 32; ++e) keep |= unsigned(acc[e] >= thr) << e;
                    if (g0 + 32 > nvis)  // past the visible groups
                        keep &= nvis > g0 ? (1u << (nvis - g0)) - 1u : 0u;
                    if (keep) {
                        // the row's values go to the warp's staging block (row =
                        // lane, chunks swizzled as for the dense store) so that a
                        // kept column is one shared load, not a register select
                        float *stg = stage_all + warp * 32 * 32 + lane * 32;
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(stg + (((j >> 2) ^ (lane & 7)) << 2)) =
                                make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                        const int64_t rrow = int64_t(b) * T + t;
                        unsigned pos = atomicAdd(ps.ccount + rrow, unsigned(__popc(keep)));
                        unsigned long long *dst = ps.cand + rrow * ps.cap;
                        while (keep) {
                            const int e = __ffs(keep) - 1;
                            keep &= keep - 1u;
                            const float v = stg[(((e >> 2) ^ (lane & 7)) << 2) + (e & 3)] + 0.0f;
                            if (pos < unsigned(ps.cap))
                                dst[pos] = score_key(v) | ((unsigned long long)(g0 + e) << 32);
                            ++pos;
                        }
                    }
                }
                continue;
            }
            // masked row values -> the warp's staging block (row = lane, 16-byte
            // chunks XOR-swizzled by row) -> eight lanes per 128-byte row segment
            float *stg = stage_all + warp * 32 * 32;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const int g = g0 + j;
                float4 v;
                v.x = g + 0 < nvis ? acc[j + 0] + 0.0f : -INFINITY;
                v.y = g + 1 < nvis ? acc[j + 1] + 0.0f : -INFINITY;
                v.z = g + 2 < nvis ? acc[j + 2] + 0.0f : -INFINITY;
                v.w = g + 3 < nvis ? acc[j + 3] + 0.0f : -INFINITY;
                *reinterpret_cast<float4 *>(stg + lane * 32 + (((j >> 2) ^ (lane & 7)) << 2)) = v;
            }
            __syncwarp();
            {
                const int ch = lane & 7;
                const int64_t oc = int64_t(gt) * kTN + c0 + ch * 4;  // output column
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int r = (lane >> 3) + 4 * m, tr = qb * kTM + (warp & 3) * 32 + r;
                    if (tr < T && oc < ps.ldo) {
                        const float4 v = *reinterpret_cast<const float4 *>(
                            stg + r * 32 + ((ch ^ (r & 7)) << 2));
                        float *dst = ps.out + (int64_t(b) * T + tr) * ps.ldo + oc;
                        if ((ps.ldo & 3) == 0) {
                            __stcs(reinterpret_cast<float4 *>(dst), v);
                        } else {
                            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (oc + e < ps.ldo) __stcs(dst + e, vv[e]);
                        }
                    }
                }
            }
            __syncwarp();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0 && status) atomicCAS(status, 0, int(LCSW_ERR_TIMEOUT) * 256 + 9);
    if (warp == 0) tmem_free(tb, 512);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool index_scores_tc_supported(int B, int T, int H_i, int G_max, int64_t sp_b) {
    // the group tiles read up to G_max rows of every sequence's cache
    return T >= 64 && H_i >= 1 && H_i <= 16 && B >= 1 && B <= 65535 && G_max >= 1 &&
           (T + kTM - 1) / kTM <= 65535 && sp_b % 8 == 0 && sp_b >= int64_t(64) * G_max &&
           encode_fn() != nullptr;
}

namespace {

// Tensor maps of the queries ([B*T][H_i][64]: one box = 128 queries of one
// head) and of the pooled keys ([B][G_max][64] with the batch stride: one box
// = 128 groups), both 128-byte swizzled.
bool make_maps(const uint16_t *q_idx, const uint16_t *k_pooled, int64_t sp_b, int B, int T,
               int H_i, int G_max, CUtensorMap *tq, CUtensorMap *tk) {
    auto enc = encode_fn();
    const cuuint64_t qdim[3] = {64, cuuint64_t(H_i), cuuint64_t(B) * T};
    const cuuint64_t qstr[2] = {128, cuuint64_t(H_i) * 128};
    const cuuint32_t qbox[3] = {64, 1, kTM};
    const cuuint64_t kdim[3] = {64, cuuint64_t(G_max), cuuint64_t(B)};
    const cuuint64_t kstr[2] = {128, cuuint64_t(sp_b) * 2};
    const cuuint32_t kbox[3] = {64, kTN, 1};
    const cuuint32_t ones[3] = {1, 1, 1};
    return enc(tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(q_idx), qdim, qstr,
               qbox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
               CUDA_SUCCESS &&
           enc(tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(k_pooled), kdim,
               kstr, kbox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
               CUDA_SUCCESS;
}

template <bool kCands>
cudaError_t launch_persist(const CUtensorMap &tq, const CUtensorMap &tk, const float *w_head,
                           const int32_t *seq_len, const int32_t *q_pos, int B, int T, int H_i,
                           int P, int G_max, const ScorePass &ps, int *status, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(scores_tc_persist_kernel<kCands>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    scores_tc_persist_kernel<kCands><<<sms, kPThr, kPSmem, st>>>(tq, tk, w_head, seq_len, q_pos, B,
                                                                 T, H_i, P, G_max, ps, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_index_scores_tc(const uint16_t *q_idx, const float *w_head,
                                   const uint16_t *k_pooled, int64_t sp_b,
                                   const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                   int H_i, int P, int G_max, float *scores, int *status,
                                   cudaStream_t st, const int *run_if) {
    if (!index_scores_tc_supported(B, T, H_i, G_max, sp_b)) return cudaErrorNotSupported;
    CUtensorMap tq, tk;
    if (!make_maps(q_idx, k_pooled, sp_b, B, T, H_i, G_max, &tq, &tk)) return cudaErrorInvalidValue;
    if (H_i <= 8) {
        ScorePass ps = {};
        ps.gt_count = (G_max + kTN - 1) / kTN;
        ps.gt_stride = 1;
        ps.out = scores;
        ps.ldo = G_max;
        ps.run_if = run_if;
        return launch_persist<false>(tq, tk, w_head, seq_len, q_pos, B, T, H_i, P, G_max, ps,
                                     status, st);
    }
    if (run_if) return cudaErrorNotSupported;  // the per-tile kernel has no gated form
    cudaError_t e = cudaFuncSetAttribute(scores_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(unsigned((G_max + kTN - 1) / kTN), unsigned((T + kTM - 1) / kTM), unsigned(B));
    scores_tc_kernel<<<grid, kThr, kSmem, st>>>(tq, tk, w_head, seq_len, q_pos, T, H_i, P, G_max,
                                                 scores, status);
    return cudaGetLastError();
}

int prefill_sample_tiles(int G_max) { return min((G_max + kTN - 1) / kTN, kSampleTiles); }

cudaError_t launch_prefill_sample_scores(const uint16_t *q_idx, const float *w_head,
                                         const uint16_t *k_pooled, int64_t sp_b,
                                         const int32_t *seq_len, const int32_t *q_pos, int B,
                                         int T, int H_i, int P, int G_max, float *samp,
                                         int *status, cudaStream_t st) {
    if (H_i > 8 || !index_scores_tc_supported(B, T, H_i, G_max, sp_b)) return cudaErrorNotSupported;
    CUtensorMap tq, tk;
    if (!make_maps(q_idx, k_pooled, sp_b, B, T, H_i, G_max, &tq, &tk)) return cudaErrorInvalidValue;
    const int ngt = (G_max + kTN - 1) / kTN, n_st = prefill_sample_tiles(G_max);
    ScorePass ps = {};
    ps.gt_count = n_st;
    ps.gt_stride = ngt / n_st;  // spread over the whole sequence
    ps.out = samp;
    ps.ldo = int64_t(n_st) * kTN;
    return launch_persist<false>(tq, tk, w_head, seq_len, q_pos, B, T, H_i, P, G_max, ps, status,
                                 st);
}

cudaError_t launch_prefill_candidates(const uint16_t *q_idx, const float *w_head,
                                      const uint16_t *k_pooled, int64_t sp_b,
                                      const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                      int H_i, int P, int G_max, const uint32_t *thr,
                                      unsigned *ccount, unsigned long long *cand, int cap,
                                      int *status, cudaStream_t st) {
    if (H_i > 8 || !index_scores_tc_supported(B, T, H_i, G_max, sp_b)) return cudaErrorNotSupported;
    CUtensorMap tq, tk;
    if (!make_maps(q_idx, k_pooled, sp_b, B, T, H_i, G_max, &tq, &tk)) return cudaErrorInvalidValue;
    ScorePass ps = {};
    ps.gt_count = (G_max + kTN - 1) / kTN;
    ps.gt_stride = 1;
    ps.thr = thr;
    ps.ccount = ccount;
    ps.cand = cand;
    ps.cap = cap;
    return launch_persist<true>(tq, tk, w_head, seq_len, q_pos, B, T, H_i, P, G_max, ps, status,
                                st);
}

}  // namespace lcsw
