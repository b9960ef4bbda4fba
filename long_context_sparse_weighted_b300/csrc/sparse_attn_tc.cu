// Sparse attention over the selected history on the fifth-generation tensor
// cores, for many query rows at once (chunked prefill): "G2C Brief --
// GLM-5.3-Flash", DSA section (attention over the selected tokens, one
// shared K/V head serving every query head).  A row's k selected groups
// expand to k*P tokens, taken in chunks of 128.
//
// One persistent CTA per SM walks the rows; its warps have fixed roles:
//   warps 4-8  gather.  Ring item n (a chunk's 128 key rows or value rows)
//              belongs to warp 4 + n % 5, which copies it with 16-byte
//              cp.async into slot n % 5 of a ring of 32 KB 128B-swizzled tiles
//              (zero fill for padding and for groups past the sequence), waits
//              for its copies, fences them for the tensor core and arrives on
//              the slot's mbarrier.  The chunk's 128 token rows are computed
//              once per item into shared memory (four index loads per lane),
//              so a copy costs a shared load and a few adds.  The warp
//              holding a row's first item also loads the row's head tile.
//   warp 9     MMA.  S^T = K Q^T (M = 128 tokens, N = 32 heads, K = 128) into
//              TMEM, and O_c^T = V^T P^T (M = 128 value dims, N = 64: the 32
//              heads padded to one 128-byte row of P, K = 128 tokens).  Per
//              row it issues QK_0, then QK_c and PV_(c-1) for c = 1..n-1, then
//              PV_(n-1); the ring holds the matching item sequence.
//   warps 0-3  softmax.  Thread t owns TMEM lane t.  Per chunk it reads its
//              token's head scores z and writes its token's row of P (bf16),
//              p = 2^(z - m) for the row's reference m of each head.  The
//              reference is lazy: only when some score exceeds it by more than
//              kLazy does the block vote to take the exact chunk maximum of
//              every head (a warp maximum, then the four warps'), move m to
//              it with the rescale a = 2^(m_old - m_new), and rewrite P; a
//              row's first chunk always does.  The warp's sums of p per head go
//              to shared memory, and lane h of warp 0 keeps head h's running
//              sum l = a (l + sum of the previous chunk).  Then the thread
//              folds O_(c-1)^T (lane t = value dim t) into its running output
//              row, o = a o + O.  At the row's end the normalised bf16 output
//              and the log-sum-exp are written.
// S and O_c are double-buffered in TMEM (S: columns 0-63, O: 64-191), P in
// shared memory.  Every hand-off is an mbarrier; every wait is bounded and a
// wait that runs out stops all roles, which record LCSW_ERR_TIMEOUT in the
// status word.  TMEM is released on every exit.
#include "../../include/lcsw.h"
#include "common.cuh"
#include "kernels.cuh"
#include "tc_core.cuh"

namespace lcsw {
namespace {

constexpr int kTok = 128;                 // tokens per chunk (M of S^T)
constexpr int kDim = 128;                 // d_qk = d_v
constexpr int kNH = 32;                   // heads (N of S^T; H_q padded)
constexpr int kNPV = 64;                  // N of O^T: one 128-byte row of P
constexpr int kSlots = 5;                 // gather ring
constexpr int kSlotBytes = kTok * kDim * 2;   // 32 KB: a chunk's key or value rows
constexpr int kAtomCol = kTok * 128;          // 16 KB: 64 elements of every row
constexpr int kQBytes = kNH * kDim * 2;       // 8 KB head tile
constexpr int kQAtomCol = kNH * 128;          // 4 KB
constexpr int kPBytes = kTok * 128;           // 16 KB: 128 tokens x 64 heads (bf16)
constexpr int kSmRing = 0;
constexpr int kSmQ = kSmRing + kSlots * kSlotBytes;
constexpr int kSmP = kSmQ + 2 * kQBytes;
constexpr int kSmMisc = kSmP + 2 * kPBytes;
constexpr int kMiscBytes = 6144;
constexpr int kSmemBytes = kSmMisc + kMiscBytes + 1024;  // + alignment slack
constexpr int kThr = 320;                 // 10 warps
constexpr int kGatherWarp0 = 4, kMmaWarp = 9;
constexpr int kGatherWarps = kMmaWarp - kGatherWarp0;
constexpr int kColS = 0, kColO = 64, kTmemCols = 256;
constexpr float kLn2f = 0.6931471805599453f;
// The softmax reference of a head changes only when a score exceeds it by more
// than kLazy (log2 units), so p <= 2^kLazy; otherwise a chunk keeps it.
constexpr float kLazy = 8.f;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// Item i (0-based) of a row with n chunks: (is a value chunk, chunk index).
__device__ __forceinline__ void item_of(int i, int n, bool &is_v, int &c) {
    if (i == 0) {
        is_v = false;
        c = 0;
    } else if (i == 2 * n - 1) {
        is_v = true;
        c = n - 1;
    } else if (i & 1) {
        is_v = false;
        c = (i + 1) >> 1;
    } else {
        is_v = true;
        c = (i >> 1) - 1;
    }
}

// Bounded wait for the phase of the given parity; gives up when about a
// second of the global timer has passed or another role has given up.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity,
                                           const volatile int *abort_flag) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try(a, parity)) return true;
        if (*abort_flag || globaltimer_ns() - t0 > kWaitNs) return false;
    }
}

__device__ __forceinline__ void bar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier 1 over the 128 softmax threads; returns the OR of `v` over them.
__device__ __forceinline__ bool softmax_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 128, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(uint32_t(v))
        : "memory");
    return r != 0;
}

// Maximum over the warp (every lane gets it).
__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// 2^x with the hardware approximation (relative error ~2^-22; p is rounded
// to bf16 for the product).
__device__ __forceinline__ float exp2_hw(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Two floats -> bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(kThr, 1) sparse_attn_tc_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ K, int64_t sK_b,
    const uint16_t *__restrict__ V, int64_t sV_b, const int32_t *__restrict__ seq_len,
    const int32_t *__restrict__ idx, int T, int H_q, int P, int k, int64_t rows,
    float scale_log2, uint16_t *__restrict__ out, float *__restrict__ lse, int *status,
    int test_skip_gather) {
    extern __shared__ unsigned char smem_raw[];
    // the swizzled tiles need 1024-byte alignment
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kSmMisc);
    uint64_t *full = bars, *empty = bars + kSlots;          // ring slots
    uint64_t *qfull = bars + 2 * kSlots, *qempty = qfull + 2;  // head tiles
    uint64_t *sfull = qempty + 2, *sfree = sfull + 2;        // S^T in TMEM
    uint64_t *pfull = sfree + 2, *pempty = pfull + 2;        // P in shared memory
    uint64_t *ofull = pempty + 2, *ofree = ofull + 2;        // O_c^T in TMEM
    uint64_t *mma_done = ofree + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
    float *wmax = reinterpret_cast<float *>(smem + kSmMisc + 256);        // [2][4][32]
    float *alph = wmax + 2 * 4 * 32 + 2 * 32;                             // [2][32]
    float *lsum = alph + 2 * 32;                                          // [2][4][32]
    float *ltot = lsum + 2 * 4 * 32;                                      // [32]
    int *toff = reinterpret_cast<int *>(ltot + 32);           // [kGatherWarps][128]
    float *mcur = reinterpret_cast<float *>(toff + kGatherWarps * kTok);  // [32] reference
    const int lp2 = 31 - __clz(P);
    const int nck = (k * P + kTok - 1) / kTok;
    const int gpc = kTok >> lp2;  // groups per chunk

    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull + i, 1);
            mbar_init(qempty + i, 1);
            mbar_init(sfull + i, 1);
            mbar_init(sfree + i, 4);
            mbar_init(pfull + i, 4);
            mbar_init(pempty + i, 1);
            mbar_init(ofull + i, 1);
            mbar_init(ofree + i, 4);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;
    auto give_up = [&](int where) {
        *abort_flag = 1;
        if (status) atomicCAS(status, 0, int(LCSW_ERR_TIMEOUT) * 256 + where);
    };

    if (warp >= kGatherWarp0 && warp < kMmaWarp) {
        // ------------------------------------------------------------ gather
        const int gw = warp - kGatherWarp0;
        uint32_t n_item = 0;
        int qi = 0;
        bool ok = true;
        const int c16 = lane & 15;                            // 16-byte column of a row
        const uint32_t dcol = uint32_t(c16 >> 3) * kAtomCol;  // its 64-element atom column
        for (int64_t row = blockIdx.x; row < rows && ok; row += gridDim.x, ++qi) {
            const int b = int(row / T);
            const int G = __ldg(seq_len + b) / P;
            const int32_t *gl = idx + row * k;
            const uint16_t *kb = K + int64_t(b) * sK_b, *vb = V + int64_t(b) * sV_b;
            for (int i = 0; i < 2 * nck && ok; ++i, ++n_item) {
                if (int(n_item % kGatherWarps) != gw) continue;
                if (i == 0) {  // the row's head tile first (heads past H_q are zero)
                    const int qs = qi & 1;
                    ok = __all_sync(0xffffffffu,
                                    wait_phase(qempty + qs, (uint32_t(qi >> 1) & 1u) ^ 1u, abort_flag));
                    if (!ok) break;
                    unsigned char *qt = smem + kSmQ + qs * kQBytes;
                    const uint16_t *qrow = q + row * int64_t(H_q) * kDim;
                    for (int e = lane; e < kNH * 16; e += 32) {
                        const int h = e >> 4, cc = e & 15;
                        const bool hv = h < H_q;
                        cp_async16(smem_u32(qt + (cc >> 3) * kQAtomCol + sw128_offset(h, (cc & 7) * 8, 1024)),
                                   hv ? qrow + h * kDim + cc * 8 : qrow, hv ? 16 : 0);
                    }
                    cp_async_commit();
                    cp_async_wait<0>();
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) bar_arrive(qfull + qs);
                }
                bool is_v;
                int c;
                item_of(i, nck, is_v, c);
                const int slot = int(n_item % kSlots);
                ok = __all_sync(0xffffffffu,
                                wait_phase(empty + slot, ((n_item / kSlots) & 1u) ^ 1u, abort_flag));
                if (!ok) break;
                // every token's row in the chunk (-1: zero fill)
                int *to = toff + gw * kTok;
#pragma unroll
                for (int v = 0; v < kTok / 32; ++v) {
                    const int t = lane + 32 * v, j = c * gpc + (t >> lp2);
                    const int g = j < k ? __ldg(gl + j) : -1;
                    to[t] = (g >= 0 && g < G) ? g * P + (t & (P - 1)) : -1;
                }
                __syncwarp();
                const uint32_t tbase = smem_u32(smem + kSmRing + slot * kSlotBytes) + dcol;
                const uint16_t *base = (is_v ? vb : kb) + c16 * 8;
                const int hi = lane >> 4;
#pragma unroll 8
                for (int u = 0; u < kTok / 2; ++u) {
                    const int t = 2 * u + hi;
                    const int r = to[t];
                    cp_async16(tbase + uint32_t((t >> 3) << 10) + uint32_t((t & 7) << 7) +
                                   uint32_t(((c16 & 7) ^ (t & 7)) << 4),
                               r >= 0 ? base + int64_t(r) * kDim : base, r >= 0 ? 16 : 0);
                }
                cp_async_commit();
                cp_async_wait<0>();
                fence_async_smem();  // the copies, for the tensor core's reads
                __syncwarp();
                // (failure-detection test: the CTA's first item is never handed over)
                if (lane == 0 && !(test_skip_gather && n_item == 0)) bar_arrive(full + slot);
            }
        }
        cp_async_wait<0>();
        if (!ok && lane == 0) give_up(11);
    } else if (warp == kMmaWarp) {
        // --------------------------------------------------------------- MMA
        const uint32_t id_qk = idesc_bf16_f32(128, kNH, false, false);
        const uint32_t id_pv = idesc_bf16_f32(128, kNPV, true, true);
        uint32_t n_item = 0, n_ck = 0;
        int qi = 0;
        bool ok = true;
        for (int64_t row = blockIdx.x; row < rows && ok; row += gridDim.x, ++qi) {
            const int qs = qi & 1;
            ok = __all_sync(0xffffffffu, wait_phase(qfull + qs, uint32_t(qi >> 1) & 1u, abort_flag));
            const uint32_t qa = smem_u32(smem + kSmQ + qs * kQBytes);
            for (int i = 0; i < 2 * nck && ok; ++i, ++n_item) {
                bool is_v;
                int c;
                item_of(i, nck, is_v, c);
                const int slot = int(n_item % kSlots);
                const uint32_t ta = smem_u32(smem + kSmRing + slot * kSlotBytes);
                const uint32_t gc = n_ck + uint32_t(c);  // chunk index over the CTA's rows
                const int buf = int(gc & 1u);
                const uint32_t bpar = (gc >> 1) & 1u;
                ok = __all_sync(0xffffffffu,
                                wait_phase(full + slot, (n_item / kSlots) & 1u, abort_flag));
                if (!is_v) {
                    ok = ok && __all_sync(0xffffffffu, wait_phase(sfree + buf, bpar ^ 1u, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < kDim / 16; ++ks) {
                            const uint32_t ka = ta + (ks >> 2) * kAtomCol + (ks & 3) * 32;
                            const uint32_t qk = qa + (ks >> 2) * kQAtomCol + (ks & 3) * 32;
                            tc_mma_bf16(tb + kColS + buf * kNH, smem_desc(ka, 16, 1024),
                                        smem_desc(qk, 16, 1024), id_qk, ks > 0);
                        }
                        tc_commit(sfull + buf);
                        tc_commit(empty + slot);
                        if (c == nck - 1) tc_commit(qempty + qs);
                    }
                    __syncwarp();
                } else {
                    ok = ok && __all_sync(0xffffffffu, wait_phase(pfull + buf, bpar, abort_flag));
                    ok = ok && __all_sync(0xffffffffu, wait_phase(ofree + buf, bpar ^ 1u, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t pa = smem_u32(smem + kSmP + buf * kPBytes);
                    if (elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < kTok / 16; ++ks)
                            tc_mma_bf16(tb + kColO + buf * kNPV,
                                        smem_desc(ta + ks * 2048, kAtomCol, 1024),
                                        smem_desc(pa + ks * 2048, kAtomCol, 1024), id_pv, ks > 0);
                        tc_commit(ofull + buf);
                        tc_commit(empty + slot);
                        tc_commit(pempty + buf);
                    }
                    __syncwarp();
                }
            }
            n_ck += uint32_t(nck);
        }
        if (!ok && lane == 0) give_up(12);
        // every product issued so far completes before TMEM is released
        if (elect_one()) tc_commit(mma_done);
        __syncwarp();
        mbar_wait(mma_done, 0u, kWaitNs);  // bounded; not cut short by an abort
    } else {
        // ----------------------------------------------------------- softmax
        // warps 0-3: thread tid owns TMEM lane tid -- its token of each S^T
        // chunk and value dim tid of each O_c^T
        const uint32_t lane_addr = tb + (uint32_t(warp * 32) << 16);
        uint32_t n_ck = 0;
        bool ok = true;
        float m_run = -INFINITY;  // warp 0, lane h: running maximum of head h
        float l_run = 0.f;        // warp 0, lane h: running sum of p of head h
        for (int64_t row = blockIdx.x; row < rows && ok; row += gridDim.x) {
            const int b = int(row / T);
            const int G = __ldg(seq_len + b) / P;
            const int32_t *gl = idx + row * k;
            float o[kNH];
#pragma unroll
            for (int h = 0; h < kNH; ++h) o[h] = 0.f;
            m_run = -INFINITY;
            l_run = 0.f;
            // o = a o + O_c for the chunk with index gcf over the CTA's rows
            auto fold = [&](uint32_t gcf) {
                const int fb = int(gcf & 1u);
                ok = ok && __all_sync(0xffffffffu, wait_phase(ofull + fb, (gcf >> 1) & 1u, abort_flag));
                tc_fence_after();
                uint32_t r[32];
                if (ok) {
                    tc_ld32(lane_addr + kColO + fb * kNPV, r);
                    tc_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) bar_arrive(ofree + fb);
                if (ok) {
#pragma unroll
                    for (int h4 = 0; h4 < kNH / 4; ++h4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(alph + fb * 32 + 4 * h4);
                        o[4 * h4 + 0] = fmaf(o[4 * h4 + 0], a4.x, __uint_as_float(r[4 * h4 + 0]));
                        o[4 * h4 + 1] = fmaf(o[4 * h4 + 1], a4.y, __uint_as_float(r[4 * h4 + 1]));
                        o[4 * h4 + 2] = fmaf(o[4 * h4 + 2], a4.z, __uint_as_float(r[4 * h4 + 2]));
                        o[4 * h4 + 3] = fmaf(o[4 * h4 + 3], a4.w, __uint_as_float(r[4 * h4 + 3]));
                    }
                }
            };
            // mcur: the row's softmax reference per head, in shared memory
            // (uniform; only warp 0 writes it, between the slow path's barriers)
            if (warp == 0) mcur[lane] = -INFINITY;
            softmax_sync_or(false);
            unsigned char *pt_base = smem + kSmP;
            // p = 2^(z - mref) for this token's heads -> its row of P (bf16,
            // 128B-swizzled MN-major: 8 heads per 16-byte chunk); s: z in, p out
            auto write_p = [&](uint32_t (&s)[32], unsigned char *pt) {
#pragma unroll
                for (int h8 = 0; h8 < kNH / 8; ++h8) {
                    uint32_t pw[4];
#pragma unroll
                    for (int hq = 0; hq < 2; ++hq) {
                        const int h0 = 8 * h8 + 4 * hq;
                        const float4 m4 = *reinterpret_cast<const float4 *>(mcur + h0);
                        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
                        float pp[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float z = __uint_as_float(s[h0 + e]);
                            pp[e] = z == -INFINITY ? 0.f : exp2_hw(z - mm[e]);
                            s[h0 + e] = __float_as_uint(pp[e]);
                        }
                        pw[2 * hq] = pack_bf2_rn(pp[0], pp[1]);
                        pw[2 * hq + 1] = pack_bf2_rn(pp[2], pp[3]);
                    }
                    *reinterpret_cast<uint4 *>(pt + sw128_offset(tid, 8 * h8, 1024)) =
                        make_uint4(pw[0], pw[1], pw[2], pw[3]);
                }
            };
            // the group of this thread's token in chunk c (loaded a chunk ahead)
            auto group_of = [&](int c) {
                const int j = (c * kTok + tid) >> lp2;
                return (c < nck && j < k) ? __ldg(gl + j) : -1;
            };
            int g_next = group_of(0);
            for (int c = 0; c < nck; ++c) {
                const uint32_t gc = n_ck + uint32_t(c);
                const int buf = int(gc & 1u);
                const uint32_t bpar = (gc >> 1) & 1u;
                const int g = g_next;
                g_next = group_of(c + 1);
                ok = ok && __all_sync(0xffffffffu, wait_phase(sfull + buf, bpar, abort_flag));
                tc_fence_after();
                uint32_t s[32];
                if (ok) {
                    tc_ld32(lane_addr + kColS + buf * kNH, s);
                    tc_wait_ld();
                }
                // this thread's token: z = scale * q.k in the log2 domain, or
                // -inf for padding and groups past the sequence
                const bool tv = ok && g >= 0 && g < G;
                bool exceed = false;  // a score above its head's reference + kLazy
#pragma unroll
                for (int h4 = 0; h4 < kNH / 4; ++h4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(mcur + 4 * h4);
                    const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = 4 * h4 + e;
                        const float z = tv ? __uint_as_float(s[h]) * scale_log2 : -INFINITY;
                        s[h] = __float_as_uint(z);
                        exceed |= z > mm[e] + kLazy;
                    }
                }
                // P with the current reference (kept unless a score exceeds it)
                ok = ok && __all_sync(0xffffffffu, wait_phase(pempty + buf, bpar ^ 1u, abort_flag));
                unsigned char *pt = pt_base + buf * kPBytes;
                write_p(s, pt);
                if (softmax_sync_or(exceed || !ok)) {
                    // a new reference: the exact chunk maximum of every head
                    // (the scores again from TMEM; the buffer is still held)
                    if (ok) {
                        tc_ld32(lane_addr + kColS + buf * kNH, s);
                        tc_wait_ld();
                    }
#pragma unroll
                    for (int h = 0; h < kNH; ++h)
                        s[h] = __float_as_uint(tv ? __uint_as_float(s[h]) * scale_log2 : -INFINITY);
                    float *wrow = wmax + (buf * 4 + warp) * 32;
#pragma unroll
                    for (int h = 0; h < kNH; ++h) {
                        const float m = warp_max(__uint_as_float(s[h]));
                        if (lane == 0) wrow[h] = m;
                    }
                    if (softmax_sync_or(!ok)) {
                        ok = false;
                        break;
                    }
                    if (warp == 0) {  // lane h: head h's new reference and rescale
                        const float *w4 = wmax + buf * 4 * 32 + lane;
                        const float cm = fmaxf(fmaxf(w4[0], w4[32]), fmaxf(w4[64], w4[96]));
                        const float mn = fmaxf(m_run, cm);
                        const float a = mn == -INFINITY ? 1.f : exp2_hw(m_run - mn);
                        alph[buf * 32 + lane] = a;
                        mcur[lane] = mn;
                        m_run = mn;
                        if (c > 0) {  // the previous chunk's sums, then the rescale
                            const float *ls = lsum + (buf ^ 1) * 4 * 32 + lane;
                            l_run += (ls[0] + ls[32]) + (ls[64] + ls[96]);
                        }
                        l_run *= a;
                    }
                    softmax_sync_or(false);
                    write_p(s, pt);
                } else if (warp == 0) {  // same reference: rescale 1
                    alph[buf * 32 + lane] = 1.f;
                    if (c > 0) {
                        const float *ls = lsum + (buf ^ 1) * 4 * 32 + lane;
                        l_run += (ls[0] + ls[32]) + (ls[64] + ls[96]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) bar_arrive(sfree + buf);
                fence_async_smem();  // P, for the tensor core's reads
                __syncwarp();
                if (lane == 0) bar_arrive(pfull + buf);
                // the warp's sums of p: halve the 32 values at every step so
                // that lane h ends with head h's sum
#pragma unroll
                for (int hw = 16; hw >= 1; hw >>= 1) {
                    const bool upper = (lane & hw) != 0;
#pragma unroll
                    for (int i = 0; i < hw; ++i) {
                        const float keep = __uint_as_float(upper ? s[i + hw] : s[i]);
                        const float send = __uint_as_float(upper ? s[i] : s[i + hw]);
                        s[i] = __float_as_uint(keep + __shfl_xor_sync(0xffffffffu, send, hw));
                    }
                }
                lsum[(buf * 4 + warp) * 32 + lane] = __uint_as_float(s[0]);
                if (c > 0) fold(gc - 1u);
            }
            // (this barrier also orders warp 0's rescale of the last chunk,
            // written after the chunk's vote, before the other warps' fold)
            if (softmax_sync_or(!ok)) {
                ok = false;
                break;
            }
            if (ok) fold(n_ck + uint32_t(nck) - 1u);
            if (warp == 0) {  // the last chunk's sums complete the row's
                const float *ls = lsum + ((n_ck + uint32_t(nck) - 1u) & 1u) * 4 * 32 + lane;
                const float L = l_run + ((ls[0] + ls[32]) + (ls[64] + ls[96]));
                ltot[lane] = L;
                if (lse && lane < H_q)
                    lse[row * H_q + lane] = L > 0.f ? (m_run + log2f(L)) * kLn2f : -INFINITY;
            }
            if (softmax_sync_or(!ok)) {  // the fold can give up: leave together
                ok = false;
                break;
            }
            // the normalised output: thread tid is value dim tid of every head
            uint16_t *orow = out + row * int64_t(H_q) * kDim + tid;
#pragma unroll
            for (int h = 0; h < kNH; ++h) {
                if (h < H_q) {
                    const float L = ltot[h];
                    orow[h * kDim] = f2bf(L > 0.f ? o[h] * (1.f / L) : 0.f);
                }
            }
            n_ck += uint32_t(nck);
        }
        if (!ok && tid == 0) give_up(13);
    }
    // every role is done (the MMA warp saw its last products complete)
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_free(tb, kTmemCols);
}

int sm_count() {
    static int n[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (n[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
            v = 148;
        n[dev] = v;
    }
    return n[dev];
}

}  // namespace

bool sparse_attn_tc_supported(int64_t rows, int H_q, int d_qk, int d_v, int P, int k) {
    return rows >= 1 && H_q >= 1 && H_q <= kNH && d_qk == kDim && d_v == kDim &&
           (P == 1 || P == 2 || P == 4 || P == 8) && k >= 1 && int64_t(k) * P <= (1 << 24);
}

cudaError_t launch_sparse_attn_tc(const uint16_t *q, const uint16_t *K, int64_t sK_b,
                                  const uint16_t *V, int64_t sV_b, const int32_t *seq_len,
                                  const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v,
                                  int P, int k, float scale, uint16_t *out, float *lse,
                                  int *status, cudaStream_t st, bool test_skip_gather) {
    const int64_t rows = int64_t(B) * T;
    if (rows == 0) return cudaSuccess;
    if (!sparse_attn_tc_supported(rows, H_q, d_qk, d_v, P, k)) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t grid = rows < sm_count() ? rows : sm_count();
    sparse_attn_tc_kernel<<<unsigned(grid), kThr, kSmemBytes, st>>>(
        q, K, sK_b, V, sV_b, seq_len, idx, T, H_q, P, k, rows, scale * 1.4426950408889634f, out,
        lse, status, test_skip_gather ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace lcsw
