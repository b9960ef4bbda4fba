// Sparse attention in the MLA latent geometry: one 576-wide row per token
// holds the rank-512 latent c and a 64-wide rotary key part; the latent is
// both the key's first 512 dims and the value ("G2C Brief -- GLM-5.3-Flash":
// MLA rank 512 per token, kv_lora_rank 512, in "The release in one page" and
// the DSA section's "MLA latent cache (rank 512 per token)").  With the query
// absorbed into the latent space (q = [q_c (512) | q_rope (64)] per head),
//
//   z_j = scale * q . kv_j              (576 dims)
//   o   = sum_j softmax(z)_j kv_j[0:512]
//
// over the tokens of the selected groups, one latent row shared by every
// query head.  The pages give the rank, not the rotary width; 64 is taken.
//
// Kernel 1 (split): block (split s, row, 32-head group), 8 warps.  Chunks of
// 64 tokens are gathered with 16-byte cp.async into two shared buffers of
// [64][576] rows (the value operand is the same buffer's first 512 columns,
// so each token is read once: 1,152 bytes).  Warp (t, q): head tile t (16
// heads) scores token quarter q of the chunk (S = Q K^T on mma.sync), the
// four quarters exchange row maxima and P = 2^(s - m) (bf16) through shared
// memory, then warp (t, q) accumulates value dims [128 q, 128 q + 128) of
// O += P V over all 64 tokens for its 16 heads.  Each block writes its
// partial (m, l, O) per head, or the normalised output with one split.
// Kernel 2 (combine): one block per (row, head) merges the splits.
//
// Both launch as programmatic dependents of the kernel before them in the
// stream where that is safe (sm_90+ dependent launch): the combine always
// (its only input is the split kernel's output), the split kernel when the
// decode step's selection kernel precedes it.  Such a kernel may be
// scheduled before its predecessor ends; it reads what the predecessor
// writes (idx, the partial states) only after griddepcontrol.wait, which
// returns once that grid has completed and its writes are visible, and is
// a no-op in a kernel launched the ordinary way.
#include "common.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

__device__ __forceinline__ void wait_for_predecessor() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void let_dependents_start() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kLat = 512;              // latent (value) width
constexpr int kDqk = 576;              // latent + rotary key width
constexpr int kTok = 64;               // tokens per chunk
constexpr int kHg = 32;                // heads per block
constexpr int kThr = 256;              // 8 warps: 2 head tiles x 4 quarters
constexpr int kQP = kDqk + 8;          // padded row pitch (elements)
constexpr int kPP = kTok + 8;
constexpr int kTarget = 296;           // blocks wanted per launch
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct MlaSmem {
    static constexpr int q = 0;                                  // [kHg][kQP] bf16
    static constexpr int kv = q + kHg * kQP * 2;                 // [2][kTok][kQP] bf16
    static constexpr int p = kv + 2 * kTok * kQP * 2;            // [kHg][kPP] bf16
    static constexpr int rm = p + kHg * kPP * 2;                 // [4][kHg] f32
    static constexpr int rl = rm + 4 * kHg * 4;                  // [4][kHg] f32
    static constexpr int g = rl + 4 * kHg * 4;                   // [2][kTok] int
    static constexpr int total = g + 2 * kTok * 4;
};
static_assert(MlaSmem::total <= 227 * 1024, "MLA attention operands overflow shared memory");

// cp.async gather of one chunk: the rows of groups glist[0..n) (n <= kTok/P)
// of a sequence with complete groups [0, G); invalid groups are zero-filled
// and get id -1.
__device__ __forceinline__ void gather_rows(uint16_t *dst, int *sg, const int32_t *glist, int n,
                                            int P, int G, const uint16_t *kvb) {
    const int tid = threadIdx.x;
    if (tid < kTok / P) {
        const int g = tid < n ? glist[tid] : -1;
        sg[tid] = (g >= 0 && g < G) ? g : -1;
    }
    for (int e = tid; e < kTok * (kDqk / 8); e += kThr) {
        const int tr = e / (kDqk / 8), c8 = e % (kDqk / 8);
        const int q = tr / P;
        const int g = q < n ? glist[q] : -1;
        const bool ok = g >= 0 && g < G;
        const uint16_t *src = ok ? kvb + (int64_t(g) * P + tr % P) * kDqk + c8 * 8 : kvb;
        cp_async16(smem_u32(dst + tr * kQP + c8 * 8), src, ok ? 16 : 0);
    }
    cp_async_commit();
}

__global__ void __launch_bounds__(kThr, 1) sparse_attn_mla_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ kv, int64_t skv_b,
    const int32_t *__restrict__ seq_len, const int32_t *__restrict__ idx, int T, int H_q, int P,
    int k, int S, float scale_log2, uint16_t *__restrict__ out, float *__restrict__ lse,
    float *__restrict__ part_o, float2 *__restrict__ part_ml) {
    extern __shared__ __align__(16) unsigned char smem[];
    using L = MlaSmem;
    uint16_t *sq = reinterpret_cast<uint16_t *>(smem + L::q);
    uint16_t *skv = reinterpret_cast<uint16_t *>(smem + L::kv);
    uint16_t *sp = reinterpret_cast<uint16_t *>(smem + L::p);
    float *red_m = reinterpret_cast<float *>(smem + L::rm);
    float *red_l = reinterpret_cast<float *>(smem + L::rl);
    int *sgid = reinterpret_cast<int *>(smem + L::g);

    const int s = blockIdx.x;
    const int64_t row = blockIdx.y;
    const int hg0 = blockIdx.z * kHg;
    const int HG = min(kHg, H_q - hg0);  // 16 or 32
    const int b = int(row / T);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = lane & 3, gq = lane >> 2;
    const int mt = warp & 1, qq = warp >> 1;
    const bool wact = mt * 16 < HG;
    const int G = __ldg(seq_len + b) / P;
    const int gps = (k + S - 1) / S;
    const int j0 = s * gps, j1 = min(k, j0 + gps);
    const int gpc = kTok / P;
    const int nchunks = j1 > j0 ? (j1 - j0 + gpc - 1) / gpc : 0;
    const int32_t *irow = idx + row * k;
    const uint16_t *kvb = kv + int64_t(b) * skv_b;

    // Q rows of the head group, then the first chunk
    const uint16_t *qrow = q + (row * H_q + hg0) * kDqk;
    for (int e = tid; e < HG * (kDqk / 8); e += kThr) {
        const int h = e / (kDqk / 8), c8 = e % (kDqk / 8);
        cp_async16(smem_u32(sq + h * kQP + c8 * 8), qrow + int64_t(h) * kDqk + c8 * 8, 16);
    }
    cp_async_commit();
    let_dependents_start();  // the combine may be scheduled now; it waits for this grid
    // idx is the output of the selection kernel before this one (in the
    // decode step): read only after it has completed
    wait_for_predecessor();
    auto issue = [&](int ci) {
        const int jb = j0 + ci * gpc;
        gather_rows(skv + (ci & 1) * kTok * kQP, sgid + (ci & 1) * kTok, irow + jb,
                    min(gpc, j1 - jb), P, G, kvb);
    };
    if (nchunks > 0) issue(0);

    constexpr int NTV = (kLat / 4) / 8;  // 16 n-tiles of 8 value dims per warp
    float o[NTV][4];
#pragma unroll
    for (int i = 0; i < NTV; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int h0 = mt * 16 + gq, h1 = h0 + 8;  // heads within the group
    const int lp2 = 31 - __clz(P);

    for (int ci = 0; ci < nchunks; ++ci) {
        __syncthreads();  // every warp is done with chunk ci - 1, whose buffer comes next
        if (ci + 1 < nchunks) {
            issue(ci + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint16_t *ck = skv + (ci & 1) * kTok * kQP;
        const int *cg = sgid + (ci & 1) * kTok;
        float sacc[2][4];
        if (wact) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll 4
            for (int kk = 0; kk < kDqk / 16; kk += 2) {
                uint32_t a[2][4];
                const int qr = mt * 16 + (lane & 15), qc = (lane >> 4) * 8;
                ldmatrix_x4(smem_u32(sq + qr * kQP + kk * 16 + qc), a[0][0], a[0][1], a[0][2],
                            a[0][3]);
                ldmatrix_x4(smem_u32(sq + qr * kQP + (kk + 1) * 16 + qc), a[1][0], a[1][1],
                            a[1][2], a[1][3]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int trow = qq * 16 + nt * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(smem_u32(ck + trow * kQP + kk * 16 + (lane >> 3) * 8), b0, b1, b2,
                                b3);
                    mma_bf16_16816(sacc[nt], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
                    mma_bf16_16816(sacc[nt], a[1][0], a[1][1], a[1][2], a[1][3], b2, b3);
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int n0 = qq * 16 + nt * 8 + 2 * c;
                const bool v0 = cg[n0 >> lp2] >= 0, v1 = cg[(n0 + 1) >> lp2] >= 0;
                sacc[nt][0] = v0 ? sacc[nt][0] * scale_log2 : -INFINITY;
                sacc[nt][1] = v1 ? sacc[nt][1] * scale_log2 : -INFINITY;
                sacc[nt][2] = v0 ? sacc[nt][2] * scale_log2 : -INFINITY;
                sacc[nt][3] = v1 ? sacc[nt][3] * scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(sacc[nt][0], sacc[nt][1]));
                mx1 = fmaxf(mx1, fmaxf(sacc[nt][2], sacc[nt][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            if (c == 0) {
                red_m[qq * kHg + h0] = mx0;
                red_m[qq * kHg + h1] = mx1;
            }
        }
        __syncthreads();
        float al0 = 1.f, al1 = 1.f;
        if (wact) {
            float cm0 = red_m[h0], cm1 = red_m[h1];
#pragma unroll
            for (int q2 = 1; q2 < 4; ++q2) {
                cm0 = fmaxf(cm0, red_m[q2 * kHg + h0]);
                cm1 = fmaxf(cm1, red_m[q2 * kHg + h1]);
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
                sacc[nt][0] = exp2f(sacc[nt][0] - ref0);
                sacc[nt][1] = exp2f(sacc[nt][1] - ref0);
                sacc[nt][2] = exp2f(sacc[nt][2] - ref1);
                sacc[nt][3] = exp2f(sacc[nt][3] - ref1);
                ls0 += sacc[nt][0] + sacc[nt][1];
                ls1 += sacc[nt][2] + sacc[nt][3];
                const int col = qq * 16 + nt * 8 + 2 * c;
                *reinterpret_cast<uint32_t *>(sp + h0 * kPP + col) = pack_bf2(sacc[nt][0], sacc[nt][1]);
                *reinterpret_cast<uint32_t *>(sp + h1 * kPP + col) = pack_bf2(sacc[nt][2], sacc[nt][3]);
            }
            ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
            ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
            ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
            ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
            if (c == 0) {
                red_l[qq * kHg + h0] = ls0;
                red_l[qq * kHg + h1] = ls1;
            }
        }
        __syncthreads();
        if (wact) {
            l0 = l0 * al0 + red_l[h0] + red_l[kHg + h0] + red_l[2 * kHg + h0] + red_l[3 * kHg + h0];
            l1 = l1 * al1 + red_l[h1] + red_l[kHg + h1] + red_l[2 * kHg + h1] + red_l[3 * kHg + h1];
#pragma unroll
            for (int i = 0; i < NTV; ++i) {
                o[i][0] *= al0; o[i][1] *= al0;
                o[i][2] *= al1; o[i][3] *= al1;
            }
            // O += P V over the chunk's 64 tokens, value dims [128 qq, 128 qq + 128)
#pragma unroll
            for (int kt = 0; kt < kTok / 16; ++kt) {
                uint32_t pa0, pa1, pa2, pa3;
                ldmatrix_x4(smem_u32(sp + (mt * 16 + (lane & 15)) * kPP + kt * 16 + (lane >> 4) * 8),
                            pa0, pa1, pa2, pa3);
                const int vrow = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int dt = 0; dt < NTV; dt += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(
                        smem_u32(ck + vrow * kQP + qq * (kLat / 4) + (dt + (lane >> 4)) * 8), b0,
                        b1, b2, b3);
                    mma_bf16_16816(o[dt], pa0, pa1, pa2, pa3, b0, b1);
                    mma_bf16_16816(o[dt + 1], pa0, pa1, pa2, pa3, b2, b3);
                }
            }
        }
    }
    cp_async_wait<0>();  // the Q rows, when there was no chunk

    if (!wact) return;
    const int hA = hg0 + h0, hB = hg0 + h1;
    if (S == 1) {
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
        for (int i = 0; i < NTV; ++i) {
            const int d = qq * (kLat / 4) + i * 8 + 2 * c;
            *reinterpret_cast<uint32_t *>(out + (row * H_q + hA) * kLat + d) =
                pack_bf2(o[i][0] * i0, o[i][1] * i0);
            *reinterpret_cast<uint32_t *>(out + (row * H_q + hB) * kLat + d) =
                pack_bf2(o[i][2] * i1, o[i][3] * i1);
        }
        if (lse && qq == 0 && c == 0) {
            lse[row * H_q + hA] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
            lse[row * H_q + hB] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
        }
    } else {
        const int64_t pA = (row * S + s) * H_q + hA, pB = (row * S + s) * H_q + hB;
#pragma unroll
        for (int i = 0; i < NTV; ++i) {
            const int d = qq * (kLat / 4) + i * 8 + 2 * c;
            *reinterpret_cast<float2 *>(part_o + pA * kLat + d) = make_float2(o[i][0], o[i][1]);
            *reinterpret_cast<float2 *>(part_o + pB * kLat + d) = make_float2(o[i][2], o[i][3]);
        }
        if (qq == 0 && c == 0) {
            part_ml[pA] = make_float2(l0 > 0.f ? m0 : -INFINITY, l0);
            part_ml[pB] = make_float2(l1 > 0.f ? m1 : -INFINITY, l1);
        }
    }
}

// One block of 128 threads per (row, head): out = sum_s 2^(m_s - M) o_s /
// sum_s 2^(m_s - M) l_s.  Every thread takes the split weights (S <= 64
// words, cached) and four value dims; the splits' rows are loaded eight at a
// time so that their latencies overlap.
constexpr int kCombThreads = kLat / 4;
__global__ void __launch_bounds__(kCombThreads) mla_combine_kernel(
    const float *__restrict__ part_o, const float2 *__restrict__ part_ml, int H_q, int S,
    uint16_t *__restrict__ out, float *__restrict__ lse) {
    const int64_t w = blockIdx.x;  // row * H_q + h
    const int64_t row = w / H_q;
    const int h = int(w % H_q);
    const int t = threadIdx.x;
    auto pidx = [&](int s) { return (row * S + s) * H_q + h; };
    wait_for_predecessor();  // the split kernel's partial states
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldg(&part_ml[pidx(s)].x));
    const float ref = M == -INFINITY ? 0.f : M;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float Lsum = 0.f;
    for (int s0 = 0; s0 < S; s0 += 8) {
        float4 v[8];
        float wgt[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            wgt[u] = 0.f;
            if (s0 + u < S) {
                const float2 ml = __ldg(&part_ml[pidx(s0 + u)]);
                if (ml.y > 0.f) {
                    wgt[u] = exp2f(ml.x - ref);
                    Lsum += wgt[u] * ml.y;
                    v[u] = __ldg(reinterpret_cast<const float4 *>(part_o + pidx(s0 + u) * kLat) + t);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            acc.x += wgt[u] * v[u].x;
            acc.y += wgt[u] * v[u].y;
            acc.z += wgt[u] * v[u].z;
            acc.w += wgt[u] * v[u].w;
        }
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    *reinterpret_cast<uint2 *>(out + w * kLat + t * 4) =
        make_uint2(pack_bf2(acc.x * inv, acc.y * inv), pack_bf2(acc.z * inv, acc.w * inv));
    if (lse && t == 0) lse[w] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
}

}  // namespace

int sparse_attn_mla_splits(int64_t rows, int H_q, int k, int P) {
    const int64_t HGs = (H_q + kHg - 1) / kHg;
    const int64_t chunks = (int64_t(k) * P + kTok - 1) / kTok;
    int64_t want = (kTarget + rows * HGs - 1) / (rows * HGs);
    if (want > chunks) want = chunks;
    if (want < 1) want = 1;
    return int(want);
}

size_t sparse_attn_mla_ws_bytes(int64_t rows, int H_q, int k, int P) {
    const int S = sparse_attn_mla_splits(rows, H_q, k, P);
    if (S == 1) return 0;
    return size_t(rows) * S * H_q * (size_t(kLat) * sizeof(float) + sizeof(float2));
}

cudaError_t launch_sparse_attn_mla(const uint16_t *q, const uint16_t *kv, int64_t skv_b,
                                   const int32_t *seq_len, const int32_t *idx, int B, int T,
                                   int H_q, int P, int k, float scale, uint16_t *out, float *lse,
                                   void *ws, cudaStream_t st, bool after_selection) {
    const int64_t rows = int64_t(B) * T;
    if (rows == 0) return cudaSuccess;
    if (rows > 65535) return cudaErrorInvalidConfiguration;
    const int S = sparse_attn_mla_splits(rows, H_q, k, P);
    const int HGs = (H_q + kHg - 1) / kHg;
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_mla_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         MlaSmem::total);
    if (e != cudaSuccess) return e;
    float *part_o = reinterpret_cast<float *>(ws);
    float2 *part_ml = reinterpret_cast<float2 *>(
        reinterpret_cast<char *>(ws) + size_t(rows) * S * H_q * kLat * sizeof(float));
    cudaLaunchAttribute dep[1];
    dep[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    dep[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, unsigned(rows), HGs);
    cfg.blockDim = dim3(kThr);
    cfg.dynamicSmemBytes = MlaSmem::total;
    cfg.stream = st;
    // (standalone, the kernel before may be the one that writes q: an
    // ordinary launch; after the decode step's selection, q is an input)
    cfg.attrs = after_selection ? dep : nullptr;
    cfg.numAttrs = after_selection ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, sparse_attn_mla_kernel, q, kv, skv_b, seq_len, idx, T, H_q, P, k,
                           S, scale * kLog2e, out, lse, part_o, part_ml);
    if (e != cudaSuccess || S == 1) return e;
    cudaLaunchConfig_t cc = {};
    cc.gridDim = dim3(unsigned(rows * H_q));
    cc.blockDim = dim3(kCombThreads);
    cc.stream = st;
    cc.attrs = dep;
    cc.numAttrs = 1;
    return cudaLaunchKernelEx(&cc, mla_combine_kernel, static_cast<const float *>(part_o),
                              static_cast<const float2 *>(part_ml), H_q, S, out, lse);
}

}  // namespace lcsw
