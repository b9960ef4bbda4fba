// Sparse attention over the selected history ("G2C Brief -- GLM-5.3-Flash",
// DSA section: "attention over selected history"), one shared K/V head for
// every query head (the MQA form of absorbed latent attention), split-K over
// the selected tokens.
//
// Kernel 1 (split): thread block (split s, row, head group) owns a contiguous
// slice of the row's selected groups.  It gathers their P*|slice| key/value
// rows with 16-byte cp.async into double-buffered shared memory (64 tokens a
// chunk; groups outside [0, seq_len/P) are zero-filled and masked), computes
// S = Q K^T and O += P V on the tensor cores (mma.sync m16n8k16, fp32
// accumulators) with an online softmax in the log2 domain, merges the warps
// that shared a head tile, and writes (m, l, o) for its slice -- or the
// normalised bf16 output directly when the row has one split.
//
// Kernel 2 (combine): one warp per (row, head) merges the S partial states:
// M = max m_s, L = sum exp2(m_s - M) l_s, out = sum exp2(m_s - M) o_s / L.
#include "common.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kChunk = 64;        // tokens per chunk
constexpr int kHeadGroup = 64;    // heads per thread block (4 warps x 16)
constexpr int kTargetBlocks = 296;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int DQK, int DV>
struct AttnSmem {
    static constexpr int QP = DQK + 8;  // row pitch in elements (16-byte pad)
    static constexpr int VP = DV + 8;
    static constexpr int q_bytes = kHeadGroup * QP * 2;
    static constexpr int k_bytes = kChunk * QP * 2;
    static constexpr int v_bytes = kChunk * VP * 2;
    static constexpr int kv_bytes = 2 * (k_bytes + v_bytes);
    static constexpr int state_bytes = 4 * 16 * (DV + 2) * 4;
    static constexpr int body = kv_bytes > state_bytes ? kv_bytes : state_bytes;
    static constexpr int total = q_bytes + body + 2 * kChunk * 4;
};

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

template <int DQK, int DV>
__global__ void __launch_bounds__(kAttnThreads) sparse_attn_split_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ K, int64_t sK_b,
    const uint16_t *__restrict__ V, int64_t sV_b, const int32_t *__restrict__ seq_len,
    const int32_t *__restrict__ idx, int T, int H_q, int P, int k, int S, float scale_log2,
    uint16_t *__restrict__ out, float *__restrict__ lse, float *__restrict__ part_o,
    float2 *__restrict__ part_ml) {
    using L = AttnSmem<DQK, DV>;
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t *sq = reinterpret_cast<uint16_t *>(smem);
    uint16_t *sk = reinterpret_cast<uint16_t *>(smem + L::q_bytes);
    uint16_t *sv = reinterpret_cast<uint16_t *>(smem + L::q_bytes + 2 * L::k_bytes);
    float *state = reinterpret_cast<float *>(smem + L::q_bytes);
    int *sgrp = reinterpret_cast<int *>(smem + L::q_bytes + L::body);  // [2][kChunk]

    const int s = blockIdx.x;
    const int64_t row = blockIdx.y;
    const int hg0 = blockIdx.z * kHeadGroup;
    const int HG = min(kHeadGroup, H_q - hg0);
    const int b = int(row / T);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = __ldg(seq_len + b) / P;
    const int gps = (k + S - 1) / S;
    const int j0 = s * gps, j1 = min(k, j0 + gps);
    const int gpc = kChunk / P;  // groups per chunk
    const int nchunks = j1 > j0 ? (j1 - j0 + gpc - 1) / gpc : 0;
    const int32_t *irow = idx + row * k;

    // warp -> (head tile, token quarter)
    const int MT = HG / 16;                 // 1, 2 or 4
    const int TS = 4 / MT;                  // token splits of a chunk
    const int mt = warp % MT, ts = warp / MT;
    const int ntok = kChunk / TS;           // 64, 32 or 16 tokens per warp
    const int tok0 = ts * ntok;

    // ---- Q tile to shared, then A fragments to registers -----------------
    const uint16_t *qrow = q + (row * H_q + hg0) * DQK;
    for (int p = tid; p < HG * (DQK / 8); p += kAttnThreads) {
        const int h = p / (DQK / 8), c8 = p % (DQK / 8);
        *reinterpret_cast<uint4 *>(sq + h * L::QP + c8 * 8) =
            ld_nc16(qrow + int64_t(h) * DQK + c8 * 8);
    }

    auto issue_chunk = [&](int ci, int buf) {
        const int jb = j0 + ci * gpc;
        if (tid < gpc) {
            const int j = jb + tid;
            int g = (j < j1) ? __ldg(irow + j) : -1;
            sgrp[buf * kChunk + tid] = (g >= 0 && g < G) ? g : -1;
        }
        uint16_t *dk = sk + buf * kChunk * L::QP;
        uint16_t *dv = sv + buf * kChunk * L::VP;
        const uint16_t *kb = K + int64_t(b) * sK_b;
        const uint16_t *vb = V + int64_t(b) * sV_b;
        for (int p = tid; p < kChunk * (DQK / 8); p += kAttnThreads) {
            const int tr = p / (DQK / 8), c8 = p % (DQK / 8);
            const int j = jb + tr / P;
            int g = (j < j1) ? __ldg(irow + j) : -1;
            const bool ok = g >= 0 && g < G;
            const uint16_t *src = ok ? kb + (int64_t(g) * P + tr % P) * DQK + c8 * 8 : kb;
            cp_async16(smem_u32(dk + tr * L::QP + c8 * 8), src, ok ? 16 : 0);
        }
        for (int p = tid; p < kChunk * (DV / 8); p += kAttnThreads) {
            const int tr = p / (DV / 8), c8 = p % (DV / 8);
            const int j = jb + tr / P;
            int g = (j < j1) ? __ldg(irow + j) : -1;
            const bool ok = g >= 0 && g < G;
            const uint16_t *src = ok ? vb + (int64_t(g) * P + tr % P) * DV + c8 * 8 : vb;
            cp_async16(smem_u32(dv + tr * L::VP + c8 * 8), src, ok ? 16 : 0);
        }
        cp_async_commit();
    };

    if (nchunks > 0) issue_chunk(0, 0);
    __syncthreads();  // Q in shared

    uint32_t qa[DQK / 16][4];
    {
        const int r = mt * 16 + (lane & 15), cc = (lane >> 4) * 8;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
            ldmatrix_x4(smem_u32(sq + r * L::QP + kk * 16 + cc), qa[kk][0], qa[kk][1], qa[kk][2],
                        qa[kk][3]);
    }

    float o[DV / 8][4];
#pragma unroll
    for (int i = 0; i < DV / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int c = lane & 3;

    for (int ci = 0; ci < nchunks; ++ci) {
        const int buf = ci & 1;
        if (ci + 1 < nchunks) {
            issue_chunk(ci + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint16_t *ck = sk + buf * kChunk * L::QP;
        const uint16_t *cv = sv + buf * kChunk * L::VP;
        const int *cg = sgrp + buf * kChunk;

        constexpr int MAXNT = kChunk / 8;  // 8 n-tiles max
        float sacc[MAXNT][4];
#pragma unroll
        for (int nt = 0; nt < MAXNT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
        for (int nt = 0; nt < MAXNT; ++nt) {
            if (nt * 8 >= ntok) break;
            const int trow = tok0 + nt * 8 + (lane & 7);
#pragma unroll
            for (int kk = 0; kk < DQK / 16; kk += 2) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(smem_u32(ck + trow * L::QP + kk * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
                mma_bf16_16816(sacc[nt], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                if (kk + 1 < DQK / 16)
                    mma_bf16_16816(sacc[nt], qa[kk + 1][0], qa[kk + 1][1], qa[kk + 1][2],
                                   qa[kk + 1][3], b2, b3);
            }
        }
        // scale, mask, online softmax
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < MAXNT; ++nt) {
            if (nt * 8 >= ntok) break;
            const int n0 = tok0 + nt * 8 + 2 * c;
            const bool v0 = cg[n0 / P] >= 0, v1 = cg[(n0 + 1) / P] >= 0;
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
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
        const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m0 - ref0), al1 = fast_exp2(m1 - ref1);
        m0 = mn0;
        m1 = mn1;
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int i = 0; i < DV / 8; ++i) {
            o[i][0] *= al0; o[i][1] *= al0;
            o[i][2] *= al1; o[i][3] *= al1;
        }
#pragma unroll
        for (int nt = 0; nt < MAXNT; ++nt) {
            if (nt * 8 >= ntok) break;
            sacc[nt][0] = fast_exp2(sacc[nt][0] - ref0);
            sacc[nt][1] = fast_exp2(sacc[nt][1] - ref0);
            sacc[nt][2] = fast_exp2(sacc[nt][2] - ref1);
            sacc[nt][3] = fast_exp2(sacc[nt][3] - ref1);
            l0 += sacc[nt][0] + sacc[nt][1];
            l1 += sacc[nt][2] + sacc[nt][3];
        }
        // O += P V
#pragma unroll
        for (int kt = 0; kt < MAXNT / 2; ++kt) {
            if (kt * 16 >= ntok) break;
            const uint32_t pa0 = pack_bf2(sacc[2 * kt][0], sacc[2 * kt][1]);
            const uint32_t pa1 = pack_bf2(sacc[2 * kt][2], sacc[2 * kt][3]);
            const uint32_t pa2 = pack_bf2(sacc[2 * kt + 1][0], sacc[2 * kt + 1][1]);
            const uint32_t pa3 = pack_bf2(sacc[2 * kt + 1][2], sacc[2 * kt + 1][3]);
            const int vrow = tok0 + kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int dt = 0; dt < DV / 8; dt += 2) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(smem_u32(cv + vrow * L::VP + (dt + (lane >> 4)) * 8), b0, b1,
                                  b2, b3);
                mma_bf16_16816(o[dt], pa0, pa1, pa2, pa3, b0, b1);
                mma_bf16_16816(o[dt + 1], pa0, pa1, pa2, pa3, b2, b3);
            }
        }
        __syncthreads();  // buffer reuse
    }

    // ---- per-warp state -> shared, merge warps of the same head tile ------
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __syncthreads();
    {
        float *ws_ = state + warp * 16 * (DV + 2);
        const int r0 = lane >> 2;
#pragma unroll
        for (int i = 0; i < DV / 8; ++i) {
            ws_[r0 * (DV + 2) + i * 8 + 2 * c] = o[i][0];
            ws_[r0 * (DV + 2) + i * 8 + 2 * c + 1] = o[i][1];
            ws_[(r0 + 8) * (DV + 2) + i * 8 + 2 * c] = o[i][2];
            ws_[(r0 + 8) * (DV + 2) + i * 8 + 2 * c + 1] = o[i][3];
        }
        if (c == 0) {
            ws_[r0 * (DV + 2) + DV] = m0;
            ws_[r0 * (DV + 2) + DV + 1] = l0;
            ws_[(r0 + 8) * (DV + 2) + DV] = m1;
            ws_[(r0 + 8) * (DV + 2) + DV + 1] = l1;
        }
    }
    __syncthreads();
    // one thread per (head, 2 dims)
    for (int p = tid; p < HG * (DV / 2); p += kAttnThreads) {
        const int hl = p / (DV / 2), d2 = (p % (DV / 2)) * 2;
        const int tile = hl / 16, rr = hl % 16;
        float M = -INFINITY;
        for (int t2 = 0; t2 < TS; ++t2) {
            const float *st = state + (t2 * MT + tile) * 16 * (DV + 2) + rr * (DV + 2);
            M = fmaxf(M, st[DV]);
        }
        const float ref = M == -INFINITY ? 0.f : M;
        float Lsum = 0.f, oa = 0.f, ob = 0.f;
        for (int t2 = 0; t2 < TS; ++t2) {
            const float *st = state + (t2 * MT + tile) * 16 * (DV + 2) + rr * (DV + 2);
            const float f = fast_exp2(st[DV] - ref);
            Lsum += f * st[DV + 1];
            oa += f * st[d2];
            ob += f * st[d2 + 1];
        }
        const int h = hg0 + hl;
        if (S == 1) {
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
            *reinterpret_cast<uint32_t *>(out + (row * H_q + h) * DV + d2) =
                pack_bf2(oa * inv, ob * inv);
            if (lse && d2 == 0)
                lse[row * H_q + h] = Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY;
        } else {
            const int64_t pi = (row * S + s) * H_q + h;
            *reinterpret_cast<float2 *>(part_o + pi * DV + d2) = make_float2(oa, ob);
            if (d2 == 0) part_ml[pi] = make_float2(M, Lsum);
        }
    }
}

template <int DV>
__global__ void __launch_bounds__(256) splitk_combine_kernel(
    const float *__restrict__ part_o, const float2 *__restrict__ part_ml, int H_q, int S,
    uint16_t *__restrict__ out, float *__restrict__ lse) {
    const int64_t row = blockIdx.x;
    const int h = blockIdx.y * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (h >= H_q) return;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, part_ml[(row * S + s) * H_q + h].x);
    const float ref = M == -INFINITY ? 0.f : M;
    constexpr int PER = DV / 32;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float Lsum = 0.f;
    for (int s = 0; s < S; ++s) {
        const int64_t pi = (row * S + s) * H_q + h;
        const float2 ml = part_ml[pi];
        const float f = exp2f(ml.x - ref);
        Lsum += f * ml.y;
        const float *po = part_o + pi * DV + lane * PER;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] += f * po[i];
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    uint16_t *orow = out + (row * H_q + h) * DV + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; i += 2)
        *reinterpret_cast<uint32_t *>(orow + i) = pack_bf2(acc[i] * inv, acc[i + 1] * inv);
    if (lse && lane == 0) lse[row * H_q + h] = Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY;
}

template <int DQK, int DV>
cudaError_t launch_typed(const uint16_t *q, const uint16_t *K, int64_t sK_b, const uint16_t *V,
                         int64_t sV_b, const int32_t *seq_len, const int32_t *idx, int B, int T,
                         int H_q, int P, int k, float scale, uint16_t *out, float *lse,
                         void *ws, cudaStream_t st) {
    const int64_t rows = int64_t(B) * T;
    const int S = sparse_attn_splits(rows, H_q, k, P);
    const int HGs = (H_q + kHeadGroup - 1) / kHeadGroup;
    using L = AttnSmem<DQK, DV>;
    auto kern = sparse_attn_split_kernel<DQK, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
    if (e != cudaSuccess) return e;
    float *part_o = reinterpret_cast<float *>(ws);
    float2 *part_ml = reinterpret_cast<float2 *>(
        reinterpret_cast<char *>(ws) + size_t(rows) * S * H_q * DV * sizeof(float));
    if (rows > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid(S, unsigned(rows), HGs);
    kern<<<grid, kAttnThreads, L::total, st>>>(q, K, sK_b, V, sV_b, seq_len, idx, T, H_q, P, k, S,
                                               scale * kLog2e, out, lse, part_o, part_ml);
    e = cudaGetLastError();
    if (e != cudaSuccess || S == 1) return e;
    dim3 g2(unsigned(rows), (H_q + 7) / 8);
    splitk_combine_kernel<DV><<<g2, 256, 0, st>>>(part_o, part_ml, H_q, S, out, lse);
    return cudaGetLastError();
}

}  // namespace

int sparse_attn_splits(int64_t rows, int H_q, int k, int P) {
    const int64_t HGs = (H_q + kHeadGroup - 1) / kHeadGroup;
    const int64_t chunks = (int64_t(k) * P + kChunk - 1) / kChunk;
    int64_t want = (kTargetBlocks + rows * HGs - 1) / (rows * HGs);
    if (want > chunks) want = chunks;
    if (want > k) want = k;
    if (want < 1) want = 1;
    return int(want);
}

size_t sparse_attn_ws_bytes(int64_t rows, int H_q, int d_v, int k, int P) {
    const int S = sparse_attn_splits(rows, H_q, k, P);
    if (S == 1) return 0;
    return size_t(rows) * S * H_q * (size_t(d_v) * sizeof(float) + sizeof(float2));
}

cudaError_t launch_sparse_attn(const uint16_t *q, const uint16_t *K, int64_t sK_b,
                               const uint16_t *V, int64_t sV_b, const int32_t *seq_len,
                               const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v,
                               int P, int k, float scale, uint16_t *out, float *lse, void *ws,
                               cudaStream_t st) {
    if (int64_t(B) * T == 0) return cudaSuccess;
#define LCSW_ATT(DQ, DVV)                                                                   \
    if (d_qk == DQ && d_v == DVV)                                                          \
        return launch_typed<DQ, DVV>(q, K, sK_b, V, sV_b, seq_len, idx, B, T, H_q, P, k,  \
                                     scale, out, lse, ws, st);
    LCSW_ATT(64, 64)
    LCSW_ATT(128, 64)
    LCSW_ATT(128, 128)
    LCSW_ATT(192, 128)
    LCSW_ATT(192, 64)
    LCSW_ATT(64, 128)
#undef LCSW_ATT
    return cudaErrorInvalidValue;
}

}  // namespace lcsw
