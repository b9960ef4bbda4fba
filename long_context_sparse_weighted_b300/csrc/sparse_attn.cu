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
#include "attn_core.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

constexpr int kAttnThreads = 128;
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
    const int tid = threadIdx.x, warp = tid >> 5;
    const int G = __ldg(seq_len + b) / P;
    const int gps = (k + S - 1) / S;
    const int j0 = s * gps, j1 = min(k, j0 + gps);
    const int gpc = kChunk / P;  // groups per chunk
    const int nchunks = j1 > j0 ? (j1 - j0 + gpc - 1) / gpc : 0;
    const int32_t *irow = idx + row * k;
    const uint16_t *kb = K + int64_t(b) * sK_b;
    const uint16_t *vb = V + int64_t(b) * sV_b;

    // warp -> (head tile, token quarter)
    const int MT = HG / 16;  // 1, 2 or 4
    const int TS = 4 / MT;   // token splits of a chunk
    const int mt = warp % MT, ts = warp / MT;
    const int ntok = kChunk / TS;
    const int tok0 = ts * ntok;

    const uint16_t *qrow = q + (row * H_q + hg0) * DQK;
    for (int p = tid; p < HG * (DQK / 8); p += kAttnThreads) {
        const int h = p / (DQK / 8), c8 = p % (DQK / 8);
        *reinterpret_cast<uint4 *>(sq + h * L::QP + c8 * 8) =
            ld_nc16(qrow + int64_t(h) * DQK + c8 * 8);
    }
    auto issue = [&](int ci, int buf) {
        const int jb = j0 + ci * gpc;
        gather_chunk<DQK, DV>(sk + buf * kChunk * L::QP, sv + buf * kChunk * L::VP,
                              sgrp + buf * kChunk, irow + jb, min(gpc, j1 - jb), P, G, kb, vb,
                              L::QP, L::VP, tid, kAttnThreads);
    };
    if (nchunks > 0) issue(0, 0);
    __syncthreads();  // Q in shared

    uint32_t qa[DQK / 16][4];
    load_q_frags<DQK>(qa, sq, L::QP, mt);
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
        attn_chunk<DQK, DV>(st, qa, sk + buf * kChunk * L::QP, sv + buf * kChunk * L::VP,
                            sgrp + buf * kChunk, L::QP, L::VP, P, tok0, ntok, scale_log2);
        __syncthreads();  // buffer reuse
    }
    store_warp_state<DV>(st, state + warp * 16 * (DV + 2));
    __syncthreads();
    for (int p = tid; p < HG * (DV / 2); p += kAttnThreads) {
        const int hl = p / (DV / 2), d2 = (p % (DV / 2)) * 2;
        float Lsum;
        const float4 r = merge_states<DV>(state, MT, TS, hl, d2, Lsum);
        const int h = hg0 + hl;
        if (S == 1) {
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
            *reinterpret_cast<uint32_t *>(out + (row * H_q + h) * DV + d2) =
                pack_bf2(r.z * inv, r.w * inv);
            if (lse && d2 == 0)
                lse[row * H_q + h] = Lsum > 0.f ? (r.x + log2f(Lsum)) * kLn2 : -INFINITY;
        } else {
            const int64_t pi = (row * S + s) * H_q + h;
            *reinterpret_cast<float2 *>(part_o + pi * DV + d2) = make_float2(r.z, r.w);
            if (d2 == 0) part_ml[pi] = make_float2(r.x, Lsum);
        }
    }
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
