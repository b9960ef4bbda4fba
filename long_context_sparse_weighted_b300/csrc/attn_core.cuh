// Tensor-core tile math of the sparse attention (shared by the split-K kernel
// and the fused decode kernel).
//
// A chunk holds kChunk = 64 gathered tokens (K rows at pitch QP, V rows at
// pitch VP elements, bf16, in shared memory) and the selected-group id of each
// group of P tokens (-1 = masked).  A warp owns one 16-head tile (rows of Q)
// and a contiguous slice of ntok = 64 / TS tokens of the chunk; it keeps an
// online-softmax state (m, l, O) for its 16 heads in the log2 domain.
#pragma once

#include "common.cuh"

namespace lcsw {

constexpr int kChunk = 64;

template <int DV>
struct AttnWarpState {
    float o[DV / 8][4];
    float m0, m1, l0, l1;
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int i = 0; i < DV / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    }
};

// A fragments of the warp's 16-head tile of Q (rows mt*16.., pitch QP).
template <int DQK>
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[DQK / 16][4], const uint16_t *sq,
                                             int QP, int mt) {
    const int lane = threadIdx.x & 31;
    const int r = mt * 16 + (lane & 15), cc = (lane >> 4) * 8;
#pragma unroll
    for (int kk = 0; kk < DQK / 16; ++kk)
        ldmatrix_x4(smem_u32(sq + r * QP + kk * 16 + cc), qa[kk][0], qa[kk][1], qa[kk][2],
                    qa[kk][3]);
}

// One chunk: S = Q K^T (scaled to log2 units), mask, online softmax, O += P V.
// MAXNT bounds the warp's token slice (ntok <= 8*MAXNT).  With QSMEM the Q
// fragments are re-read from shared memory (sq, rows mt*16..) at every k-step
// instead of living in registers (qa unused), for register-limited callers.
//
// With per-token scales (an FP8 K/V cache whose codes were widened exactly to
// bf16): kscale[t] multiplies token t's scores, and vscale[t] its softmax
// weight in the P V product (the sums l use the weights without it).
template <int DQK, int DV, int MAXNT = kChunk / 8, bool QSMEM = false>
__device__ __forceinline__ void attn_chunk(AttnWarpState<DV> &st, const uint32_t (&qa)[DQK / 16][4],
                                           const uint16_t *ck, const uint16_t *cv,
                                           const int *cg, int QP, int VP, int P, int tok0,
                                           int ntok, float scale_log2,
                                           const uint16_t *sq = nullptr, int mt = 0,
                                           const float *kscale = nullptr,
                                           const float *vscale = nullptr) {
    const int lane = threadIdx.x & 31, c = lane & 3;
    float sacc[MAXNT][4];
#pragma unroll
    for (int nt = 0; nt < MAXNT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DQK / 16; kk += 2) {
        uint32_t a[2][4];
        if constexpr (QSMEM) {
            const int qr = mt * 16 + (lane & 15), qc = (lane >> 4) * 8;
            ldmatrix_x4(smem_u32(sq + qr * QP + kk * 16 + qc), a[0][0], a[0][1], a[0][2], a[0][3]);
            ldmatrix_x4(smem_u32(sq + qr * QP + (kk + 1) * 16 + qc), a[1][0], a[1][1], a[1][2],
                        a[1][3]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[0][i] = qa[kk][i];
                a[1][i] = qa[kk + 1][i];
            }
        }
#pragma unroll
        for (int nt = 0; nt < MAXNT; ++nt) {
            if (nt * 8 >= ntok) break;
            const int trow = tok0 + nt * 8 + (lane & 7);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(smem_u32(ck + trow * QP + kk * 16 + (lane >> 3) * 8), b0, b1, b2, b3);
            mma_bf16_16816(sacc[nt], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
            mma_bf16_16816(sacc[nt], a[1][0], a[1][1], a[1][2], a[1][3], b2, b3);
        }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < MAXNT; ++nt) {
        if (nt * 8 >= ntok) break;
        const int n0 = tok0 + nt * 8 + 2 * c;
        const bool v0 = cg[n0 / P] >= 0, v1 = cg[(n0 + 1) / P] >= 0;
        if (kscale) {
            const float k0 = kscale[n0], k1 = kscale[n0 + 1];
            sacc[nt][0] *= k0;
            sacc[nt][1] *= k1;
            sacc[nt][2] *= k0;
            sacc[nt][3] *= k1;
        }
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
    const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
    const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
    const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(st.m0 - ref0), al1 = exp2f(st.m1 - ref1);
    st.m0 = mn0;
    st.m1 = mn1;
    st.l0 *= al0;
    st.l1 *= al1;
#pragma unroll
    for (int i = 0; i < DV / 8; ++i) {
        st.o[i][0] *= al0; st.o[i][1] *= al0;
        st.o[i][2] *= al1; st.o[i][3] *= al1;
    }
#pragma unroll
    for (int nt = 0; nt < MAXNT; ++nt) {
        if (nt * 8 >= ntok) break;
        sacc[nt][0] = exp2f(sacc[nt][0] - ref0);
        sacc[nt][1] = exp2f(sacc[nt][1] - ref0);
        sacc[nt][2] = exp2f(sacc[nt][2] - ref1);
        sacc[nt][3] = exp2f(sacc[nt][3] - ref1);
        st.l0 += sacc[nt][0] + sacc[nt][1];
        st.l1 += sacc[nt][2] + sacc[nt][3];
    }
#pragma unroll
    for (int kt = 0; kt < (MAXNT + 1) / 2; ++kt) {
        if (kt * 16 >= ntok) break;
        float w0 = 1.f, w1 = 1.f, w2 = 1.f, w3 = 1.f;  // value scales of the four tokens
        if (vscale) {
            const int t0 = tok0 + kt * 16 + 2 * c;
            w0 = vscale[t0];
            w1 = vscale[t0 + 1];
            w2 = vscale[t0 + 8];
            w3 = vscale[t0 + 9];
        }
        const uint32_t pa0 = pack_bf2(sacc[2 * kt][0] * w0, sacc[2 * kt][1] * w1);
        const uint32_t pa1 = pack_bf2(sacc[2 * kt][2] * w0, sacc[2 * kt][3] * w1);
        const uint32_t pa2 = pack_bf2(sacc[2 * kt + 1][0] * w2, sacc[2 * kt + 1][1] * w3);
        const uint32_t pa3 = pack_bf2(sacc[2 * kt + 1][2] * w2, sacc[2 * kt + 1][3] * w3);
        const int vrow = tok0 + kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int dt = 0; dt < DV / 8; dt += 2) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(smem_u32(cv + vrow * VP + (dt + (lane >> 4)) * 8), b0, b1, b2, b3);
            mma_bf16_16816(st.o[dt], pa0, pa1, pa2, pa3, b0, b1);
            mma_bf16_16816(st.o[dt + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
    }
}

// Issue the cp.async gather of one chunk: groups glist[0..n) (n <= 64/P; a
// generic pointer, global or shared) of one sequence whose complete groups are
// [0, G).  Invalid or missing groups are zero-filled and marked -1 in sg.
template <int DQK, int DV>
__device__ __forceinline__ void gather_chunk(uint16_t *dk, uint16_t *dv, int *sg,
                                             const int32_t *glist, int n, int P, int G,
                                             const uint16_t *kb, const uint16_t *vb, int QP,
                                             int VP, int tid, int nthreads) {
    const int gpc = kChunk / P;
    if (tid < gpc) {
        const int g = tid < n ? glist[tid] : -1;
        sg[tid] = (g >= 0 && g < G) ? g : -1;
    }
    for (int p = tid; p < kChunk * (DQK / 8); p += nthreads) {
        const int tr = p / (DQK / 8), c8 = p % (DQK / 8);
        const int q = tr / P;
        const int g = q < n ? glist[q] : -1;
        const bool ok = g >= 0 && g < G;
        const uint16_t *src = ok ? kb + (int64_t(g) * P + tr % P) * DQK + c8 * 8 : kb;
        cp_async16(smem_u32(dk + tr * QP + c8 * 8), src, ok ? 16 : 0);
    }
    for (int p = tid; p < kChunk * (DV / 8); p += nthreads) {
        const int tr = p / (DV / 8), c8 = p % (DV / 8);
        const int q = tr / P;
        const int g = q < n ? glist[q] : -1;
        const bool ok = g >= 0 && g < G;
        const uint16_t *src = ok ? vb + (int64_t(g) * P + tr % P) * DV + c8 * 8 : vb;
        cp_async16(smem_u32(dv + tr * VP + c8 * 8), src, ok ? 16 : 0);
    }
    cp_async_commit();
}

// Merge the TS warp states of each 16-head tile held in `state`
// ([warps][16][DV + 2], warp = ts * MT + tile) for head hl (0-based within the
// block's head group) and dims d2, d2+1.  Returns (M, L, o_a, o_b).
template <int DV>
__device__ __forceinline__ float4 merge_states(const float *state, int MT, int TS, int hl,
                                               int d2, float &Lsum) {
    const int tile = hl / 16, rr = hl % 16;
    float M = -INFINITY;
    for (int t2 = 0; t2 < TS; ++t2)
        M = fmaxf(M, state[((t2 * MT + tile) * 16 + rr) * (DV + 2) + DV]);
    const float ref = M == -INFINITY ? 0.f : M;
    float L = 0.f, oa = 0.f, ob = 0.f;
    for (int t2 = 0; t2 < TS; ++t2) {
        const float *stt = state + ((t2 * MT + tile) * 16 + rr) * (DV + 2);
        const float f = exp2f(stt[DV] - ref);
        L += f * stt[DV + 1];
        oa += f * stt[d2];
        ob += f * stt[d2 + 1];
    }
    Lsum = L;
    return make_float4(M, L, oa, ob);
}

// Write the warp's (m, l, O) rows to shared `state` [16][DV + 2] (after the
// quad reduction of l).
template <int DV>
__device__ __forceinline__ void store_warp_state(AttnWarpState<DV> &st, float *state) {
    const int lane = threadIdx.x & 31, c = lane & 3, r0 = lane >> 2;
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 1);
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 2);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 1);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 2);
#pragma unroll
    for (int i = 0; i < DV / 8; ++i) {
        state[r0 * (DV + 2) + i * 8 + 2 * c] = st.o[i][0];
        state[r0 * (DV + 2) + i * 8 + 2 * c + 1] = st.o[i][1];
        state[(r0 + 8) * (DV + 2) + i * 8 + 2 * c] = st.o[i][2];
        state[(r0 + 8) * (DV + 2) + i * 8 + 2 * c + 1] = st.o[i][3];
    }
    if (c == 0) {
        state[r0 * (DV + 2) + DV] = st.m0;
        state[r0 * (DV + 2) + DV + 1] = st.l0;
        state[(r0 + 8) * (DV + 2) + DV] = st.m1;
        state[(r0 + 8) * (DV + 2) + DV + 1] = st.l1;
    }
}

// Merge of split-K partial states (part_o [rows][S][H_q][DV] unnormalised,
// part_ml [rows][S][H_q] = (m in log2 units, l)): one warp per (row, head),
// grid (rows, ceil(H_q / 8)) of 256 threads.
namespace {
constexpr float kCombLn2 = 0.6931471805599453f;
template <int DV>
__global__ void __launch_bounds__(256) splitk_combine_kernel(
    const float *__restrict__ part_o, const float2 *__restrict__ part_ml, int H_q, int S,
    uint16_t *__restrict__ out, float *__restrict__ lse) {
    const int64_t row = blockIdx.x;
    const int h = blockIdx.y * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (h >= H_q) return;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldg(&part_ml[(row * S + s) * H_q + h].x));
    const float ref = M == -INFINITY ? 0.f : M;
    constexpr int PER = DV / 32;  // 2 or 4 value dims per lane
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float Lsum = 0.f;
    // eight splits at a time, their loads issued together
    for (int s0 = 0; s0 < S; s0 += 8) {
        float v[8][PER];
        float f[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            f[u] = 0.f;
#pragma unroll
            for (int i = 0; i < PER; ++i) v[u][i] = 0.f;
            if (s0 + u < S) {
                const int64_t pi = (row * S + s0 + u) * H_q + h;
                const float2 ml = __ldg(&part_ml[pi]);
                f[u] = exp2f(ml.x - ref);
                Lsum += f[u] * ml.y;
                const float *po = part_o + pi * DV + lane * PER;
#pragma unroll
                for (int i = 0; i < PER; ++i) v[u][i] = __ldg(po + i);
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int i = 0; i < PER; ++i) acc[i] += f[u] * v[u][i];
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    uint16_t *orow = out + (row * H_q + h) * DV + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; i += 2)
        *reinterpret_cast<uint32_t *>(orow + i) = pack_bf2(acc[i] * inv, acc[i + 1] * inv);
    if (lse && lane == 0) lse[row * H_q + h] = Lsum > 0.f ? (M + log2f(Lsum)) * kCombLn2 : -INFINITY;
}

}  // namespace

}  // namespace lcsw
