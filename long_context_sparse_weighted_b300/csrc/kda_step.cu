// KDA step: the linear-attention half of the hybrid ("G2C Brief --
// GLM-5.3-Flash", section "KDA carries fixed state through most layers": a
// gated delta-rule descendant of linear attention with a fixed matrix state
// per head, a short convolution of kernel size 4 and learned gates; 64 heads
// of width 128, so 64 x 128 x 128 state values per layer).
//
// Per sequence b, head h and token t (S: D x D fp32, key channels as rows):
//   window = inputs of tokens t-3 .. t (the conv history supplies t < 0)
//   a_c    = SiLU(sum_j w[c][j] * window[j][c])      for the head's q, k, v channels
//   q = a_q / sqrt(|a_q|^2 + 1e-6) / sqrt(D),  k = a_k / sqrt(|a_k|^2 + 1e-6),  v = a_v
//   S'     = Diag(exp(g_t)) S
//   S      = S' + k (beta_t (v - S'^T k))^T          (= (I - beta k k^T) S' + beta k v^T)
//   o_t    = S^T q = S'^T q + (q . k) beta_t (v - S'^T k)
//
// One block per (head, sequence), 256 threads.  The 64 KB state is the only
// large operand: it is read once into registers at the start (16 float4 per
// thread: lane l holds columns 4l..4l+3, warp w rows 16w..16w+15), stays there
// for every token of the call, and is written back once at the end, so a
// decode step moves 128 KB per head and is bound by HBM bandwidth.  The
// per-token work (convolution of 384 channels, two norms, the two column
// reductions over the 128 key channels) runs while the state loads are in
// flight for the first token.
#include "common.cuh"
#include "kernels.cuh"

namespace lcsw {
namespace {

constexpr int kD = 128;           // head width (key and value)
constexpr int kThreads = 256;     // 8 warps
constexpr int kRows = kD / 8;     // key-channel rows per warp
constexpr float kL2Eps = 1e-6f;

__device__ __forceinline__ float silu(float y) { return y / (1.0f + expf(-y)); }

__device__ __forceinline__ float4 ld_state(const float *p) {
    float4 v;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_state(float *p, float4 v) {
    asm volatile("st.global.L1::no_allocate.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// Input of channel gc at token position p of sequence b: the token's own
// projection for p >= 0, the conv history (oldest first) for p in [-3, 0).
__device__ __forceinline__ float conv_input(const uint16_t *qkv_b, const uint16_t *hist_b,
                                            int64_t C, int p, int64_t gc) {
    return p >= 0 ? bf2f(qkv_b[int64_t(p) * C + gc]) : bf2f(hist_b[int64_t(3 + p) * C + gc]);
}

__global__ void __launch_bounds__(kThreads, 2)
    kda_step_kernel(const uint16_t *__restrict__ qkv, const uint16_t *__restrict__ conv_w,
                    uint16_t *__restrict__ conv_state, const float *__restrict__ g,
                    const float *__restrict__ beta, float *__restrict__ state,
                    uint16_t *__restrict__ out, int T, int H) {
    const int h = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t HD = int64_t(H) * kD, C = 3 * HD;

    __shared__ __align__(16) float act[3 * kD];        // q (normalised, scaled), k (normalised), v
    __shared__ float alpha[kD];          // exp(g) per key channel
    __shared__ __align__(16) float red[8][2][kD];      // per-warp partial column sums: S'^T k, S'^T q
    __shared__ float nrm[4];             // 1/|q|, 1/|k|, q.k (raw), beta

    // the state, issued first so that its latency hides behind the token prologue
    float *S_g = state + (int64_t(b) * H + h) * kD * kD;
    float4 S[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) S[r] = ld_state(S_g + (warp * kRows + r) * kD + lane * 4);

    const uint16_t *qkv_b = qkv + int64_t(b) * T * C;
    uint16_t *hist_b = conv_state + int64_t(b) * 3 * C;
    const float scale = rsqrtf(float(kD));

    for (int t = 0; t < T; ++t) {
        // -- short convolution + SiLU over the head's 384 channels ----------
        for (int c = tid; c < 3 * kD; c += kThreads) {
            const int part = c / kD, i = c % kD;
            const int64_t gc = part * HD + int64_t(h) * kD + i;
            const uint2 wv = *reinterpret_cast<const uint2 *>(conv_w + gc * 4);
            const float w0 = bf_lo(wv.x), w1 = bf_hi(wv.x), w2 = bf_lo(wv.y), w3 = bf_hi(wv.y);
            float y = w0 * conv_input(qkv_b, hist_b, C, t - 3, gc);
            y = fmaf(w1, conv_input(qkv_b, hist_b, C, t - 2, gc), y);
            y = fmaf(w2, conv_input(qkv_b, hist_b, C, t - 1, gc), y);
            y = fmaf(w3, conv_input(qkv_b, hist_b, C, t, gc), y);
            act[c] = silu(y);
        }
        if (tid < kD) alpha[tid] = expf(g[((int64_t(b) * T + t) * H + h) * kD + tid]);
        __syncthreads();
        // -- norms of q and k, and q.k, one warp each ------------------------
        if (warp < 3) {
            const float *x = act + (warp == 1 ? kD : 0);
            const float *y = act + (warp == 0 ? 0 : kD);
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < kD / 32; ++j) s = fmaf(x[lane + 32 * j], y[lane + 32 * j], s);
#pragma unroll
            for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) nrm[warp] = warp < 2 ? rsqrtf(s + kL2Eps) : s;
        } else if (tid == 96) {
            nrm[3] = beta[(int64_t(b) * T + t) * H + h];
        }
        __syncthreads();
        const float rq = nrm[0] * scale, rk = nrm[1];
        const float qk = nrm[2] * rq * rk, bt = nrm[3];
        // -- decay, then the two column reductions over the warp's rows -----
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f), p = u;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int i = warp * kRows + r;
            const float a = alpha[i], kk = act[kD + i] * rk, qq = act[i] * rq;
            S[r].x *= a; S[r].y *= a; S[r].z *= a; S[r].w *= a;
            u.x = fmaf(kk, S[r].x, u.x); u.y = fmaf(kk, S[r].y, u.y);
            u.z = fmaf(kk, S[r].z, u.z); u.w = fmaf(kk, S[r].w, u.w);
            p.x = fmaf(qq, S[r].x, p.x); p.y = fmaf(qq, S[r].y, p.y);
            p.z = fmaf(qq, S[r].z, p.z); p.w = fmaf(qq, S[r].w, p.w);
        }
        *reinterpret_cast<float4 *>(&red[warp][0][lane * 4]) = u;
        *reinterpret_cast<float4 *>(&red[warp][1][lane * 4]) = p;
        __syncthreads();
        u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float4 x = *reinterpret_cast<const float4 *>(&red[w][0][lane * 4]);
            u.x += x.x; u.y += x.y; u.z += x.z; u.w += x.w;
        }
        // -- delta-rule write: S += k (beta (v - S'^T k))^T ------------------
        const float4 vv = *reinterpret_cast<const float4 *>(&act[2 * kD + lane * 4]);
        const float4 dw = make_float4(bt * (vv.x - u.x), bt * (vv.y - u.y), bt * (vv.z - u.z),
                                      bt * (vv.w - u.w));
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float kk = act[kD + warp * kRows + r] * rk;
            S[r].x = fmaf(kk, dw.x, S[r].x); S[r].y = fmaf(kk, dw.y, S[r].y);
            S[r].z = fmaf(kk, dw.z, S[r].z); S[r].w = fmaf(kk, dw.w, S[r].w);
        }
        // -- read-out o = S'^T q + (q.k) beta (v - S'^T k), by warp 0 --------
        if (warp == 0) {
            p = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const float4 x = *reinterpret_cast<const float4 *>(&red[w][1][lane * 4]);
                p.x += x.x; p.y += x.y; p.z += x.z; p.w += x.w;
            }
            const uint2 o2 = make_uint2(pack_bf2(fmaf(qk, dw.x, p.x), fmaf(qk, dw.y, p.y)),
                                        pack_bf2(fmaf(qk, dw.z, p.z), fmaf(qk, dw.w, p.w)));
            *reinterpret_cast<uint2 *>(out + ((int64_t(b) * T + t) * H + h) * kD + lane * 4) = o2;
        }
        __syncthreads();  // act, alpha, red and nrm are rewritten by the next token
    }

#pragma unroll
    for (int r = 0; r < kRows; ++r) st_state(S_g + (warp * kRows + r) * kD + lane * 4, S[r]);

    // -- conv history: the raw inputs of the last three positions ----------
    for (int c = tid; c < 3 * kD; c += kThreads) {
        const int part = c / kD, i = c % kD;
        const int64_t gc = part * HD + int64_t(h) * kD + i;
        uint16_t x[3];
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int p = T - 3 + j;
            x[j] = p >= 0 ? qkv_b[int64_t(p) * C + gc] : hist_b[int64_t(3 + p) * C + gc];
        }
#pragma unroll
        for (int j = 0; j < 3; ++j) hist_b[int64_t(j) * C + gc] = x[j];
    }
}

}  // namespace

cudaError_t launch_kda_step(const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                            const float *g, const float *beta, float *state, uint16_t *out,
                            int B, int T, int H, cudaStream_t st) {
    if (B == 0 || T == 0) return cudaSuccess;
    kda_step_kernel<<<dim3(unsigned(H), unsigned(B)), kThreads, 0, st>>>(qkv, conv_w, conv_state,
                                                                        g, beta, state, out, T, H);
    return cudaGetLastError();
}

}  // namespace lcsw
