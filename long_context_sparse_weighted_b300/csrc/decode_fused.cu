// Persistent fused decode step: the host side (supported shapes, workspace,
// launch) of the kernel in decode_fused_kernel.cuh, bf16 pooled keys.
#include "decode_fused_kernel.cuh"

namespace lcsw {

bool fused_decode_supported(int B, int G_max, int H_i, int H_q, int d_qk, int d_v, int k, int P) {
    const int ncta = num_sms();
    if (ncta > kMaxCtas || B < 1 || 2 * B > ncta) return false;
    if (H_i > 16 || k > kMaxK || k < 1) return false;
    if (!((d_qk == 64 || d_qk == 128 || d_qk == 192) && (d_v == 64 || d_v == 128))) return false;
    if (!(H_q % 16 == 0 && H_q <= 64)) return false;  // one M = 128 tensor-core tile of heads
    // 16-bit shared counters: a block's chunk must stay below 65536 groups.
    // Blocks go to sequences by cost w_b = 2 G_b + min(k, G_b) P (d_qk + d_v) / 16
    // (64-byte units) >= 2 G_b, so a chunk holds at most sum_b w_b / (2 (ncta - B))
    // groups, plus tile rounding.
    const long long w_max = 2LL * G_max + (long long)k * P * ((d_qk + d_v) / 16);
    const long long bound =
        B == 1 ? (long long)G_max / ncta + 32 : (long long)B * w_max / (2LL * (ncta - B)) + 32;
    if (bound >= 65535) return false;
    return true;
}

size_t fused_decode_ws_bytes(int B, int G_max, int H_q, int d_v, int k, int P) {
    if (!fused_decode_supported(B, G_max, 1, H_q, 128, d_v, k, P)) return 0;
    return ws_layout(B, G_max, H_q, d_v, k, num_sms()).total;
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
    return launch_shape<false>(make_params(a, ws, status), a, st);
}

cudaError_t launch_fused_select(const lcsw_decode_args *a, int32_t *idx_out, void *ws,
                                int *status, cudaStream_t st) {
    // the selection alone: the 128-wide attention instance, whose attention
    // and merge phases are skipped (q, K, V are not read)
    lcsw_decode_args s = *a;
    s.d_qk = 128;
    s.d_v = 128;
    s.idx_out = idx_out;
    Params prm = make_params(&s, ws, status);
    prm.select_only = 1;
    return launch_shape<false>(prm, &s, st);
}

bool reuse_decode_supported(int B, int H_q, int d_qk, int d_v, int k) {
    const int ncta = num_sms();
    if (ncta > kMaxCtas || B < 1 || 2 * B > ncta || k < 1 || k > kMaxK) return false;
    if (!((d_qk == 64 || d_qk == 128 || d_qk == 192) && (d_v == 64 || d_v == 128))) return false;
    return H_q % 16 == 0 && H_q <= 64;
}

cudaError_t launch_reuse_decode(const lcsw_decode_args *a, const int32_t *idx_in, void *ws,
                                int *status, cudaStream_t st) {
    Params prm = make_params(a, ws, status);
    prm.idx_in = idx_in;
    return launch_reuse_shape(prm, a, st);
}

}  // namespace lcsw
