// C ABI of liblcsw.so (declared in include/lcsw.h): argument validation,
// workspace carving and kernel sequencing.  No entry point allocates device
// memory, synchronises the host (lcsw_get_status excepted) or lets a C++
// exception escape.
#include <nvtx3/nvToolsExt.h>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/lcsw.h"
#include "fused.cuh"
#include "kernels.cuh"

// NVTX ranges around the C entry points (header-only NVTX 3: free when no
// profiler is attached), so a timeline shows which library call issued which
// kernels.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define LCSW_RANGE(name) NvtxRange lcsw_nvtx_range_(name)

// Readers of the per-translation-unit check words of a -DLCSW_CHECKS=1 build
// (registered by static initialisers in common.cuh; none in a normal build).
namespace lcsw {
static std::vector<int (*)()> &check_readers() {
    static std::vector<int (*)()> readers;
    return readers;
}
void register_check_reader(int (*reader)()) { check_readers().push_back(reader); }
}  // namespace lcsw

namespace {

thread_local char g_err[512] = "";

lcsw_status fail(lcsw_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

lcsw_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return LCSW_OK;
    return fail(LCSW_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool p_ok(int P) { return P == 1 || P == 2 || P == 4 || P == 8; }

#define CHECK(cond, ...)                                   \
    do {                                                   \
        if (!(cond)) return fail(LCSW_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

// bf16 tensor with rows of `row_elems` and batch stride `sb` elements: base and
// every row must be 16-byte aligned.
bool bf16_rows_ok(const void *p, int64_t row_elems, int64_t sb) {
    return aligned(p, 16) && (row_elems * 2) % 16 == 0 && (sb * 2) % 16 == 0;
}

// Workspace layout shared by decode and prefill:
//   [0, 256)            status word (int) + reserved
//   then 256-byte aligned regions, in order of request.
struct Carver {
    char *base;
    size_t off = 256;
    explicit Carver(void *b) : base(static_cast<char *>(b)) {}
    void *take(size_t bytes) {
        void *p = base ? base + off : nullptr;
        off += (bytes + 255) & ~size_t(255);
        return p;
    }
};

// The MLA latent geometry: 576-wide rows (latent 512 + rotary 64), the latent
// as the value (out rows of 512).
bool mla_shape(int d_qk, int d_v) { return d_qk == LCSW_MLA_DQK && d_v == LCSW_MLA_DV; }

bool attn_shape_ok(int H_q, int d_qk, int d_v) {
    const bool heads = H_q > 0 && H_q % 16 == 0 && (H_q <= 32 || H_q % 64 == 0);
    const bool dims = (d_qk == 64 || d_qk == 128 || d_qk == 192) && (d_v == 64 || d_v == 128);
    return heads && dims;
}

}  // namespace

// ------------------------------------------------ fixed split-K scratch ----
// Device memory of lcsw_sparse_attn_noalloc: the split-K partial states live
// in this file-scope array (one instance per device, created with the
// library's module), so that entry point needs no workspace and allocates
// nothing.  Nothing in it has to start at zero: each call writes every partial
// state it reads.  Calls that overlap in time on one device share it and race.
static __device__ __align__(256) unsigned char g_attn_scratch[LCSW_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Set-up, once per device, with that device current: look up the array's
// device address.  Runs inside the first lcsw_sparse_attn_noalloc call on the
// device.
lcsw_status attn_scratch(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(LCSW_ERR_UNSUPPORTED, "device ordinal %d above the %d the fixed scratch covers",
                    dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return cuda_status(e, "cudaGetSymbolAddress(split-K scratch)");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return LCSW_OK;
}

}  // namespace

extern "C" {

const char *lcsw_last_error(void) { return g_err; }

const char *lcsw_version(void) { return "lcsw 0.1 (sm_103a)"; }

lcsw_status lcsw_pool_keys(const lcsw_bf16 *k_idx, int64_t sk_b, const float *pool_w,
                           int64_t sw_b, const int32_t *seq_len, const int32_t *g_begin, int B,
                           int g_span, int d_idx, int P, lcsw_bf16 *k_pooled, int64_t sp_b,
                           lcsw_stream stream) {
    LCSW_RANGE("lcsw_pool_keys");
    CHECK(B >= 0 && g_span >= 0, "B and g_span must be >= 0");
    CHECK(p_ok(P), "P must be 1, 2, 4 or 8 (got %d)", P);
    CHECK(d_idx > 0 && d_idx % 8 == 0, "d_idx must be a positive multiple of 8");
    if (B == 0 || g_span == 0) return LCSW_OK;
    CHECK(k_idx && pool_w && seq_len && k_pooled, "null pointer argument");
    CHECK(bf16_rows_ok(k_idx, d_idx, sk_b) && bf16_rows_ok(k_pooled, d_idx, sp_b),
          "k_idx/k_pooled rows must be 16-byte aligned");
    CHECK(aligned(pool_w, 4) && aligned(seq_len, 4) && (!g_begin || aligned(g_begin, 4)),
          "fp32/int32 arrays must be 4-byte aligned");
    CHECK(sk_b >= 0 && sw_b >= 0 && sp_b >= 0, "strides must be >= 0");
    return cuda_status(lcsw::launch_pool_keys(k_idx, sk_b, pool_w, sw_b, seq_len, g_begin, B,
                                              g_span, d_idx, P, 0, 0, k_pooled, sp_b,
                                              (cudaStream_t)stream),
                       "pool_keys launch");
}

lcsw_status lcsw_visible_counts(const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                int P, int32_t *n_valid, lcsw_stream stream) {
    LCSW_RANGE("lcsw_visible_counts");
    CHECK(B >= 0 && T >= 0 && p_ok(P), "bad B/T/P");
    if (int64_t(B) * T == 0) return LCSW_OK;
    CHECK(seq_len && n_valid, "null pointer argument");
    return cuda_status(lcsw::launch_visible_counts(seq_len, q_pos, B, T, P, n_valid,
                                                   (cudaStream_t)stream),
                       "visible_counts launch");
}

lcsw_status lcsw_index_scores(const lcsw_bf16 *q_idx, const float *w_head,
                              const lcsw_bf16 *k_pooled, int64_t sp_b, const int32_t *seq_len,
                              const int32_t *q_pos, int B, int T, int H_i, int d_idx, int P,
                              int G_max, float *scores, lcsw_stream stream) {
    LCSW_RANGE("lcsw_index_scores");
    CHECK(B >= 0 && T >= 0 && G_max >= 0, "negative dimension");
    CHECK(d_idx == 64, "d_idx must be 64 (got %d)", d_idx);
    CHECK(H_i >= 1 && H_i <= 16, "H_i must be in [1, 16] (got %d)", H_i);
    CHECK(p_ok(P), "P must be 1, 2, 4 or 8");
    if (int64_t(B) * T * G_max == 0) return LCSW_OK;
    CHECK(q_idx && w_head && k_pooled && seq_len && scores, "null pointer argument");
    CHECK(bf16_rows_ok(q_idx, d_idx, 0) && bf16_rows_ok(k_pooled, d_idx, sp_b),
          "q_idx/k_pooled rows must be 16-byte aligned");
    CHECK(aligned(w_head, 4) && aligned(scores, 4) && aligned(seq_len, 4), "misaligned array");
    cudaStream_t st = (cudaStream_t)stream;
    if (T > 1 && lcsw::index_scores_tc_supported(B, T, H_i, G_max, sp_b)) {
        return cuda_status(lcsw::launch_index_scores_tc(q_idx, w_head, k_pooled, sp_b, seq_len,
                                                        q_pos, B, T, H_i, P, G_max, scores,
                                                        nullptr, st),
                           "index_scores (tcgen05) launch");
    }
    CHECK(int64_t(B) * ((T + 3) / 4) <= 65535, "B * ceil(T/4) must be <= 65535");
    return cuda_status(lcsw::launch_index_scores_mma(q_idx, w_head, k_pooled, sp_b, seq_len,
                                                     q_pos, B, T, H_i, P, G_max, scores, st),
                       "index_scores launch");
}

size_t lcsw_topk_workspace_size(int64_t rows, int G_max, int k) {
    if (rows <= 0 || G_max <= 0 || k < 1) return 0;
    return lcsw::topk_wide_ws_bytes(rows, G_max, k);
}

lcsw_status lcsw_topk_groups(const float *scores, const int32_t *n_valid, int64_t rows,
                             int G_max, int k, int32_t *idx, void *ws, size_t ws_bytes,
                             lcsw_stream stream) {
    LCSW_RANGE("lcsw_topk_groups");
    CHECK(rows >= 0 && G_max >= 0, "negative dimension");
    CHECK(k >= 1, "k must be >= 1 (got %d)", k);
    CHECK(rows <= 0x7FFFFFFF, "too many rows");
    if (rows == 0) return LCSW_OK;
    CHECK(scores && n_valid && idx, "null pointer argument");
    CHECK(aligned(scores, 4) && aligned(n_valid, 4) && aligned(idx, 4), "misaligned array");
    const size_t wide = lcsw::topk_wide_ws_bytes(rows, G_max, k);
    if (wide && ws && ws_bytes >= wide && aligned(ws, 256))
        return cuda_status(lcsw::launch_topk_rows_wide(scores, n_valid, nullptr, 1, 1, rows,
                                                       G_max, k, idx, ws, (cudaStream_t)stream),
                           "topk launch (wide rows)");
    return cuda_status(lcsw::launch_topk_rows(scores, n_valid, nullptr, 1, 1, rows, G_max, k,
                                              idx, (cudaStream_t)stream),
                       "topk launch");
}

size_t lcsw_sparse_attn_workspace_size(int B, int T, int H_q, int d_v, int k, int P) {
    if (B <= 0 || T <= 0 || H_q <= 0 || d_v <= 0 || k <= 0 || !p_ok(P)) return 0;
    return lcsw::sparse_attn_ws_bytes(int64_t(B) * T, H_q, d_v, k, P);
}

}  // extern "C"

namespace {

// Argument checks of the sparse attention entry points (shapes, pointers,
// alignment), before any workspace or scratch question.
lcsw_status check_attn(const lcsw_bf16 *q, const lcsw_bf16 *K, int64_t sK_b, const lcsw_bf16 *V,
                       int64_t sV_b, const int32_t *seq_len, const int32_t *idx, int B, int T,
                       int H_q, int d_qk, int d_v, int P, int k, const lcsw_bf16 *out,
                       const float *lse) {
    CHECK(B >= 0 && T >= 0, "negative dimension");
    CHECK(k >= 1, "k must be >= 1");
    CHECK(p_ok(P), "P must be 1, 2, 4 or 8");
    CHECK(attn_shape_ok(H_q, d_qk, d_v),
          "unsupported attention shape H_q=%d d_qk=%d d_v=%d (H_q in {16,32} or a multiple of "
          "64; d_qk in {64,128,192}; d_v in {64,128})", H_q, d_qk, d_v);
    const int64_t rows = int64_t(B) * T;
    if (rows == 0) return LCSW_OK;
    CHECK(rows <= 65535, "B*T must be <= 65535");
    CHECK(q && K && V && seq_len && idx && out, "null pointer argument");
    CHECK(bf16_rows_ok(q, d_qk, 0) && bf16_rows_ok(K, d_qk, sK_b) && bf16_rows_ok(V, d_v, sV_b) &&
              bf16_rows_ok(out, d_v, 0),
          "q/K/V/out rows must be 16-byte aligned");
    CHECK(aligned(idx, 4) && aligned(seq_len, 4) && (!lse || aligned(lse, 4)), "misaligned array");
    return LCSW_OK;
}

}  // namespace

extern "C" {

lcsw_status lcsw_sparse_attn(const lcsw_bf16 *q, const lcsw_bf16 *K, int64_t sK_b,
                             const lcsw_bf16 *V, int64_t sV_b, const int32_t *seq_len,
                             const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v,
                             int P, int k, float scale, lcsw_bf16 *out, float *lse, void *ws,
                             size_t ws_bytes, lcsw_stream stream) {
    LCSW_RANGE("lcsw_sparse_attn");
    const lcsw_status chk = check_attn(q, K, sK_b, V, sV_b, seq_len, idx, B, T, H_q, d_qk, d_v,
                                       P, k, out, lse);
    if (chk != LCSW_OK) return chk;
    const int64_t rows = int64_t(B) * T;
    if (rows == 0) return LCSW_OK;
    const size_t need = lcsw::sparse_attn_ws_bytes(rows, H_q, d_v, k, P);
    if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16)))
        return fail(LCSW_ERR_WORKSPACE, "sparse_attn needs a 16-byte aligned workspace of %zu bytes",
                    need);
    return cuda_status(lcsw::launch_sparse_attn(q, K, sK_b, V, sV_b, seq_len, idx, B, T, H_q,
                                                d_qk, d_v, P, k, scale, out, lse, ws,
                                                (cudaStream_t)stream),
                       "sparse_attn launch");
}

// ------------------------------------------------------------------ decode --

static lcsw_status check_decode(const lcsw_decode_args *a) {
    CHECK(a, "null args");
    CHECK(a->B >= 0 && a->G_max >= 0, "negative dimension");
    CHECK(a->d_idx == 64, "d_idx must be 64");
    CHECK(a->H_i >= 1 && a->H_i <= 16, "H_i must be in [1, 16]");
    CHECK(p_ok(a->P), "P must be 1, 2, 4 or 8");
    CHECK(a->k >= 1, "k must be >= 1");
    const bool mla = mla_shape(a->d_qk, a->d_v);
    CHECK(mla ? (a->H_q > 0 && a->H_q % 16 == 0) : attn_shape_ok(a->H_q, a->d_qk, a->d_v),
          "unsupported attention shape");
    CHECK(!mla || !a->V || (a->V == a->K && a->sV_b == a->sK_b),
          "MLA geometry: V is the latent part of K (pass NULL or K itself)");
    if (a->B == 0) return LCSW_OK;
    CHECK(a->B <= 65535, "B must be <= 65535");
    CHECK(a->q_idx && a->w_head && a->k_pooled && a->q && a->K && (a->V || mla) && a->seq_len &&
              a->out,
          "null pointer argument");
    CHECK(!a->k_idx || a->pool_w, "pool_w is required with k_idx");
    CHECK(bf16_rows_ok(a->q_idx, 64, 0) && bf16_rows_ok(a->k_pooled, 64, a->sp_b) &&
              (!a->k_idx || bf16_rows_ok(a->k_idx, 64, a->sk_b)) &&
              bf16_rows_ok(a->q, a->d_qk, 0) && bf16_rows_ok(a->K, a->d_qk, a->sK_b) &&
              (mla || bf16_rows_ok(a->V, a->d_v, a->sV_b)) && bf16_rows_ok(a->out, a->d_v, 0),
          "bf16 rows must be 16-byte aligned");
    CHECK(aligned(a->w_head, 4) && aligned(a->seq_len, 4) && (!a->lse || aligned(a->lse, 4)) &&
              (!a->idx_out || aligned(a->idx_out, 4)) &&
              (!a->scores_out || aligned(a->scores_out, 4)) &&
              (!a->pool_w || aligned(a->pool_w, 4)),
          "misaligned fp32/int32 array");
    return LCSW_OK;
}

struct DecodeWs {
    int *status;
    float *scores;
    int32_t *idx;
    void *attn;
    void *fused;
    void *topk;          // the few-long-rows selection's region (or none)
    size_t topk_bytes;
    size_t total;
};

static DecodeWs carve_decode(const lcsw_decode_args *a, void *ws) {
    Carver c(ws);
    DecodeWs w;
    w.status = static_cast<int *>(ws);
    // the persistent kernels' region first: its partial-state words sit at the
    // same offsets for every call that shares the workspace
    // (the MLA geometry runs the persistent kernel for its selection only, at d_v 128)
    const int dv_fused = mla_shape(a->d_qk, a->d_v) ? 128 : a->d_v;
    w.fused = c.take(lcsw::fused_decode_ws_bytes(a->B, a->G_max, a->H_q, dv_fused, a->k, a->P));
    w.scores = static_cast<float *>(c.take(size_t(a->B) * a->G_max * sizeof(float)));
    w.idx = static_cast<int32_t *>(c.take(size_t(a->B) * a->k * sizeof(int32_t)));
    w.attn = c.take(mla_shape(a->d_qk, a->d_v)
                        ? lcsw::sparse_attn_mla_ws_bytes(a->B, a->H_q, a->k, a->P)
                        : lcsw::sparse_attn_ws_bytes(a->B, a->H_q, a->d_v, a->k, a->P));
    w.topk_bytes = lcsw::topk_wide_ws_bytes(a->B, a->G_max, a->k);
    w.topk = c.take(w.topk_bytes);
    w.total = c.off;
    return w;
}

// Attention of one decode query per sequence over idx [B][k] (split-K
// launches), in the shape's geometry.
static cudaError_t decode_attend(const lcsw_decode_args *a, const int32_t *idx, void *attn_ws,
                                 cudaStream_t st, bool after_selection = false) {
    if (mla_shape(a->d_qk, a->d_v))
        return lcsw::launch_sparse_attn_mla(a->q, a->K, a->sK_b, a->seq_len, idx, a->B, 1, a->H_q,
                                            a->P, a->k, a->scale, a->out, a->lse, attn_ws, st,
                                            after_selection);
    return lcsw::launch_sparse_attn(a->q, a->K, a->sK_b, a->V, a->sV_b, a->seq_len, idx, a->B, 1,
                                    a->H_q, a->d_qk, a->d_v, a->P, a->k, a->scale, a->out, a->lse,
                                    attn_ws, st);
}

size_t lcsw_decode_workspace_size(const lcsw_decode_args *a) {
    if (!a || a->B <= 0 || a->G_max < 0 || a->k < 1 || !p_ok(a->P)) return 256;
    return carve_decode(a, nullptr).total;
}

int lcsw_decode_launches(const lcsw_decode_args *a) {
    if (check_decode(a) != LCSW_OK) return 0;
    if (a->B == 0) return 0;
    if (!(a->flags & LCSW_DECODE_FORCE_MULTIKERNEL) &&
        lcsw::fused_decode_supported(a->B, a->G_max, a->H_i, a->H_q, a->d_qk, a->d_v, a->k, a->P))
        return 1;
    if (!(a->flags & LCSW_DECODE_FORCE_MULTIKERNEL) && mla_shape(a->d_qk, a->d_v) &&
        lcsw::fused_decode_supported(a->B, a->G_max, a->H_i, a->H_q, 128, 128, a->k, a->P))
        return 1 + (lcsw::sparse_attn_mla_splits(a->B, a->H_q, a->k, a->P) > 1 ? 2 : 1);
    const int S = mla_shape(a->d_qk, a->d_v) ? lcsw::sparse_attn_mla_splits(a->B, a->H_q, a->k, a->P)
                                              : lcsw::sparse_attn_splits(a->B, a->H_q, a->k, a->P);
    // append, scores, top-k (three kernels for a few long rows), attention (+ merge)
    const int topk = lcsw::topk_wide_ws_bytes(a->B, a->G_max, a->k) ? 3 : 1;
    return (a->k_idx ? 1 : 0) + 1 + topk + 1 + (S > 1 ? 1 : 0);
}

lcsw_status lcsw_decode_fused(const lcsw_decode_args *a, void *ws, size_t ws_bytes,
                              lcsw_stream stream) {
    LCSW_RANGE("lcsw_decode_fused");
    lcsw_status s = check_decode(a);
    if (s != LCSW_OK || a->B == 0) return s;
    const size_t need = lcsw_decode_workspace_size(a);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return fail(LCSW_ERR_WORKSPACE, "decode needs a 256-byte aligned workspace of %zu bytes",
                    need);
    cudaStream_t st = (cudaStream_t)stream;
    DecodeWs w = carve_decode(a, ws);
    float *scores = a->scores_out ? a->scores_out : w.scores;
    int32_t *idx = a->idx_out ? a->idx_out : w.idx;

    if (!(a->flags & LCSW_DECODE_FORCE_MULTIKERNEL) &&
        lcsw::fused_decode_supported(a->B, a->G_max, a->H_i, a->H_q, a->d_qk, a->d_v, a->k, a->P)) {
        return cuda_status(lcsw::launch_fused_decode(a, w.fused, w.status, st), "fused decode");
    }
    if (!(a->flags & LCSW_DECODE_FORCE_MULTIKERNEL) && mla_shape(a->d_qk, a->d_v) &&
        lcsw::fused_decode_supported(a->B, a->G_max, a->H_i, a->H_q, 128, 128, a->k, a->P)) {
        // MLA geometry: the persistent kernel selects, the latent attention follows
        cudaError_t e = lcsw::launch_fused_select(a, idx, w.fused, w.status, st);
        if (e != cudaSuccess) return cuda_status(e, "fused selection");
        return cuda_status(decode_attend(a, idx, w.attn, st, true), "decode attention");
    }
    // Multi-kernel path (same results): append, score, select, attend.
    if (a->k_idx) {
        cudaError_t e = lcsw::launch_pool_keys(a->k_idx, a->sk_b, a->pool_w, a->sw_b, a->seq_len,
                                               nullptr, a->B, 1, 64, a->P, 1, 0, a->k_pooled,
                                               a->sp_b, st);
        if (e != cudaSuccess) return cuda_status(e, "decode append");
    }
    cudaError_t e = lcsw::launch_index_scores_mma(a->q_idx, a->w_head, a->k_pooled, a->sp_b,
                                                  a->seq_len, nullptr, a->B, 1, a->H_i, a->P,
                                                  a->G_max, scores, st);
    if (e != cudaSuccess) return cuda_status(e, "decode scores");
    e = w.topk_bytes ? lcsw::launch_topk_rows_wide(scores, nullptr, a->seq_len, a->P, 1, a->B,
                                                   a->G_max, a->k, idx, w.topk, st)
                     : lcsw::launch_topk_rows(scores, nullptr, a->seq_len, a->P, 1, a->B,
                                              a->G_max, a->k, idx, st);
    if (e != cudaSuccess) return cuda_status(e, "decode top-k");
    return cuda_status(decode_attend(a, idx, w.attn, st), "decode attention");
}

lcsw_status lcsw_quantize_keys_e4m3(const lcsw_bf16 *k_pooled, int64_t sp_b, int B,
                                    int n_groups, uint8_t *kq, int64_t sq_b,
                                    lcsw_stream stream) {
    LCSW_RANGE("lcsw_quantize_keys_e4m3");
    CHECK(B >= 0 && n_groups >= 0, "negative dimension");
    if (B == 0 || n_groups == 0) return LCSW_OK;
    CHECK(k_pooled && kq, "null pointer argument");
    CHECK(bf16_rows_ok(k_pooled, 64, sp_b) && sp_b >= int64_t(n_groups) * 64,
          "k_pooled rows must be 16-byte aligned and hold n_groups rows per sequence");
    const int64_t tiles = (int64_t(n_groups) + 15) / 16;
    CHECK(aligned(kq, 16) && sq_b % 16 == 0 && sq_b >= tiles * LCSW_E4M3_TILE_BYTES,
          "kq must be 16-byte aligned with a batch stride (multiple of 16) of at least "
          "ceil(n_groups/16) tiles of %d bytes", LCSW_E4M3_TILE_BYTES);
    return cuda_status(lcsw::launch_quantize_keys_e4m3(k_pooled, sp_b, B, n_groups, kq, sq_b,
                                                       (cudaStream_t)stream),
                       "quantize keys launch");
}

lcsw_status lcsw_decode_fused_e4m3(const lcsw_decode_args *a, uint8_t *kq, int64_t sq_b,
                                   void *ws, size_t ws_bytes, lcsw_stream stream) {
    LCSW_RANGE("lcsw_decode_fused_e4m3");
    CHECK(a, "null args");
    CHECK(a->B >= 0 && a->G_max >= 0, "negative dimension");
    CHECK(a->d_idx == 64, "d_idx must be 64");
    CHECK(a->H_i >= 1 && a->H_i <= 16, "H_i must be in [1, 16]");
    CHECK(p_ok(a->P), "P must be 1, 2, 4 or 8");
    CHECK(a->k >= 1, "k must be >= 1");
    CHECK(attn_shape_ok(a->H_q, a->d_qk, a->d_v), "unsupported attention shape");
    if (a->B == 0) return LCSW_OK;
    CHECK(a->q_idx && a->w_head && kq && a->q && a->K && a->V && a->seq_len && a->out,
          "null pointer argument");
    CHECK(!a->k_idx || a->pool_w, "pool_w is required with k_idx");
    CHECK(bf16_rows_ok(a->q_idx, 64, 0) && (!a->k_idx || bf16_rows_ok(a->k_idx, 64, a->sk_b)) &&
              bf16_rows_ok(a->q, a->d_qk, 0) && bf16_rows_ok(a->K, a->d_qk, a->sK_b) &&
              bf16_rows_ok(a->V, a->d_v, a->sV_b) && bf16_rows_ok(a->out, a->d_v, 0),
          "bf16 rows must be 16-byte aligned");
    CHECK(aligned(a->w_head, 4) && aligned(a->seq_len, 4) && (!a->lse || aligned(a->lse, 4)) &&
              (!a->idx_out || aligned(a->idx_out, 4)) &&
              (!a->scores_out || aligned(a->scores_out, 4)) &&
              (!a->pool_w || aligned(a->pool_w, 4)),
          "misaligned fp32/int32 array");
    const int64_t tiles = (int64_t(a->G_max) + 15) / 16;
    CHECK(aligned(kq, 16) && sq_b % 16 == 0 && sq_b >= tiles * LCSW_E4M3_TILE_BYTES,
          "kq must be 16-byte aligned with a batch stride (multiple of 16) of at least "
          "ceil(G_max/16) tiles of %d bytes", LCSW_E4M3_TILE_BYTES);
    if ((a->flags & LCSW_DECODE_FORCE_MULTIKERNEL) ||
        !lcsw::fused_decode_supported(a->B, a->G_max, a->H_i, a->H_q, a->d_qk, a->d_v, a->k, a->P))
        return fail(LCSW_ERR_UNSUPPORTED, "FP8 decode: the shape is outside the persistent "
                    "kernel's envelope");
    const size_t need = lcsw_decode_workspace_size(a);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return fail(LCSW_ERR_WORKSPACE, "decode needs a 256-byte aligned workspace of %zu bytes",
                    need);
    DecodeWs w = carve_decode(a, ws);
    return cuda_status(lcsw::launch_fused_decode_e4m3(a, kq, sq_b, w.fused, w.status,
                                                      (cudaStream_t)stream),
                       "FP8 fused decode");
}

lcsw_status lcsw_decode_reuse(const lcsw_decode_args *a, const int32_t *idx_in, void *ws,
                              size_t ws_bytes, lcsw_stream stream) {
    LCSW_RANGE("lcsw_decode_reuse");
    CHECK(a, "null args");
    CHECK(a->B >= 0, "negative dimension");
    CHECK(p_ok(a->P), "P must be 1, 2, 4 or 8");
    CHECK(a->k >= 1, "k must be >= 1");
    const bool mla = mla_shape(a->d_qk, a->d_v);
    CHECK(mla ? (a->H_q > 0 && a->H_q % 16 == 0) : attn_shape_ok(a->H_q, a->d_qk, a->d_v),
          "unsupported attention shape");
    CHECK(!mla || !a->V || (a->V == a->K && a->sV_b == a->sK_b),
          "MLA geometry: V is the latent part of K (pass NULL or K itself)");
    if (a->B == 0) return LCSW_OK;
    CHECK(a->B <= 65535, "B must be <= 65535");
    CHECK(a->q && a->K && (a->V || mla) && a->seq_len && a->out && idx_in,
          "null pointer argument");
    CHECK(bf16_rows_ok(a->q, a->d_qk, 0) && bf16_rows_ok(a->K, a->d_qk, a->sK_b) &&
              (mla || bf16_rows_ok(a->V, a->d_v, a->sV_b)) && bf16_rows_ok(a->out, a->d_v, 0),
          "bf16 rows must be 16-byte aligned");
    CHECK(aligned(a->seq_len, 4) && aligned(idx_in, 4) && (!a->lse || aligned(a->lse, 4)),
          "misaligned int32/fp32 array");
    const size_t need = lcsw_decode_workspace_size(a);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return fail(LCSW_ERR_WORKSPACE, "decode reuse needs a 256-byte aligned workspace of %zu bytes",
                    need);
    DecodeWs w = carve_decode(a, ws);
    if (!(a->flags & LCSW_DECODE_FORCE_MULTIKERNEL) &&
        lcsw::reuse_decode_supported(a->B, a->H_q, a->d_qk, a->d_v, a->k) &&
        lcsw::fused_decode_ws_bytes(a->B, a->G_max, a->H_q, a->d_v, a->k, a->P) > 0)
        return cuda_status(lcsw::launch_reuse_decode(a, idx_in, w.fused, w.status,
                                                     (cudaStream_t)stream),
                           "decode reuse (persistent)");
    return cuda_status(decode_attend(a, idx_in, w.attn, (cudaStream_t)stream),
                       "decode reuse attention");
}

// ----------------------------------------------------------------- prefill --

struct PrefillWs {
    int *status;
    float *scores;  // dense scores: the fallback (and the path without fusion)
    int32_t *idx;
    int32_t *q_pos;
    int32_t *n_valid;
    void *attn;
    // fused selection
    bool fused;
    int cap;
    float *samp;
    uint32_t *thr;
    unsigned *ccount;
    int32_t *fail;  // [rows], then any_fail
    unsigned long long *cand;
    size_t total;
};

constexpr int kFusedMaxG = 524288;  // bitmap of the per-row selection in shared memory

static bool prefill_fused(const lcsw_prefill_args *a) {
    return a->H_i <= 8 && a->G_max <= kFusedMaxG &&
           lcsw::index_scores_tc_supported(a->B, a->T, a->H_i, a->G_max, a->sp_b);
}

static PrefillWs carve_prefill(const lcsw_prefill_args *a, void *ws) {
    Carver c(ws);
    PrefillWs w;
    const size_t rows = size_t(a->B) * a->T;
    w.status = static_cast<int *>(ws);
    w.scores = static_cast<float *>(c.take(rows * a->G_max * sizeof(float)));
    w.idx = static_cast<int32_t *>(c.take(rows * a->k * sizeof(int32_t)));
    w.q_pos = static_cast<int32_t *>(c.take(rows * sizeof(int32_t)));
    w.n_valid = static_cast<int32_t *>(c.take(rows * sizeof(int32_t)));
    w.attn = c.take(lcsw::sparse_attn_ws_bytes(int64_t(rows), a->H_q, a->d_v, a->k, a->P));
    w.fused = prefill_fused(a);
    w.cap = 0;
    w.samp = nullptr;
    w.thr = nullptr;
    w.ccount = nullptr;
    w.fail = nullptr;
    w.cand = nullptr;
    if (w.fused) {
        // about 3 k candidates per row are expected; room for 8 k (at least 4096)
        w.cap = a->k * 8 > 4096 ? a->k * 8 : 4096;
        const int n_samp = 128 * lcsw::prefill_sample_tiles(a->G_max);
        w.samp = static_cast<float *>(c.take(rows * n_samp * sizeof(float)));
        w.thr = static_cast<uint32_t *>(c.take(rows * sizeof(uint32_t)));
        w.ccount = static_cast<unsigned *>(c.take(rows * sizeof(unsigned)));
        w.fail = static_cast<int32_t *>(c.take((rows + 1) * sizeof(int32_t)));
        w.cand = static_cast<unsigned long long *>(c.take(rows * w.cap * sizeof(unsigned long long)));
    }
    w.total = c.off;
    return w;
}

size_t lcsw_prefill_workspace_size(const lcsw_prefill_args *a) {
    if (!a || a->B <= 0 || a->T <= 0 || a->G_max < 0 || a->k < 1 || !p_ok(a->P)) return 256;
    return carve_prefill(a, nullptr).total;
}

// query rows from which the prefill attention runs on the tensor cores
constexpr int64_t kPrefillTcRows = 256;

lcsw_status lcsw_prefill(const lcsw_prefill_args *a, void *ws, size_t ws_bytes,
                         lcsw_stream stream) {
    LCSW_RANGE("lcsw_prefill");
    CHECK(a, "null args");
    CHECK(a->B >= 0 && a->T >= 0 && a->G_max >= 0, "negative dimension");
    CHECK(a->d_idx == 64, "d_idx must be 64");
    CHECK(a->H_i >= 1 && a->H_i <= 16, "H_i must be in [1, 16]");
    CHECK(p_ok(a->P), "P must be 1, 2, 4 or 8");
    CHECK(a->k >= 1, "k must be >= 1");
    CHECK(attn_shape_ok(a->H_q, a->d_qk, a->d_v), "unsupported attention shape");
    const int64_t rows = int64_t(a->B) * a->T;
    if (rows == 0) return LCSW_OK;
    CHECK(rows <= 65535, "B*T must be <= 65535");
    CHECK(a->q_idx && a->w_head && a->k_pooled && a->k_idx && a->pool_w && a->q && a->K && a->V &&
              a->seq_len && a->out,
          "null pointer argument");
    CHECK(bf16_rows_ok(a->q_idx, 64, 0) && bf16_rows_ok(a->k_pooled, 64, a->sp_b) &&
              bf16_rows_ok(a->k_idx, 64, a->sk_b) && bf16_rows_ok(a->q, a->d_qk, 0) &&
              bf16_rows_ok(a->K, a->d_qk, a->sK_b) && bf16_rows_ok(a->V, a->d_v, a->sV_b) &&
              bf16_rows_ok(a->out, a->d_v, 0),
          "bf16 rows must be 16-byte aligned");
    CHECK(aligned(a->w_head, 4) && aligned(a->seq_len, 4) && aligned(a->pool_w, 4) &&
              (!a->lse || aligned(a->lse, 4)) && (!a->idx_out || aligned(a->idx_out, 4)),
          "misaligned fp32/int32 array");
    const size_t need = lcsw_prefill_workspace_size(a);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return fail(LCSW_ERR_WORKSPACE, "prefill needs a 256-byte aligned workspace of %zu bytes",
                    need);
    cudaStream_t st = (cudaStream_t)stream;
    PrefillWs w = carve_prefill(a, ws);
    int32_t *idx = a->idx_out ? a->idx_out : w.idx;

    // pool the groups the new chunk completes (and the one it finishes)
    cudaError_t e = lcsw::launch_pool_keys(a->k_idx, a->sk_b, a->pool_w, a->sw_b, a->seq_len,
                                           nullptr, a->B, a->T / a->P + 1, 64, a->P, 2, a->T,
                                           a->k_pooled, a->sp_b, st);
    if (e != cudaSuccess) return cuda_status(e, "prefill pool");
    e = lcsw::launch_prefill_positions(a->seq_len, a->B, a->T, w.q_pos, st);
    if (e != cudaSuccess) return cuda_status(e, "prefill positions");
    e = lcsw::launch_visible_counts(a->seq_len, w.q_pos, a->B, a->T, a->P, w.n_valid, st);
    if (e != cudaSuccess) return cuda_status(e, "prefill visible counts");
    if (w.fused) {
        // sample -> per-row thresholds -> candidates -> exact top k; rows that
        // cannot be proven complete take dense scores and the radix top-k
        const int n_samp = 128 * lcsw::prefill_sample_tiles(a->G_max);
        e = cudaMemsetAsync(w.ccount, 0, rows * sizeof(unsigned), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(w.fail, 0, (rows + 1) * sizeof(int32_t), st);
        if (e != cudaSuccess) return cuda_status(e, "prefill clear");
        e = lcsw::launch_prefill_sample_scores(a->q_idx, a->w_head, a->k_pooled, a->sp_b,
                                               a->seq_len, w.q_pos, a->B, a->T, a->H_i, a->P,
                                               a->G_max, w.samp, w.status, st);
        if (e != cudaSuccess) return cuda_status(e, "prefill sample scores");
        e = lcsw::launch_prefill_thresholds(w.samp, n_samp, w.n_valid, rows, a->k, w.thr,
                                            (a->flags & LCSW_PREFILL_FORCE_FALLBACK) != 0, st);
        if (e != cudaSuccess) return cuda_status(e, "prefill thresholds");
        e = lcsw::launch_prefill_candidates(a->q_idx, a->w_head, a->k_pooled, a->sp_b, a->seq_len,
                                            w.q_pos, a->B, a->T, a->H_i, a->P, a->G_max, w.thr,
                                            w.ccount, w.cand, w.cap, w.status, st);
        if (e != cudaSuccess) return cuda_status(e, "prefill candidates");
        e = lcsw::launch_prefill_select(w.cand, w.ccount, w.cap, w.n_valid, rows, a->G_max, a->k,
                                        idx, w.fail, w.fail + rows, st);
        if (e != cudaSuccess) return cuda_status(e, "prefill select");
        e = lcsw::launch_index_scores_tc(a->q_idx, a->w_head, a->k_pooled, a->sp_b, a->seq_len,
                                         w.q_pos, a->B, a->T, a->H_i, a->P, a->G_max, w.scores,
                                         w.status, st, w.fail + rows);
        if (e != cudaSuccess) return cuda_status(e, "prefill fallback scores");
        e = lcsw::launch_topk_rows(w.scores, w.n_valid, nullptr, a->P, a->T, rows, a->G_max,
                                   a->k, idx, st, w.fail);
        if (e != cudaSuccess) return cuda_status(e, "prefill fallback top-k");
    } else {
        if (lcsw::index_scores_tc_supported(a->B, a->T, a->H_i, a->G_max, a->sp_b)) {
            e = lcsw::launch_index_scores_tc(a->q_idx, a->w_head, a->k_pooled, a->sp_b,
                                             a->seq_len, w.q_pos, a->B, a->T, a->H_i, a->P,
                                             a->G_max, w.scores, w.status, st);
        } else {
            CHECK(int64_t(a->B) * ((a->T + 3) / 4) <= 65535, "B * ceil(T/4) must be <= 65535");
            e = lcsw::launch_index_scores_mma(a->q_idx, a->w_head, a->k_pooled, a->sp_b,
                                              a->seq_len, w.q_pos, a->B, a->T, a->H_i, a->P,
                                              a->G_max, w.scores, st);
        }
        if (e != cudaSuccess) return cuda_status(e, "prefill scores");
        e = lcsw::launch_topk_rows(w.scores, w.n_valid, nullptr, a->P, a->T, rows, a->G_max,
                                   a->k, idx, st);
        if (e != cudaSuccess) return cuda_status(e, "prefill top-k");
    }
    // many query rows: the persistent tensor-core attention (one row per CTA
    // step, no split of the selected tokens); few rows: the split-K kernel
    if (rows >= kPrefillTcRows &&
        lcsw::sparse_attn_tc_supported(rows, a->H_q, a->d_qk, a->d_v, a->P, a->k)) {
        e = lcsw::launch_sparse_attn_tc(a->q, a->K, a->sK_b, a->V, a->sV_b, a->seq_len, idx, a->B,
                                        a->T, a->H_q, a->d_qk, a->d_v, a->P, a->k, a->scale,
                                        a->out, a->lse, w.status, st,
                                        (a->flags & LCSW_PREFILL_TEST_SKIP_GATHER) != 0);
        return cuda_status(e, "prefill attention (tensor cores)");
    }
    e = lcsw::launch_sparse_attn(a->q, a->K, a->sK_b, a->V, a->sV_b, a->seq_len, idx, a->B, a->T,
                                 a->H_q, a->d_qk, a->d_v, a->P, a->k, a->scale, a->out, a->lse,
                                 w.attn, st);
    return cuda_status(e, "prefill attention");
}

lcsw_status lcsw_append_token(const lcsw_bf16 *rows, int64_t s_rows, const int32_t *seq_len,
                              int B, lcsw_bf16 *k_idx, int64_t sk_b, int d_idx, lcsw_bf16 *K,
                              int64_t sK_b, int d_qk, lcsw_bf16 *V, int64_t sV_b, int d_v,
                              lcsw_stream stream) {
    LCSW_RANGE("lcsw_append_token");
    CHECK(B >= 0 && d_idx > 0 && d_qk > 0 && d_v >= 0, "bad dimension");
    CHECK(d_idx % 8 == 0 && d_qk % 8 == 0 && d_v % 8 == 0, "row widths must be multiples of 8");
    CHECK(!V == (d_v == 0), "V and d_v: both given or neither");
    if (B == 0) return LCSW_OK;
    CHECK(rows && seq_len && k_idx && K, "null pointer argument");
    CHECK(s_rows >= d_idx + d_qk + d_v && sk_b >= 0 && sK_b >= 0 && sV_b >= 0,
          "bad stride (a packed row holds d_idx + d_qk + d_v values)");
    CHECK(bf16_rows_ok(rows, 8, s_rows) && bf16_rows_ok(k_idx, d_idx, sk_b) &&
              bf16_rows_ok(K, d_qk, sK_b) && (!V || bf16_rows_ok(V, d_v, sV_b)) &&
              aligned(seq_len, 4),
          "bf16 rows must be 16-byte aligned");
    return cuda_status(lcsw::launch_append_token(rows, s_rows, seq_len, B, k_idx, sk_b, d_idx, K,
                                                 sK_b, d_qk, V, sV_b, d_v, (cudaStream_t)stream),
                       "append launch");
}

// argument checks shared by the FP8 and INT8 row quantizers
static lcsw_status quantize_rows_args(const lcsw_bf16 *x, int64_t sx_b, const int32_t *row_begin,
                                      int B, int n_rows, int width, const void *codes,
                                      int64_t sc_b, const float *scales, int64_t ss_b) {
    CHECK(B >= 0 && n_rows >= 0 && width > 0, "bad dimension");
    CHECK(width % 16 == 0, "width must be a multiple of 16");
    if (B == 0 || n_rows == 0) return LCSW_OK;
    CHECK(x && codes && scales, "null pointer argument");
    CHECK(bf16_rows_ok(x, width, sx_b) && aligned(codes, 16) && sc_b % 16 == 0 &&
              aligned(scales, 4) && (!row_begin || aligned(row_begin, 4)),
          "misaligned argument (x rows 16-byte aligned, codes and their stride 16 bytes)");
    CHECK(sx_b >= 0 && sc_b >= 0 && ss_b >= 0, "strides must be >= 0");
    return LCSW_OK;
}

lcsw_status lcsw_quantize_rows_e4m3(const lcsw_bf16 *x, int64_t sx_b, const int32_t *row_begin,
                                    int B, int n_rows, int width, uint8_t *codes, int64_t sc_b,
                                    float *scales, int64_t ss_b, lcsw_stream stream) {
    LCSW_RANGE("lcsw_quantize_rows_e4m3");
    const lcsw_status a = quantize_rows_args(x, sx_b, row_begin, B, n_rows, width, codes, sc_b,
                                             scales, ss_b);
    if (a != LCSW_OK || B == 0 || n_rows == 0) return a;
    return cuda_status(lcsw::launch_quantize_rows_e4m3(x, sx_b, row_begin, n_rows, width, B,
                                                       codes, sc_b, scales, ss_b,
                                                       (cudaStream_t)stream),
                       "quantize rows launch");
}

lcsw_status lcsw_quantize_rows_i8(const lcsw_bf16 *x, int64_t sx_b, const int32_t *row_begin,
                                  int B, int n_rows, int width, int8_t *codes, int64_t sc_b,
                                  float *scales, int64_t ss_b, lcsw_stream stream) {
    LCSW_RANGE("lcsw_quantize_rows_i8");
    const lcsw_status a = quantize_rows_args(x, sx_b, row_begin, B, n_rows, width, codes, sc_b,
                                             scales, ss_b);
    if (a != LCSW_OK || B == 0 || n_rows == 0) return a;
    return cuda_status(lcsw::launch_quantize_rows_i8(x, sx_b, row_begin, n_rows, width, B, codes,
                                                     sc_b, scales, ss_b, (cudaStream_t)stream),
                       "INT8 quantize rows launch");
}

size_t lcsw_sparse_attn_kv8_workspace_size(int B, int T, int H_q, int d_v, int k, int P) {
    if (B <= 0 || T <= 0 || H_q <= 0 || d_v <= 0 || k <= 0 || !p_ok(P)) return 0;
    return lcsw::sparse_attn_kv8_ws_bytes(int64_t(B) * T, H_q, d_v, k, P);
}

// the FP8 and INT8 K/V attention entries: the same checks and kernel
static lcsw_status quantized_kv_attn(const lcsw_bf16 *q, const uint8_t *kc, int64_t skc_b,
                                     const float *ks, int64_t sks_b, const uint8_t *vc,
                                     int64_t svc_b, const float *vs, int64_t svs_b,
                                     const int32_t *seq_len, const int32_t *idx, int B, int T,
                                     int H_q, int d_qk, int d_v, int P, int k, float scale,
                                     lcsw_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                     bool int8_codes, lcsw_stream stream) {
    CHECK(B >= 0 && T >= 0, "negative dimension");
    CHECK(p_ok(P), "P must be 1, 2, 4 or 8");
    CHECK(k >= 1, "k must be >= 1");
    CHECK(attn_shape_ok(H_q, d_qk, d_v), "unsupported attention shape");
    const int64_t rows = int64_t(B) * T;
    if (rows == 0) return LCSW_OK;
    CHECK(rows <= 65535, "B*T must be <= 65535");
    CHECK(q && kc && ks && vc && vs && seq_len && idx && out, "null pointer argument");
    CHECK(bf16_rows_ok(q, d_qk, 0) && bf16_rows_ok(out, d_v, 0) && aligned(kc, 16) &&
              aligned(vc, 16) && skc_b % 16 == 0 && svc_b % 16 == 0 && aligned(ks, 4) &&
              aligned(vs, 4) && aligned(seq_len, 4) && aligned(idx, 4) &&
              (!lse || aligned(lse, 4)),
          "misaligned argument (code caches and their strides 16 bytes)");
    CHECK(skc_b >= 0 && svc_b >= 0 && sks_b >= 0 && svs_b >= 0, "strides must be >= 0");
    const size_t need = lcsw::sparse_attn_kv8_ws_bytes(rows, H_q, d_v, k, P);
    if (need && (!ws || ws_bytes < need || !aligned(ws, 16)))
        return fail(LCSW_ERR_WORKSPACE, "%s K/V attention needs a 16-byte aligned workspace "
                    "of %zu bytes", int8_codes ? "INT8" : "FP8", need);
    return cuda_status(lcsw::launch_sparse_attn_kv8(q, kc, skc_b, ks, sks_b, vc, svc_b, vs, svs_b,
                                                    seq_len, idx, B, T, H_q, d_qk, d_v, P, k,
                                                    scale, out, lse, ws, int8_codes,
                                                    (cudaStream_t)stream),
                       "quantized K/V attention launch");
}

lcsw_status lcsw_sparse_attn_kv8(const lcsw_bf16 *q, const uint8_t *kc, int64_t skc_b,
                                 const float *ks, int64_t sks_b, const uint8_t *vc,
                                 int64_t svc_b, const float *vs, int64_t svs_b,
                                 const int32_t *seq_len, const int32_t *idx, int B, int T,
                                 int H_q, int d_qk, int d_v, int P, int k, float scale,
                                 lcsw_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                 lcsw_stream stream) {
    LCSW_RANGE("lcsw_sparse_attn_kv8");
    return quantized_kv_attn(q, kc, skc_b, ks, sks_b, vc, svc_b, vs, svs_b, seq_len, idx, B, T,
                             H_q, d_qk, d_v, P, k, scale, out, lse, ws, ws_bytes, false, stream);
}

lcsw_status lcsw_sparse_attn_kvi8(const lcsw_bf16 *q, const int8_t *kc, int64_t skc_b,
                                  const float *ks, int64_t sks_b, const int8_t *vc,
                                  int64_t svc_b, const float *vs, int64_t svs_b,
                                  const int32_t *seq_len, const int32_t *idx, int B, int T,
                                  int H_q, int d_qk, int d_v, int P, int k, float scale,
                                  lcsw_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                  lcsw_stream stream) {
    LCSW_RANGE("lcsw_sparse_attn_kvi8");
    return quantized_kv_attn(q, reinterpret_cast<const uint8_t *>(kc), skc_b, ks, sks_b,
                             reinterpret_cast<const uint8_t *>(vc), svc_b, vs, svs_b, seq_len,
                             idx, B, T, H_q, d_qk, d_v, P, k, scale, out, lse, ws, ws_bytes, true,
                             stream);
}

size_t lcsw_sparse_attn_mla_workspace_size(int B, int T, int H_q, int k, int P) {
    if (B <= 0 || T <= 0 || H_q <= 0 || k < 1 || !p_ok(P)) return 0;
    return lcsw::sparse_attn_mla_ws_bytes(int64_t(B) * T, H_q, k, P);
}

lcsw_status lcsw_sparse_attn_mla(const lcsw_bf16 *q, const lcsw_bf16 *kv, int64_t skv_b,
                                 const int32_t *seq_len, const int32_t *idx, int B, int T,
                                 int H_q, int P, int k, float scale, lcsw_bf16 *out, float *lse,
                                 void *ws, size_t ws_bytes, lcsw_stream stream) {
    LCSW_RANGE("lcsw_sparse_attn_mla");
    CHECK(B >= 0 && T >= 0, "negative dimension");
    CHECK(H_q > 0 && H_q % 16 == 0, "H_q must be a positive multiple of 16");
    CHECK(p_ok(P), "P must be 1, 2, 4 or 8");
    CHECK(k >= 1, "k must be >= 1");
    const int64_t rows = int64_t(B) * T;
    if (rows == 0) return LCSW_OK;
    CHECK(rows <= 65535, "B*T must be <= 65535");
    CHECK(q && kv && seq_len && idx && out, "null pointer argument");
    CHECK(bf16_rows_ok(q, LCSW_MLA_DQK, 0) && bf16_rows_ok(kv, LCSW_MLA_DQK, skv_b) &&
              bf16_rows_ok(out, LCSW_MLA_DV, 0) && skv_b >= 0,
          "bf16 rows must be 16-byte aligned");
    CHECK(aligned(seq_len, 4) && aligned(idx, 4) && (!lse || aligned(lse, 4)),
          "misaligned int32/fp32 array");
    const size_t need = lcsw::sparse_attn_mla_ws_bytes(rows, H_q, k, P);
    if (need && (!ws || ws_bytes < need || !aligned(ws, 16)))
        return fail(LCSW_ERR_WORKSPACE, "MLA sparse attention needs a 16-byte aligned workspace "
                    "of %zu bytes", need);
    return cuda_status(lcsw::launch_sparse_attn_mla(q, kv, skv_b, seq_len, idx, B, T, H_q, P, k,
                                                    scale, out, lse, ws, (cudaStream_t)stream),
                       "MLA sparse attention");
}

lcsw_status lcsw_sparse_attn_noalloc(const lcsw_bf16 *q, const lcsw_bf16 *K, int64_t sK_b,
                                     const lcsw_bf16 *V, int64_t sV_b, const int32_t *seq_len,
                                     const int32_t *idx, int B, int T, int H_q, int d_qk,
                                     int d_v, int P, int k, float scale, lcsw_bf16 *out,
                                     float *lse, lcsw_stream stream) {
    LCSW_RANGE("lcsw_sparse_attn_noalloc");
    // the argument checks of lcsw_sparse_attn first, then the scratch size:
    // neither needs the device, so a rejected call launches nothing
    const lcsw_status chk = check_attn(q, K, sK_b, V, sV_b, seq_len, idx, B, T, H_q, d_qk, d_v,
                                       P, k, out, lse);
    if (chk != LCSW_OK) return chk;
    if (int64_t(B) * T == 0) return LCSW_OK;
    const size_t need = lcsw_sparse_attn_workspace_size(B, T, H_q, d_v, k, P);
    if (need > size_t(LCSW_NOALLOC_SCRATCH_BYTES))
        return fail(LCSW_ERR_UNSUPPORTED,
                    "sparse_attn_noalloc: this shape needs %zu bytes of split-K scratch, above "
                    "the fixed %zu; call lcsw_sparse_attn with a workspace instead",
                    need, size_t(LCSW_NOALLOC_SCRATCH_BYTES));
    void *scratch = nullptr;
    const lcsw_status s = attn_scratch(&scratch);
    if (s != LCSW_OK) return s;
    return lcsw_sparse_attn(q, K, sK_b, V, sV_b, seq_len, idx, B, T, H_q, d_qk, d_v, P, k, scale,
                            out, lse, scratch, size_t(LCSW_NOALLOC_SCRATCH_BYTES), stream);
}

lcsw_status lcsw_kda_step(const lcsw_bf16 *qkv, const lcsw_bf16 *conv_w, lcsw_bf16 *conv_state,
                          const float *g, const float *beta, float *state, lcsw_bf16 *out,
                          int B, int T, int H, int D, lcsw_stream stream) {
    LCSW_RANGE("lcsw_kda_step");
    CHECK(B >= 0 && T >= 0 && H >= 1 && D >= 1, "bad dimension");
    if (D != 128) return fail(LCSW_ERR_UNSUPPORTED, "KDA step: head width %d (only 128)", D);
    CHECK(B <= 65535, "B must be at most 65535");
    if (B == 0 || T == 0) return LCSW_OK;
    CHECK(qkv && conv_w && conv_state && g && beta && state && out, "null pointer argument");
    CHECK(aligned(qkv, 2) && aligned(conv_w, 8) && aligned(conv_state, 2) && aligned(g, 4) &&
              aligned(beta, 4) && aligned(state, 16) && aligned(out, 8),
          "misaligned argument (conv_w 8 bytes, state 16, out 8)");
    return cuda_status(lcsw::launch_kda_step(qkv, conv_w, conv_state, g, beta, state, out, B, T,
                                             H, (cudaStream_t)stream),
                       "KDA step launch");
}

int lcsw_checks_enabled(void) {
#ifdef LCSW_CHECKS
    return 1;
#else
    return 0;
#endif
}

int lcsw_check_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    int first = 0;
    for (auto reader : lcsw::check_readers()) {
        const int v = reader();
        if (v && !first) first = v;
    }
    return first;
}

lcsw_status lcsw_get_status(void *ws, lcsw_stream stream) {
    LCSW_RANGE("lcsw_get_status");
    CHECK(ws && aligned(ws, 4), "null or misaligned workspace");
    cudaStream_t st = (cudaStream_t)stream;
    int word = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e, "stream synchronize");
    e = cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e, "status read");
    if (word == 0) return LCSW_OK;
    const int zero = 0;
    e = cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_status(e, "status clear");
    return fail(LCSW_ERR_TIMEOUT, "a device-side bounded wait ran out (code %d); zero-fill the "
                "workspace before reusing it", word);
}

}  // extern "C"
