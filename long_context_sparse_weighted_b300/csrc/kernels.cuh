// Internal launchers of the liblcsw kernels.  Arguments are validated by the
// C-ABI layer (lcsw_api.cu) before any of these is called; each returns the
// launch's cudaError_t.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lcsw {

// IndexPool.  mode 0: groups [g_begin[b] (or 0), +g_span); mode 1: only the
// group completed by the newest token (g = L/P - 1 when L % P == 0); mode 2:
// groups from the one holding token L - tail on, g_span of them.
cudaError_t launch_pool_keys(const uint16_t *k_idx, int64_t sk_b, const float *pool_w,
                             int64_t sw_b, const int32_t *seq_len, const int32_t *g_begin,
                             int B, int g_span, int d_idx, int P, int mode, int tail,
                             uint16_t *k_pooled, int64_t sp_b, cudaStream_t st);

// FP8 pooled keys: groups [0, n_groups) of every sequence's bf16 pooled keys
// into the tile-major E4M3 cache (e4m3_core.cuh).
cudaError_t launch_quantize_keys_e4m3(const uint16_t *k_pooled, int64_t sp_b, int B, int n_groups,
                                      uint8_t *kq, int64_t sq_b, cudaStream_t st);

// KDA step over T tokens for B sequences, H heads of width 128 (kda_step.cu).
cudaError_t launch_kda_step(const uint16_t *qkv, const uint16_t *conv_w, uint16_t *conv_state,
                            const float *g, const float *beta, float *state, uint16_t *out,
                            int B, int T, int H, cudaStream_t st);

// FP8 K/V cache rows: rows [r0_b, r0_b + n_rows) of every sequence (r0_b =
// row_begin[b], or 0), `width` bf16 values each -> E4M3 codes (row-major,
// batch stride sc_b bytes) and one fp32 scale per row (batch stride ss_b).
cudaError_t launch_quantize_rows_e4m3(const uint16_t *x, int64_t sx_b, const int32_t *row_begin,
                                      int n_rows, int width, int B, uint8_t *codes, int64_t sc_b,
                                      float *scales, int64_t ss_b, cudaStream_t st);
// The newest token's rows (position seq_len[b] - 1) of k_idx, K and V (V may
// be null with d_v 0) from packed rows [B][d_idx + d_qk + d_v] (stride s_rows).
cudaError_t launch_append_token(const uint16_t *rows, int64_t s_rows, const int32_t *seq_len,
                                int B, uint16_t *k_idx, int64_t sk_b, int d_idx, uint16_t *K,
                                int64_t sK_b, int d_qk, uint16_t *V, int64_t sV_b, int d_v,
                                cudaStream_t st);
// INT8 K/V cache rows, as launch_quantize_rows_e4m3: int8 codes (symmetric,
// scale amax / 127 per row).
cudaError_t launch_quantize_rows_i8(const uint16_t *x, int64_t sx_b, const int32_t *row_begin,
                                    int n_rows, int width, int B, int8_t *codes, int64_t sc_b,
                                    float *scales, int64_t ss_b, cudaStream_t st);

// q_pos[b][t] = seq_len[b] - T + t (the chunk's absolute positions).
cudaError_t launch_prefill_positions(const int32_t *seq_len, int B, int T, int32_t *q_pos,
                                     cudaStream_t st);

// Indexer scores with mma.sync (decode / short query blocks).
cudaError_t launch_index_scores_mma(const uint16_t *q_idx, const float *w_head,
                                    const uint16_t *k_pooled, int64_t sp_b,
                                    const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                    int H_i, int P, int G_max, float *scores, cudaStream_t st);

// Indexer scores as a tcgen05/TMEM GEMM fed by TMA (chunked prefill).
// Returns cudaErrorNotSupported when the shape is outside its envelope.  With
// run_if (H_i <= 8 only) the launch does nothing unless *run_if != 0.
cudaError_t launch_index_scores_tc(const uint16_t *q_idx, const float *w_head,
                                   const uint16_t *k_pooled, int64_t sp_b,
                                   const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                   int H_i, int P, int G_max, float *scores, int *status,
                                   cudaStream_t st, const int *run_if = nullptr);
bool index_scores_tc_supported(int B, int T, int H_i, int G_max, int64_t sp_b);

// Fused prefill selection (H_i <= 8).  Sample: dense scores of
// prefill_sample_tiles(G_max) group tiles spread over the sequence, into
// samp [B*T][128 * tiles].  Candidates: every visible group whose score key is
// at or above thr[row], appended as (key | group << 32) to cand [B*T][cap],
// counted in ccount[row] (zeroed by the caller; may exceed cap).
int prefill_sample_tiles(int G_max);
cudaError_t launch_prefill_sample_scores(const uint16_t *q_idx, const float *w_head,
                                         const uint16_t *k_pooled, int64_t sp_b,
                                         const int32_t *seq_len, const int32_t *q_pos, int B,
                                         int T, int H_i, int P, int G_max, float *samp,
                                         int *status, cudaStream_t st);
cudaError_t launch_prefill_candidates(const uint16_t *q_idx, const float *w_head,
                                      const uint16_t *k_pooled, int64_t sp_b,
                                      const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                      int H_i, int P, int G_max, const uint32_t *thr,
                                      unsigned *ccount, unsigned long long *cand, int cap,
                                      int *status, cudaStream_t st);
// Per row: the threshold key of the candidate pass from the sample, then the
// exact top k from the candidates (ascending groups, -1 padded).  A row whose
// candidates cannot be proven to hold its top k gets fail[row] = 1 and
// *any_fail = 1 (fail and any_fail zeroed by the caller).
cudaError_t launch_prefill_thresholds(const float *samp, int n_samp, const int32_t *n_valid,
                                      int64_t rows, int k, uint32_t *thr, bool force_fallback,
                                      cudaStream_t st);
cudaError_t launch_prefill_select(const unsigned long long *cand, const unsigned *ccount, int cap,
                                  const int32_t *n_valid, int64_t rows, int G_max, int k,
                                  int32_t *idx, int *fail, int *any_fail, cudaStream_t st);

cudaError_t launch_visible_counts(const int32_t *seq_len, const int32_t *q_pos, int B, int T,
                                  int P, int32_t *n_valid, cudaStream_t st);

// Top-k per row, one thread block per row.  n_valid may be NULL, in which case
// row r = b*T + t has seq_len[b]/P valid groups (seq_len/P/T must be given).
cudaError_t launch_topk_rows(const float *scores, const int32_t *n_valid,
                             const int32_t *seq_len, int P, int T, int64_t rows, int G_max,
                             int k, int32_t *idx, cudaStream_t st,
                             const int32_t *row_mask = nullptr);
// The same selection for a few long rows, spread over many blocks (three
// launches and a memset; topk.cu).  Supported for rows <= 32 and
// 16384 <= G_max <= 524288; ws of topk_wide_ws_bytes bytes, 256-aligned.
bool topk_wide_supported(int64_t rows, int G_max, int k);
size_t topk_wide_ws_bytes(int64_t rows, int G_max, int k);
cudaError_t launch_topk_rows_wide(const float *scores, const int32_t *n_valid,
                                  const int32_t *seq_len, int P, int T, int64_t rows, int G_max,
                                  int k, int32_t *idx, void *ws, cudaStream_t st);

// Sparse attention for many query rows on tcgen05 (H_q <= 32, d_qk = d_v =
// 128): one persistent CTA per SM, no workspace; records a timed-out wait in
// *status (nullable).
bool sparse_attn_tc_supported(int64_t rows, int H_q, int d_qk, int d_v, int P, int k);
cudaError_t launch_sparse_attn_tc(const uint16_t *q, const uint16_t *K, int64_t sK_b,
                                  const uint16_t *V, int64_t sV_b, const int32_t *seq_len,
                                  const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v,
                                  int P, int k, float scale, uint16_t *out, float *lse,
                                  int *status, cudaStream_t st, bool test_skip_gather = false);

// Split-K sparse attention + combine.
int sparse_attn_splits(int64_t rows, int H_q, int k, int P);
// The same attention over an FP8 (E4M3) K/V cache with one fp32 scale per
// token row (sparse_attn_kv8.cu): codes kc [B][*][d_qk], vc [B][*][d_v]
// (batch strides in bytes), scales ks, vs [B][*] (strides in elements); with
// int8_codes the codes are INT8 (i8_core.cuh) instead.
int sparse_attn_kv8_splits(int64_t rows, int H_q, int k, int P);
size_t sparse_attn_kv8_ws_bytes(int64_t rows, int H_q, int d_v, int k, int P);
cudaError_t launch_sparse_attn_kv8(const uint16_t *q, const uint8_t *kc, int64_t skc_b,
                                   const float *ks, int64_t sks_b, const uint8_t *vc,
                                   int64_t svc_b, const float *vs, int64_t svs_b,
                                   const int32_t *seq_len, const int32_t *idx, int B, int T,
                                   int H_q, int d_qk, int d_v, int P, int k, float scale,
                                   uint16_t *out, float *lse, void *ws, bool int8_codes,
                                   cudaStream_t st);
// MLA latent geometry (sparse_attn_mla.cu): rows of 576 = latent 512 + rotary
// 64, the latent doubling as the value; out rows of 512.
int sparse_attn_mla_splits(int64_t rows, int H_q, int k, int P);
size_t sparse_attn_mla_ws_bytes(int64_t rows, int H_q, int k, int P);
cudaError_t launch_sparse_attn_mla(const uint16_t *q, const uint16_t *kv, int64_t skv_b,
                                   const int32_t *seq_len, const int32_t *idx, int B, int T,
                                   int H_q, int P, int k, float scale, uint16_t *out, float *lse,
                                   void *ws, cudaStream_t st,
                                   bool after_selection = false);
size_t sparse_attn_ws_bytes(int64_t rows, int H_q, int d_v, int k, int P);
cudaError_t launch_sparse_attn(const uint16_t *q, const uint16_t *K, int64_t sK_b,
                               const uint16_t *V, int64_t sV_b, const int32_t *seq_len,
                               const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v,
                               int P, int k, float scale, uint16_t *out, float *lse, void *ws,
                               cudaStream_t st);

}  // namespace lcsw
